// ep_device.cuh — device helpers shared by the libep_b300 kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ep {

// Bits of the workspace status word (sticky until ep_get_error clears them).
constexpr uint32_t kStatusBadIndex = 1u;
constexpr uint32_t kStatusTimeout = 2u;

__device__ __forceinline__ void raise_status(uint32_t* status, uint32_t bit) {
  atomicOr(status, bit);
}

// ---- programmatic dependent launch ----------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialisation, so it may start while the kernel before it in the stream is
// still finishing. pdl_wait() blocks until that kernel has completed and its
// memory is visible (a no-op when there is no programmatic predecessor);
// nothing the predecessor writes may be read, and nothing it reads or writes
// may be written, before it. pdl_launch_dependents() lets the next kernel
// start launching; each kernel calls it only after its own pdl_wait(), so by
// induction everything older than the immediate predecessor has completed
// once a kernel starts: its pre-wait code may read the outputs of kernels two
// or more launches back.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- 16-byte global memory access ----------------------------------------
// Streaming read of data that this kernel touches once: skip L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_v2(void* p, uint2 v) {
  asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// ---- L2 residency ------------------------------------------------------------
// The dispatch reads x once and writes the payload once; neither is reused
// within the step. The scatter marks what it touches as the first to be
// evicted from L2: its x reads (.L2::evict_first) and its payload stores (an
// evict-first cache policy), so that the payload stream recycles its own
// lines rather than pushing out lines that are read again (the routing
// metadata, and the combine's inputs in a step that follows).

// A cache policy under which the lines an access allocates are the first
// candidates for eviction from L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void st_v4_hint(void* p, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(pol)
               : "memory");
}

__device__ __forceinline__ void st_v2_hint(void* p, uint2 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1,%2}, %3;" ::"l"(p), "r"(v.x), "r"(v.y), "l"(pol) : "memory");
}

__device__ __forceinline__ uint4 ld_stream_v4_hint(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

// ---- bf16 pairs ----------------------------------------------------------
// A 32-bit word holds two bf16: the low half is the lower-addressed element.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---- warp reductions -------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Exclusive scan of one value per thread over the block (at most 32 warps);
// returns the exclusive prefix and sets `total` (same in every thread).
// warp_s holds one int per warp.
__device__ __forceinline__ int block_exclusive_scan(int v, int& total, int* warp_s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int incl = warp_inclusive_scan(v);
  __syncthreads();  // warp_s may still be read by a previous call
  if (lane == 31) warp_s[warp] = incl;
  __syncthreads();
  int wpre = 0, tot = 0;
  for (int i = 0; i < nw; ++i) {
    const int x = warp_s[i];
    wpre += i < warp ? x : 0;
    tot += x;
  }
  total = tot;
  return wpre + incl - v;
}

// Per-tile expert masks mask[e][w] (bit b of word w: token 32w+b of the tile
// chose e; TW words per expert, TW a power of two <= 32): pre[e][w] = set bits
// of e in the words before w, and tile_counts[e * ntiles + b] = set bits in
// the whole tile. One thread per (e, w) and a segmented warp scan of log2(TW)
// steps; the loop bound is the same for the whole block, so every lane takes
// part in every shuffle (blockDim a multiple of 32).
__device__ __forceinline__ void tile_word_prefix(const uint32_t* mask, uint32_t* pre, int E, int TW,
                                                 int32_t* __restrict__ tile_counts, int ntiles, int b) {
  const int lane = threadIdx.x & 31;
  const int n = E * TW;
  for (int i0 = 0; i0 < n; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    const bool ok = i < n;
    const int c = ok ? __popc(mask[i]) : 0;
    int v = c;
    for (int o = 1; o < TW; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if ((lane & (TW - 1)) >= o) v += u;
    }
    if (ok) {
      pre[i] = static_cast<uint32_t>(v - c);
      if ((i & (TW - 1)) == TW - 1) tile_counts[static_cast<int64_t>(i / TW) * ntiles + b] = v;
    }
  }
}

// ---- per-token int8 code of 16 consecutive elements --------------------------
// scale = amax / 127 (IEEE division); q = clamp(rint(x / scale), -127, 127)
// with IEEE division and ties-to-even; scale == 0 codes every element as 0.
__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, float scale) {
  auto q1 = [scale](float v) -> uint32_t {
    int q = (scale == 0.0f) ? 0 : __float2int_rn(__fdiv_rn(v, scale));
    q = max(-127, min(127, q));
    return static_cast<uint32_t>(q) & 0xffu;
  };
  return q1(a) | (q1(b) << 8) | (q1(c) << 16) | (q1(d) << 24);
}

// 16 bf16 (two 16-byte words) -> 16 int8 codes (one 16-byte word).
__device__ __forceinline__ uint4 quant16(uint4 a0, uint4 a1, float scale) {
  uint4 r;
  r.x = quant4(bf16_lo(a0.x), bf16_hi(a0.x), bf16_lo(a0.y), bf16_hi(a0.y), scale);
  r.y = quant4(bf16_lo(a0.z), bf16_hi(a0.z), bf16_lo(a0.w), bf16_hi(a0.w), scale);
  r.z = quant4(bf16_lo(a1.x), bf16_hi(a1.x), bf16_lo(a1.y), bf16_hi(a1.y), scale);
  r.w = quant4(bf16_lo(a1.z), bf16_hi(a1.z), bf16_lo(a1.w), bf16_hi(a1.w), scale);
  return r;
}

// The same code without a division per element, for a scale of at least
// 2^-100. With inv = 1/scale rounded to nearest, the quotient estimate
// q0 = fl(x * inv) is corrected once with its exact remainder,
// rem = fma(-q0, scale, x), as q1 = fma(rem, inv, q0) (the classic
// remainder-based correction of a division by multiplication with a rounded
// reciprocal), and q = rint(q1) is formed by adding 1.5 * 2^23, which rounds
// to nearest-even at unit spacing for |q1| < 2^22 and leaves q in the low
// byte of the sum's bits. rint(q1) equals rint(fl(x / scale)) for every bf16
// amax with amax/127 >= 2^-100 and every bf16 |x| <= amax: checked
// exhaustively on the host (523,237,695 pairs, no mismatch) and on the GPU by
// the tests. Without the correction, 5,304 of those pairs round differently.
// |q| <= 127 on that domain, so the clamp never binds. Two elements are
// processed per packed fp32x2 instruction (mul/fma/add .rn.f32x2: IEEE
// round-to-nearest per element, denormals kept).
constexpr float kFastScaleMin = 0x1p-100f;

__device__ __forceinline__ uint64_t f32x2_pack(uint32_t lo, uint32_t hi) {
  return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_splat(float v) {
  return f32x2_pack(__float_as_uint(v), __float_as_uint(v));
}
__device__ __forceinline__ float f32x2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f32x2_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }

__device__ __forceinline__ uint32_t pack4_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// 16 bf16 -> 16 int8 codes by the corrected-quotient path (scale >= 2^-100).
__device__ __forceinline__ uint4 quant16_fast(uint4 a0, uint4 a1, float scale, float inv) {
  const uint64_t inv2 = f32x2_pack(__float_as_uint(inv), __float_as_uint(inv));
  const uint64_t nsc2 = f32x2_pack(__float_as_uint(-scale), __float_as_uint(-scale));
  const uint64_t mg2 = f32x2_pack(0x4B400000u, 0x4B400000u);  // 1.5 * 2^23 in both halves
  const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  uint32_t tb[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint64_t x2 = f32x2_pack(w[i] << 16, w[i] & 0xffff0000u);  // (lower, upper) element
    const uint64_t q0 = f32x2_mul(x2, inv2);
    const uint64_t rem = f32x2_fma(q0, nsc2, x2);
    const uint64_t t = f32x2_add(f32x2_fma(rem, inv2, q0), mg2);
    tb[2 * i] = static_cast<uint32_t>(t);
    tb[2 * i + 1] = static_cast<uint32_t>(t >> 32);
  }
  return make_uint4(pack4_low_bytes(tb[0], tb[1], tb[2], tb[3]), pack4_low_bytes(tb[4], tb[5], tb[6], tb[7]),
                    pack4_low_bytes(tb[8], tb[9], tb[10], tb[11]), pack4_low_bytes(tb[12], tb[13], tb[14], tb[15]));
}

// The int8 code of 16 elements given the row's scale and inv = 1/scale
// (rounded to nearest): the corrected-quotient path, or IEEE division for
// the tiny scales where it is not covered.
__device__ __forceinline__ uint4 quant16_coded(uint4 a0, uint4 a1, float scale, float inv) {
  if (scale >= kFastScaleMin) return quant16_fast(a0, a1, scale, inv);
  return quant16(a0, a1, scale);
}

// ---- per-token FP8 E4M3 code of 16 consecutive elements ----------------------
// scale = amax / 448 (IEEE division; 448 is the largest finite E4M3 value);
// q = E4M3 round-to-nearest-even of fl(x / scale), saturated to +-448, by the
// hardware conversion cvt.rn.satfinite.e4m3x2.f32. The quotient is the same
// corrected quotient q1 as for the int8 code, with x's sign: its E4M3 code
// equals that of the IEEE quotient for every bf16 amax with amax/448 >= 2^-100
// and every bf16 x with |x| <= amax (checked exhaustively on the host, codes
// compared bit for bit, 1,044,457,888 signed pairs; 61,356 differ without the
// correction) and on the GPU by the tests.

// Two floats -> two E4M3 codes in one 16-bit word (lo in the low byte).
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint4 quant16_fp8_ieee(uint4 a0, uint4 a1, float scale) {
  const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t p0 = e4m3x2_rn_sat(__fdiv_rn(bf16_lo(w[2 * i]), scale), __fdiv_rn(bf16_hi(w[2 * i]), scale));
    const uint32_t p1 =
        e4m3x2_rn_sat(__fdiv_rn(bf16_lo(w[2 * i + 1]), scale), __fdiv_rn(bf16_hi(w[2 * i + 1]), scale));
    o[i] = p0 | (p1 << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint4 quant16_fp8_fast(uint4 a0, uint4 a1, float scale, float inv) {
  const uint64_t inv2 = f32x2_pack(__float_as_uint(inv), __float_as_uint(inv));
  const uint64_t nsc2 = f32x2_pack(__float_as_uint(-scale), __float_as_uint(-scale));
  const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  uint32_t pair[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint64_t x2 = f32x2_pack(w[i] << 16, w[i] & 0xffff0000u);
    const uint64_t q0 = f32x2_mul(x2, inv2);
    // the quotient takes the sign of x: the correction turns x = -0 into +0,
    // while fl(-0 / scale) is -0 (code 0x80); every other sign is already x's
    const uint64_t q1 = (f32x2_fma(f32x2_fma(q0, nsc2, x2), inv2, q0) & 0x7fffffff7fffffffull) |
                        (x2 & 0x8000000080000000ull);
    pair[i] = e4m3x2_rn_sat(__uint_as_float(static_cast<uint32_t>(q1)), __uint_as_float(static_cast<uint32_t>(q1 >> 32)));
  }
  return make_uint4(pair[0] | (pair[1] << 16), pair[2] | (pair[3] << 16), pair[4] | (pair[5] << 16),
                    pair[6] | (pair[7] << 16));
}

__device__ __forceinline__ uint4 quant16_fp8_coded(uint4 a0, uint4 a1, float scale, float inv) {
  if (scale >= kFastScaleMin) return quant16_fp8_fast(a0, a1, scale, inv);
  if (scale == 0.0f) return make_uint4(0, 0, 0, 0);
  return quant16_fp8_ieee(a0, a1, scale);
}

// ---- per-token 4-bit code of 16 consecutive elements -------------------------
// scale = amax / 7; q = clamp(rint(x / scale), -7, 7), two's-complement
// nibbles, the lower-indexed element in the low nibble: 16 elements -> 8
// bytes. The corrected quotient rounds like the IEEE quotient for every bf16
// amax with amax/7 >= 2^-100 and bf16 |x| <= amax (checked exhaustively on
// the host, 525,448,784 pairs), and |q| <= 7 there, so no clamp is needed.

// Low nibbles of four words (q mod 16 in bits 0-3 of each) -> 16 bits.
__device__ __forceinline__ uint32_t pack4_nibbles(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  uint32_t x = pack4_low_bytes(a, b, c, d) & 0x0F0F0F0Fu;  // nibble i in byte i
  x = (x | (x >> 4)) & 0x00FF00FFu;                          // pairs in bytes 0 and 2
  return (x | (x >> 8)) & 0xFFFFu;
}

__device__ __forceinline__ uint2 quant16_int4_fast(uint4 a0, uint4 a1, float scale, float inv) {
  const uint64_t inv2 = f32x2_pack(__float_as_uint(inv), __float_as_uint(inv));
  const uint64_t nsc2 = f32x2_pack(__float_as_uint(-scale), __float_as_uint(-scale));
  const uint64_t mg2 = f32x2_pack(0x4B400000u, 0x4B400000u);  // 1.5 * 2^23 in both halves
  const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  uint32_t tb[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint64_t x2 = f32x2_pack(w[i] << 16, w[i] & 0xffff0000u);
    const uint64_t q0 = f32x2_mul(x2, inv2);
    const uint64_t t = f32x2_add(f32x2_fma(f32x2_fma(q0, nsc2, x2), inv2, q0), mg2);
    tb[2 * i] = static_cast<uint32_t>(t);
    tb[2 * i + 1] = static_cast<uint32_t>(t >> 32);
  }
  return make_uint2(pack4_nibbles(tb[0], tb[1], tb[2], tb[3]) | (pack4_nibbles(tb[4], tb[5], tb[6], tb[7]) << 16),
                    pack4_nibbles(tb[8], tb[9], tb[10], tb[11]) | (pack4_nibbles(tb[12], tb[13], tb[14], tb[15]) << 16));
}

__device__ __forceinline__ uint2 quant16_int4_ieee(uint4 a0, uint4 a1, float scale) {
  const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  uint32_t q[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float v = h ? bf16_hi(w[i]) : bf16_lo(w[i]);
      int r = (scale == 0.0f) ? 0 : __float2int_rn(__fdiv_rn(v, scale));
      r = max(-7, min(7, r));
      q[2 * i + h] = static_cast<uint32_t>(r);
    }
  }
  return make_uint2(pack4_nibbles(q[0], q[1], q[2], q[3]) | (pack4_nibbles(q[4], q[5], q[6], q[7]) << 16),
                    pack4_nibbles(q[8], q[9], q[10], q[11]) | (pack4_nibbles(q[12], q[13], q[14], q[15]) << 16));
}

__device__ __forceinline__ uint2 quant16_int4_coded(uint4 a0, uint4 a1, float scale, float inv) {
  if (scale >= kFastScaleMin) return quant16_int4_fast(a0, a1, scale, inv);
  return quant16_int4_ieee(a0, a1, scale);
}

// Nibble i of a word (two's complement) as an exact float: 2^23 + (q ^ 8),
// built from the bits, minus 2^23 + 8.
__device__ __forceinline__ float i4_at(uint32_t w, int i) {
  return __fsub_rn(__uint_as_float(0x4B000000u | (((w >> (4 * i)) & 0xFu) ^ 0x8u)), 8388616.0f);
}

// Payload formats of the row codes.
enum PayloadFmt : int { kFmtBf16 = 0, kFmtInt8 = 1, kFmtFp8 = 2, kFmtInt4 = 3 };

// Largest code magnitude: the scale is amax / kCodeMax.
template <int FMT>
struct CodeMax;
template <>
struct CodeMax<kFmtInt8> {
  static constexpr float kValue = 127.0f;
};
template <>
struct CodeMax<kFmtFp8> {
  static constexpr float kValue = 448.0f;
};
template <>
struct CodeMax<kFmtInt4> {
  static constexpr float kValue = 7.0f;
};

template <int FMT>
__device__ __forceinline__ uint4 quant16_fmt(uint4 a0, uint4 a1, float scale, float inv) {
  if constexpr (FMT == kFmtFp8)
    return quant16_fp8_coded(a0, a1, scale, inv);
  else
    return quant16_coded(a0, a1, scale, inv);
}

// Two E4M3 codes (one 16-bit word, lo in the low byte) -> two exact floats.
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t codes16, float& lo, float& hi) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(codes16)));
  lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
  hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
}

// max |x| over 16 bf16 (two 16-byte words). With the sign bits cleared, the
// bit patterns of non-negative floats order like unsigned integers (subnormals
// included), so a per-halfword unsigned max gives the exact maximum.
__device__ __forceinline__ float absmax_bf16x16(uint4 a0, uint4 a1) {
  const uint32_t m = 0x7fff7fffu;
  uint32_t r = __vmaxu2(__vmaxu2(a0.x & m, a0.y & m), __vmaxu2(a0.z & m, a0.w & m));
  r = __vmaxu2(r, __vmaxu2(__vmaxu2(a1.x & m, a1.y & m), __vmaxu2(a1.z & m, a1.w & m)));
  const uint32_t hi = r >> 16, lo = r & 0xffffu;
  return __uint_as_float((hi > lo ? hi : lo) << 16);
}

__device__ __forceinline__ float absmax_bf16x8(uint4 a) {
  float m = fabsf(bf16_lo(a.x));
  m = fmaxf(m, fabsf(bf16_hi(a.x)));
  m = fmaxf(m, fabsf(bf16_lo(a.y)));
  m = fmaxf(m, fabsf(bf16_hi(a.y)));
  m = fmaxf(m, fabsf(bf16_lo(a.z)));
  m = fmaxf(m, fabsf(bf16_hi(a.z)));
  m = fmaxf(m, fabsf(bf16_lo(a.w)));
  m = fmaxf(m, fabsf(bf16_hi(a.w)));
  return m;
}

// The four signed int8 codes of a word, widened exactly to float without the
// conversion unit: with its sign bit flipped, byte i is q + 128, which one
// byte permute places as the low mantissa byte of 2^23 (0x4B000000), giving
// the float 2^23 + 128 + q; subtracting 2^23 + 128 leaves q exactly.
__device__ __forceinline__ void i8x4_to_f32(uint32_t w, float (&f)[4]) {
  const uint32_t b = w ^ 0x80808080u;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    f[i] = __fsub_rn(__uint_as_float(__byte_perm(b, 0x4B000000u, 0x7440u | static_cast<unsigned>(i))), 8388736.0f);
}

}  // namespace ep
