// combine.cu — weighted top-k recombination of expert outputs, and the
// stand-alone per-row int8 code for an expert side that returns int8.
//
// The combine is step 4 of the EP flow in ThunderEP on consumer GPUs
// (bjdmk.com.cn, §1.3): each token's expert results come back to its source
// card, which takes the gate-weighted sum. Here, per token t and element h:
//   acc = 0; for j = 0..k-1 (slot order, dropped slots skipped):
//     v = float(bf16 row)  or  (float)q * scale   (one fp32 multiply)
//     acc = fmaf(w[t,j], v, acc)
//   y[t,h] = bf16 round-to-nearest-even(acc)
// The fixed slot order and the explicit fma make the result reproducible.
//
// Design: one warp per work unit in flight (a token, or a slice of a token's
// row when the batch is short), no block-level synchronisation.
//   - lanes j < k read slot j's row, weight (and int8 scale) one token ahead;
//   - a ballot drops the dropped slots and the kept ones are gathered, in
//     slot order, into registers of every lane (row address, weight, scale),
//     so a token with few kept slots costs only their loads;
//   - the row is walked in 16-byte chunks per lane (8 bf16, 16 int8 / E4M3
//     or 32 int4 elements); the loads of all kept slots for several chunks
//     are issued back to back before any arithmetic, a fixed number per lane
//     in flight whatever the number of kept slots (bf16: 16 = 2 slots x 8
//     chunks, 4 x 4 or 8 x 2; coded rows: 8);
//   - the arithmetic runs on packed pairs of elements (f32x2), and coded
//     rows are widened by integer operations, not the conversion unit;
//   - more than 8 kept slots (k > 8) are taken in groups of 8 in slot order,
//     with the accumulators carried across groups, so the order of the fmas is
//     the same in every case.
#include "ep_internal.h"

namespace ep {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Elements of one 16-byte chunk: 8 bf16, 16 int8 / E4M3 codes or 32 int4 codes.
template <int FMT>
struct Chunk {
  static constexpr int kElems = FMT == kFmtBf16 ? 8 : (FMT == kFmtInt4 ? 32 : 16);
};

// Float whose low mantissa byte is byte i of b: 2^23 + byte (a byte permute).
__device__ __forceinline__ uint32_t magic_byte(uint32_t b, int i) {
  return __byte_perm(b, 0x4B000000u, 0x7440u | static_cast<unsigned>(i));
}

__device__ __forceinline__ uint64_t splat2(float v) { return f32x2_pack(__float_as_uint(v), __float_as_uint(v)); }

// acc[0..EL/2) += w * v for one 16-byte chunk of a kept row: the accumulators
// are packed pairs of consecutive elements (element 2j in the low half) and
// every step is a packed add / mul / fma .rn.f32x2, the same IEEE operation
// per element as its scalar form: fmaf(w, v, acc) with v = float(bf16), or
// v = (float)code * scale with the code widened exactly by integer operations
// only (no conversion unit):
//   bf16:  the halfword shifted into the top of a float;
//   int8:  byte ^ 0x80 = q + 128 as the low byte of 2^23, minus 2^23 + 128;
//   int4:  nibble ^ 8 = q + 8 (bytes of lo/hi nibbles), minus 2^23 + 8;
//   E4M3:  the code's exponent and mantissa moved to float bits 20..26 and its
//          sign to bit 31 is the value times 2^-120 (subnormal codes land on
//          float subnormals), scaled back by 2^120 exactly. The NaN codes 0x7F
//          / 0xFF, which no encoder here writes, read as +-480.
template <int FMT>
__device__ __forceinline__ void fma_chunk(uint64_t* acc, uint4 v, uint64_t w2, uint64_t s2) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
  if constexpr (FMT == kFmtBf16) {
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = f32x2_fma(w2, f32x2_pack(u[q] << 16, u[q] & 0xffff0000u), acc[q]);
  } else if constexpr (FMT == kFmtInt8) {
    const uint64_t c2 = splat2(-8388736.0f);  // -(2^23 + 128)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t b = u[q] ^ 0x80808080u;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint64_t f2 = f32x2_pack(magic_byte(b, 2 * j), magic_byte(b, 2 * j + 1));
        acc[2 * q + j] = f32x2_fma(w2, f32x2_mul(f32x2_add(f2, c2), s2), acc[2 * q + j]);
      }
    }
  } else if constexpr (FMT == kFmtInt4) {
    const uint64_t c2 = splat2(-8388616.0f);  // -(2^23 + 8)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t lo = (u[q] & 0x0F0F0F0Fu) ^ 0x08080808u;         // nibbles 0, 2, 4, 6
      const uint32_t hi = ((u[q] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;  // nibbles 1, 3, 5, 7
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t f2 = f32x2_pack(magic_byte(lo, j), magic_byte(hi, j));
        acc[4 * q + j] = f32x2_fma(w2, f32x2_mul(f32x2_add(f2, c2), s2), acc[4 * q + j]);
      }
    }
  } else {  // E4M3
    const uint64_t e2 = f32x2_pack(0x7B800000u, 0x7B800000u);  // 2^120
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)  // byte i to the top, then an arithmetic shift by 4
        r[i] = static_cast<uint32_t>(static_cast<int32_t>(u[q] << (24 - 8 * i)) >> 4) & 0x87F00000u;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint64_t f2 = f32x2_mul(f32x2_pack(r[2 * j], r[2 * j + 1]), e2);
        acc[2 * q + j] = f32x2_fma(w2, f32x2_mul(f2, s2), acc[2 * q + j]);
      }
    }
  }
}

// Round EL fp32 accumulators (EL/2 packed pairs) to bf16 (RNE) and store them
// at y (16-byte aligned).
template <int EL>
__device__ __forceinline__ void store_bf16(char* y, const uint64_t* acc) {
#pragma unroll
  for (int s = 0; s < EL / 8; ++s) {
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = pack_bf16x2_rn(__uint_as_float(static_cast<uint32_t>(acc[4 * s + j])),
                            __uint_as_float(static_cast<uint32_t>(acc[4 * s + j] >> 32)));
    st_v4(y + 16 * s, make_uint4(o[0], o[1], o[2], o[3]));
  }
}

// Gathers the next (up to) 8 kept slots of `mask` (lowest slot first) from the
// lanes that hold them into registers of every lane; returns how many.
template <int FMT>
__device__ __forceinline__ int gather_group(unsigned& mask, int row, float w, float sc, const char* base,
                                            int64_t row_bytes, const char* (&p)[8], float (&wv)[8],
                                            float (&sv)[8]) {
  int n = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int src = mask ? __ffs(mask) - 1 : 0;  // uniform across the warp
    const int r = __shfl_sync(kFull, row, src);
    wv[i] = __shfl_sync(kFull, w, src);
    if constexpr (FMT != kFmtBf16) sv[i] = __shfl_sync(kFull, sc, src);
    p[i] = base + static_cast<int64_t>(r < 0 ? 0 : r) * row_bytes;
    if (mask) ++n;
    mask &= mask - 1u;
  }
  return n;
}

// One token's chunks with at most NS kept slots (gathered in p/wv/sv): UNR
// chunks per lane per pass, all NS*UNR loads issued before any arithmetic.
template <int FMT, int NS, int UNR>
__device__ __forceinline__ void combine_token(int nk, int cbeg, int nchunk, int lane, const char* const (&p)[8],
                                              const float (&wv)[8], const float (&sv)[8], char* yrow) {
  constexpr int EL = Chunk<FMT>::kElems;
  uint64_t w2[NS], s2[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    w2[i] = splat2(wv[i]);
    s2[i] = splat2(sv[i]);
  }
  for (int c0 = cbeg + lane; c0 < nchunk; c0 += 32 * UNR) {
    uint4 v[UNR][NS];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int c = c0 + 32 * u;
#pragma unroll
      for (int i = 0; i < NS; ++i)
        v[u][i] = (i < nk && c < nchunk) ? ld_stream_v4(p[i] + 16 * static_cast<int64_t>(c)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int c = c0 + 32 * u;
      uint64_t acc[EL / 2];
#pragma unroll
      for (int e = 0; e < EL / 2; ++e) acc[e] = 0ull;
#pragma unroll
      for (int i = 0; i < NS; ++i)
        if (i < nk) fma_chunk<FMT>(acc, v[u][i], w2[i], s2[i]);
      if (c < nchunk) store_bf16<EL>(yrow + 2 * static_cast<int64_t>(c) * EL, acc);
    }
  }
}

// LOADS = 16-byte loads in flight per lane: a token with few kept slots walks
// more chunks per pass, so the bytes in flight do not shrink with drops.
// int8 and E4M3 rows spend more instructions per byte than bf16 (widening,
// the scale): they run 8 loads per lane with three CTAs per SM, which hides
// the arithmetic better than 16 loads with two (int8 84.9 -> 74.8 us, E4M3
// 121.8 -> 84.1 us on the capacity combine); int4 (32 elements per chunk)
// keeps two.
template <int FMT>
constexpr int combine_min_ctas() {
  return (FMT == kFmtInt8 || FMT == kFmtFp8) ? 3 : 2;
}

template <int FMT, int LOADS>
__global__ void __launch_bounds__(256, combine_min_ctas<FMT>()) combine_kernel(const CombineArgs a) {
  constexpr int EL = Chunk<FMT>::kElems;
  constexpr bool kCoded = FMT != kFmtBf16;
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int nchunk = a.H / EL;
  const int64_t row_bytes = static_cast<int64_t>(a.H) * (FMT == kFmtBf16 ? 2 : 1) / (FMT == kFmtInt4 ? 2 : 1);
  const char* base = static_cast<const char*>(a.expert_out);
  pdl_wait();  // slot rows, weights and expert outputs come from earlier kernels
  pdl_launch_dependents();

  // lane j < k: slot j of token t (row, weight, scale); -1 / 0 elsewhere
  auto load_slot = [&](int64_t t, int& row, float& w, float& sc) {
    row = -1;
    w = 0.f;
    sc = 0.f;
    if (t < a.T && lane < a.k) {
      const int64_t s = t * a.k + lane;
      row = a.slot_row[s];
      if (row < -1 || static_cast<int64_t>(row) >= a.max_rows) {
        raise_status(a.status, kStatusBadIndex);
        row = -1;
      }
      w = a.topk_w[s];
      if constexpr (kCoded) sc = row >= 0 ? a.out_scales[row] : 0.f;
    }
  };

  // Work unit u = (token u / ns, slice u % ns): slice s covers the 16-byte
  // chunks [s * cslice, (s + 1) * cslice) of the token's row, so that short
  // batches still spread over every warp and long ones end with a small tail.
  const int ns = a.slices;
  const int cslice = (nchunk + ns - 1) / ns;
  const int64_t units = static_cast<int64_t>(a.T) * ns;
  // A warp's units: warp0, warp0 + nwarps, ... (the static order); for bf16
  // rows with a.counter set (few units a warp: see the launcher) only the
  // first a.static_rounds of them, then static_end + the next value of a
  // shared counter, asked for while the next unit's slots load, so that the
  // warps finish together instead of in a ragged last round. Each unit's
  // slots are loaded one unit ahead.
  unsigned* const ctr = FMT == kFmtBf16 ? a.counter : nullptr;
  const int64_t static_end = static_cast<int64_t>(a.static_rounds) * nwarps;  // units taken in the static order
  auto claim = [&](int64_t after) -> int64_t {
    const int64_t next = after + nwarps;
    if (!ctr || next < static_end) return next;
    unsigned v = 0u;
    if (lane == 0) v = atomicAdd(ctr, 1u);
    return static_end + static_cast<int64_t>(__shfl_sync(kFull, v, 0));
  };
  int row_n, row;
  float w_n, sc_n, w, sc;
  int64_t u = warp0;
  int64_t u1 = claim(warp0);  // the next unit
  load_slot(warp0 / ns, row_n, w_n, sc_n);
  while (u < units) {
    const int64_t t = u / ns;
    const int cbeg = static_cast<int>(u - t * ns) * cslice;
    const int cend = min(nchunk, cbeg + cslice);
    row = row_n;
    w = w_n;
    sc = sc_n;
    load_slot(u1 / ns, row_n, w_n, sc_n);  // the next unit's slots, one unit ahead
    const int64_t u2 = u1 < units ? claim(u1) : units;

    const unsigned kept = __ballot_sync(kFull, row >= 0);
    const int nk = __popc(kept);
    char* yrow = static_cast<char*>(a.y) + t * 2 * static_cast<int64_t>(a.H);
    const char* p[8];
    float wv[8], sv[8];
    if (nk <= 8) {
      unsigned m = kept;
      gather_group<FMT>(m, row, w, sc, base, row_bytes, p, wv, sv);
      // coded rows: no separate 2-slot body (each body is long; fewer of
      // them keep the instruction cache warm: int4 92 -> 74 us, E4M3 84 ->
      // 80 us on the capacity combine)
      if (FMT == kFmtBf16 && nk <= 2)
        combine_token<FMT, 2, LOADS / 2>(nk, cbeg, cend, lane, p, wv, sv, yrow);
      else if (nk <= 4)
        combine_token<FMT, 4, LOADS / 4>(nk, cbeg, cend, lane, p, wv, sv, yrow);
      else
        combine_token<FMT, 8, LOADS / 8>(nk, cbeg, cend, lane, p, wv, sv, yrow);
    } else {
      // k > 8 with more than 8 kept slots: groups of 8 per chunk, slot order.
      // The loop bound is warp-uniform: the gathers shuffle across all lanes.
      for (int c0 = cbeg; c0 < cend; c0 += 32) {
        const int c = c0 + lane;
        uint64_t acc[EL / 2];
#pragma unroll
        for (int e = 0; e < EL / 2; ++e) acc[e] = 0ull;
        unsigned m = kept;
        while (m) {
          const int n = gather_group<FMT>(m, row, w, sc, base, row_bytes, p, wv, sv);
          uint4 v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            v[i] = (i < n && c < cend) ? ld_stream_v4(p[i] + 16 * static_cast<int64_t>(c)) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i < n) fma_chunk<FMT>(acc, v[i], splat2(wv[i]), splat2(sv[i]));
        }
        if (c < cend) store_bf16<EL>(yrow + 2 * static_cast<int64_t>(c) * EL, acc);
      }
    }
    u = u1;
    u1 = u2;
  }
  if (!ctr) return;
  if (lane == 0) {
    // the last warp to finish puts the counter back at zero for the next call;
    // every warp's claims come before its arrival here (release), and the last
    // one sees them all (acquire) before it resets
    unsigned* done = ctr + 1;
    unsigned prev;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(prev) : "l"(done) : "memory");
    if (prev == static_cast<unsigned>(nwarps) - 1u) {
      *reinterpret_cast<volatile unsigned*>(ctr) = 0u;
      *reinterpret_cast<volatile unsigned*>(done) = 0u;
    }
  }
}

// One row per CTA iteration; 16 elements per thread; the same code as the
// dispatch (int8: scale = amax/127; FP8 E4M3: amax/448; int4: amax/7, rows of
// H/2 bytes).
template <int FMT>
__global__ void __launch_bounds__(1024) quantize_rows_kernel(const void* __restrict__ in, int64_t n, int H,
                                                              uint8_t* __restrict__ q, float* __restrict__ scales) {
  __shared__ float amax_s[2][32];
  const int c = threadIdx.x;
  const bool on = c < (H >> 4);
  const int warp = c >> 5, lane = c & 31, nw = blockDim.x >> 5;
  pdl_wait();
  pdl_launch_dependents();
  int buf = 0;
  for (int64_t t = blockIdx.x; t < n; t += gridDim.x) {
    uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0;
    if (on) {
      const char* p = static_cast<const char*>(in) + (t * H + 16 * c) * 2;
      a0 = ld_stream_v4(p);
      a1 = ld_stream_v4(p + 16);
    }
    float m = on ? absmax_bf16x16(a0, a1) : 0.f;
    m = warp_max(m);
    if (lane == 0) amax_s[buf][warp] = m;
    __syncthreads();
    float am = amax_s[buf][0];
    for (int i = 1; i < nw; ++i) am = fmaxf(am, amax_s[buf][i]);
    const float scale = __fdiv_rn(am, CodeMax<FMT>::kValue);
    if constexpr (FMT == kFmtInt4) {
      if (on) st_v2(q + t * (H / 2) + 8 * c, quant16_int4_coded(a0, a1, scale, __frcp_rn(scale)));
    } else {
      if (on) st_v4(q + t * H + 16 * c, quant16_fmt<FMT>(a0, a1, scale, __frcp_rn(scale)));
    }
    if (c == 0) scales[t] = scale;
    buf ^= 1;
  }
}

}  // namespace

namespace {

int g_occ_combine[8][64];

constexpr int64_t kDynamicUnits = 4;  // units per warp taken from the shared counter at the end

template <int FMT, int LOADS>
cudaError_t launch_combine_t(CombineArgs a, int sms, int* cache, cudaStream_t s) {
  constexpr int kBlock = 256;
  const int per_sm = resident_ctas(combine_kernel<FMT, LOADS>, kBlock, 0, cache);
  const int64_t warps = static_cast<int64_t>(sms) * per_sm * (kBlock / 32);
  // Slices per token: enough work units for about eight per warp, but no
  // slice shorter than one pass of the warp over its chunks.
  const int nchunk = a.H / Chunk<FMT>::kElems;
  const int min_slice = 32 * (LOADS / 8);
  int ns = static_cast<int>((8 * warps + a.T - 1) / a.T);
  const int max_ns = nchunk / min_slice > 1 ? nchunk / min_slice : 1;
  a.slices = ns < 1 ? 1 : (ns > max_ns ? max_ns : ns);
  const int64_t units = static_cast<int64_t>(a.T) * a.slices;
  const int64_t blocks_needed = (units + kBlock / 32 - 1) / (kBlock / 32);
  const int64_t want = static_cast<int64_t>(sms) * per_sm;
  const int grid = static_cast<int>(blocks_needed < want ? blocks_needed : want);
  // A shared unit counter (bf16 rows only) when each warp has 4 to 31 units
  // and a unit moves at least 16 KB (its upper bound: k rows of the slice plus
  // the slice of y), so that the static order's ragged last round is worth an
  // atomic per unit and the counter sees fewer than ~0.4 claims per ns.
  // Measured: capacity (14 units a warp, <= 36 KB) 191.4 -> 189.0 us a step;
  // prefill-mid (9 units, <= 6 KB) 41.9 -> 45.4 us with it; large (55 units)
  // lost 2 %; the coded rows' combines lost 2-4 %.
  const int64_t per_warp = units / (static_cast<int64_t>(grid) * (kBlock / 32));
  const int64_t unit_bytes = (static_cast<int64_t>(a.k) * a.H * 2 + static_cast<int64_t>(a.H) * 2) / a.slices;
  if (FMT != kFmtBf16 || per_warp < 4 || per_warp >= 32 || unit_bytes < 16 * 1024) a.counter = nullptr;
  // with the counter, the first units of each warp still follow the static
  // order (no atomic) and only about the last kDynamicUnits are shared
  a.static_rounds = static_cast<int>(per_warp > kDynamicUnits ? per_warp - kDynamicUnits : 1);
  return launch_pdl(combine_kernel<FMT, LOADS>, grid, kBlock, 0, s, a);
}

template <int FMT>
cudaError_t launch_combine_fmt(const CombineArgs& a, int sms, cudaStream_t s) {
  // bf16: 16 loads in flight per lane once a row is long enough to keep them
  // busy; coded rows: 8 (see combine_kernel)
  if constexpr (FMT == kFmtBf16) {
    if (a.H / Chunk<FMT>::kElems >= 64) return launch_combine_t<FMT, 16>(a, sms, g_occ_combine[2 * FMT], s);
  }
  return launch_combine_t<FMT, 8>(a, sms, g_occ_combine[2 * FMT + 1], s);
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int sms, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  if (a.out_fmt == kFmtInt4) return launch_combine_fmt<kFmtInt4>(a, sms, s);
  if (a.out_fmt == kFmtFp8) return launch_combine_fmt<kFmtFp8>(a, sms, s);
  if (a.out_fmt == kFmtInt8) return launch_combine_fmt<kFmtInt8>(a, sms, s);
  return launch_combine_fmt<kFmtBf16>(a, sms, s);
}

cudaError_t launch_quantize_rows(const void* in, int64_t n, int H, int fmt, void* q, float* scales, int sms,
                                 cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int block = ((H / 16 + 31) / 32) * 32;
  static int occ[3][32][64];  // per format, block size / 32 and device
  auto go = [&](auto kernel, int which) {
    const int per_sm = resident_ctas(kernel, block, 0, occ[which][block / 32 - 1]);
    const int64_t want = static_cast<int64_t>(sms) * per_sm;
    const int grid = static_cast<int>(n < want ? n : want);
    return launch_pdl(kernel, grid, block, 0, s, in, n, H, static_cast<uint8_t*>(q), scales);
  };
  if (fmt == kFmtInt4) return go(quantize_rows_kernel<kFmtInt4>, 2);
  return fmt == kFmtFp8 ? go(quantize_rows_kernel<kFmtFp8>, 1) : go(quantize_rows_kernel<kFmtInt8>, 0);
}

}  // namespace ep
