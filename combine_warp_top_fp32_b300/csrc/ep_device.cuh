// ep_device.cuh — device helpers shared by the libep_b300 kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ep {

// Bits of the workspace status word (sticky until ep_get_error clears them).
constexpr uint32_t kStatusBadIndex = 1u;
constexpr uint32_t kStatusTimeout = 2u;

__device__ __forceinline__ void raise_status(uint32_t* status, uint32_t bit) {
  atomicOr(status, bit);
}

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

// Signed int8 byte i of a word, widened exactly to float.
__device__ __forceinline__ float i8_at(uint32_t w, int i) {
  return static_cast<float>(static_cast<int8_t>((w >> (8 * i)) & 0xffu));
}

}  // namespace ep
