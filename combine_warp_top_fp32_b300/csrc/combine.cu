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
// Design: grid-stride over tokens, one CTA per token in flight, 8 elements
// (one 16-byte bf16 load or one 8-byte int8 load) per thread and slot. The k
// row loads of a thread are issued back to back (up to 8 in flight) before
// any arithmetic, so each thread keeps up to 128 bytes of reads outstanding.
#include "ep_internal.h"

namespace ep {
namespace {

template <bool INT8>
__global__ void __launch_bounds__(1024) combine_kernel(const CombineArgs a) {
  __shared__ int32_t rows_s[2][32];
  __shared__ float w_s[2][32];
  __shared__ float sc_s[2][32];
  const int nchunk = a.H >> 3;
  // threads j < k carry slot j's row, weight (and scale) one token ahead
  auto load_slot = [&](int64_t t, int& row, float& w, float& sc) {
    const int64_t s = t * a.k + threadIdx.x;
    row = a.slot_row[s];
    if (row < -1 || static_cast<int64_t>(row) >= a.max_rows) {
      raise_status(a.status, kStatusBadIndex);
      row = -1;
    }
    w = a.topk_w[s];
    sc = 0.f;
    if constexpr (INT8) sc = row >= 0 ? a.out_scales[row] : 0.f;
  };
  int row_c = -1;
  float w_c = 0.f, sc_c = 0.f;
  if (blockIdx.x < a.T && threadIdx.x < a.k) load_slot(blockIdx.x, row_c, w_c, sc_c);
  int buf = 0;
  for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
    if (threadIdx.x < a.k) {
      rows_s[buf][threadIdx.x] = row_c;
      w_s[buf][threadIdx.x] = w_c;
      if constexpr (INT8) sc_s[buf][threadIdx.x] = sc_c;
      const int64_t tn = t + gridDim.x;
      if (tn < a.T) load_slot(tn, row_c, w_c, sc_c);
    }
    __syncthreads();
    for (int c = threadIdx.x; c < nchunk; c += blockDim.x) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      for (int j0 = 0; j0 < a.k; j0 += 8) {
        const int nj = min(8, a.k - j0);
        if constexpr (INT8) {
          uint2 v[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            v[jj] = make_uint2(0, 0);
            const int row = jj < nj ? rows_s[buf][j0 + jj] : -1;
            if (row >= 0) v[jj] = ld_stream_v2(static_cast<const int8_t*>(a.expert_out) +
                                               static_cast<int64_t>(row) * a.H + 8 * c);
          }
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int row = jj < nj ? rows_s[buf][j0 + jj] : -1;
            if (row >= 0) {
              const float w = w_s[buf][j0 + jj];
              const float sc = sc_s[buf][j0 + jj];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                acc[i] = __fmaf_rn(w, __fmul_rn(i8_at(v[jj].x, i), sc), acc[i]);
                acc[4 + i] = __fmaf_rn(w, __fmul_rn(i8_at(v[jj].y, i), sc), acc[4 + i]);
              }
            }
          }
        } else {
          uint4 v[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            v[jj] = make_uint4(0, 0, 0, 0);
            const int row = jj < nj ? rows_s[buf][j0 + jj] : -1;
            if (row >= 0)
              v[jj] = ld_stream_v4(static_cast<const char*>(a.expert_out) +
                                   (static_cast<int64_t>(row) * a.H + 8 * c) * 2);
          }
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int row = jj < nj ? rows_s[buf][j0 + jj] : -1;
            if (row >= 0) {
              const float w = w_s[buf][j0 + jj];
              acc[0] = __fmaf_rn(w, bf16_lo(v[jj].x), acc[0]);
              acc[1] = __fmaf_rn(w, bf16_hi(v[jj].x), acc[1]);
              acc[2] = __fmaf_rn(w, bf16_lo(v[jj].y), acc[2]);
              acc[3] = __fmaf_rn(w, bf16_hi(v[jj].y), acc[3]);
              acc[4] = __fmaf_rn(w, bf16_lo(v[jj].z), acc[4]);
              acc[5] = __fmaf_rn(w, bf16_hi(v[jj].z), acc[5]);
              acc[6] = __fmaf_rn(w, bf16_lo(v[jj].w), acc[6]);
              acc[7] = __fmaf_rn(w, bf16_hi(v[jj].w), acc[7]);
            }
          }
        }
      }
      uint4 out;
      out.x = pack_bf16x2_rn(acc[0], acc[1]);
      out.y = pack_bf16x2_rn(acc[2], acc[3]);
      out.z = pack_bf16x2_rn(acc[4], acc[5]);
      out.w = pack_bf16x2_rn(acc[6], acc[7]);
      st_v4(static_cast<char*>(a.y) + (t * a.H + 8 * c) * 2, out);
    }
    buf ^= 1;
  }
}

// One row per CTA iteration; 16 elements per thread; same code as dispatch.
__global__ void __launch_bounds__(1024) quantize_rows_kernel(const void* __restrict__ in, int64_t n, int H,
                                                              int8_t* __restrict__ q, float* __restrict__ scales) {
  __shared__ float amax_s[2][32];
  const int c = threadIdx.x;
  const bool on = c < (H >> 4);
  const int warp = c >> 5, lane = c & 31, nw = blockDim.x >> 5;
  int buf = 0;
  for (int64_t t = blockIdx.x; t < n; t += gridDim.x) {
    uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0;
    if (on) {
      const char* p = static_cast<const char*>(in) + (t * H + 16 * c) * 2;
      a0 = ld_stream_v4(p);
      a1 = ld_stream_v4(p + 16);
    }
    float m = on ? fmaxf(absmax_bf16x8(a0), absmax_bf16x8(a1)) : 0.f;
    m = warp_max(m);
    if (lane == 0) amax_s[buf][warp] = m;
    __syncthreads();
    float am = amax_s[buf][0];
    for (int i = 1; i < nw; ++i) am = fmaxf(am, amax_s[buf][i]);
    const float scale = __fdiv_rn(am, 127.0f);
    if (on) st_v4(q + t * H + 16 * c, quant16(a0, a1, scale));
    if (c == 0) scales[t] = scale;
    buf ^= 1;
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int sms, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const int nchunk = a.H / 8;
  int block = ((nchunk + 31) / 32) * 32;
  if (block > 1024) block = 1024;
  const int per_sm = 2048 / block;
  const int64_t want = static_cast<int64_t>(sms) * per_sm;
  const int grid = static_cast<int>(a.T < want ? a.T : want);
  if (a.int8_out)
    combine_kernel<true><<<grid, block, 0, s>>>(a);
  else
    combine_kernel<false><<<grid, block, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const void* in, int64_t n, int H, int8_t* q, float* scales, int sms,
                                 cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int block = ((H / 16 + 31) / 32) * 32;
  const int per_sm = 2048 / block;
  const int64_t want = static_cast<int64_t>(sms) * per_sm;
  const int grid = static_cast<int>(n < want ? n : want);
  quantize_rows_kernel<<<grid, block, 0, s>>>(in, n, H, q, scales);
  return cudaGetLastError();
}

}  // namespace ep
