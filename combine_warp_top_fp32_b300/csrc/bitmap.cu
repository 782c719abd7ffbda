// bitmap.cu — compact routing metadata: per-token expert bitmaps in place of
// explicit (expert, position) pairs (MoE sparse-communication article,
// intelliparadigm.com, §4.1: [expert, pos, data] becomes [bitmap, data]).
//
// encode  one thread per (token, 32-expert word): the bits of the token's
//         top-k ids that fall in the word (a repeated or out-of-range id sets
//         the status word instead).
// layout  what a receiving rank rebuilds from bitmaps alone: the counting
//         kernel reads each token's experts from its bitmap (increasing id
//         order; the layout does not depend on slot order, since rows within
//         an expert are in token order), the scan applies the capacity and
//         the offsets, and one thread per pair writes row_token[row] = t: the
//         source token of every row of the rank-major buffer, the same rows
//         ep_dispatch writes (row_slot[row] / k).
#include "ep_internal.h"
#include "pairs.cuh"

namespace ep {
namespace {

__global__ void __launch_bounds__(256) encode_bitmap_kernel(const int32_t* __restrict__ idx, int64_t T, int E, int k,
                                                            int W, uint32_t* __restrict__ bitmap, uint32_t* status) {
  pdl_wait();  // the expert ids come from the kernel before this one
  pdl_launch_dependents();
  const int64_t n = T * W;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / W;
    const int w = static_cast<int>(i - t * W);
    uint32_t word = 0;
    for (int j = 0; j < k; ++j) {
      const int e = idx[t * k + j];
      if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
        if (w == 0) raise_status(status, kStatusBadIndex);
        continue;
      }
      if ((e >> 5) != w) continue;
      const uint32_t bit = 1u << (e & 31);
      if (word & bit) raise_status(status, kStatusBadIndex);  // expert repeated within one token
      word |= bit;
    }
    bitmap[i] = word;
  }
}

// row_token[row] = t for every kept pair (after the count and scan kernels).
__global__ void __launch_bounds__(256) row_token_kernel(const BitmapPairs src, const int32_t* __restrict__ lrank,
                                                        const int32_t* __restrict__ tile_base,
                                                        const int32_t* __restrict__ expert_off, int64_t npairs,
                                                        int E, int k, int tile_log2, int ntiles, int cap,
                                                        int32_t* __restrict__ row_token) {
  pdl_wait();  // ranks, tile bases and offsets come from the kernels before
  pdl_launch_dependents();
  for (int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p < npairs;
       p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = p / k;
    const int e = src.expert(t, static_cast<int>(p - t * k));
    const int lr = lrank[p];
    if (static_cast<unsigned>(e) >= static_cast<unsigned>(E) || lr < 0) continue;
    const int pos = tile_base[static_cast<int64_t>(e) * ntiles + (t >> tile_log2)] + lr;
    if (pos < cap) row_token[expert_off[e] + pos] = static_cast<int32_t>(t);
  }
}

}  // namespace

cudaError_t launch_encode_bitmap(const int32_t* idx, int64_t T, int E, int k, uint32_t* bitmap, uint32_t* status,
                                 int sms, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int W = (E + 31) / 32;
  const int64_t n = T * W;
  const int64_t blocks = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  return launch_pdl(encode_bitmap_kernel, static_cast<int>(blocks < cap ? blocks : cap), 256, 0, s, idx, T, E, k, W,
                    bitmap, status);
}

cudaError_t launch_bitmap_layout(const DispatchArgs& a, const uint32_t* bitmap, int32_t* row_token, int sms,
                                 cudaStream_t s) {
  const int W = (a.E + 31) / 32;
  cudaError_t err = launch_layout_from_bitmap(a, bitmap, W, s);
  if (err != cudaSuccess || a.T == 0) return err;
  const int64_t npairs = static_cast<int64_t>(a.T) * a.k;
  const int64_t blocks = (npairs + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  const int tile_log2 = __builtin_ctz(static_cast<unsigned>(a.tile));
  return launch_pdl(row_token_kernel, static_cast<int>(blocks < cap ? blocks : cap), 256, 0, s,
                    BitmapPairs{bitmap, W, a.k}, a.lrank, a.tile_base, a.expert_off, npairs, a.E, a.k, tile_log2,
                    a.ntiles, a.cap, row_token);
}

}  // namespace ep
