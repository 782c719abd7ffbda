// pairs.cuh — the (token, slot) pairs of a batch, as the counting kernel reads
// them: from top-k expert ids, or from per-token expert bitmaps (the compact
// index metadata of the MoE sparse-communication article, intelliparadigm.com,
// §4.1: [bitmap, data] in place of [expert, position, data]).
//
// The layout depends only on the set of experts each token chose (rows within
// an expert are in token order), so a bitmap source enumerates a token's
// experts in increasing id order as its "slots".
#pragma once

#include <stdint.h>

namespace ep {

struct IdxPairs {
  const int32_t* idx;  // [T, k]
  int k;
  __device__ __forceinline__ int expert(int64_t t, int j) const { return idx[t * k + j]; }
  __device__ __forceinline__ bool count_ok(int64_t) const { return true; }
};

struct BitmapPairs {
  const uint32_t* bm;  // [T, W]: bit e % 32 of word e / 32 set iff the token chose e
  int W, k;
  // The j-th set bit of token t's bitmap, or -1 when it has fewer.
  __device__ __forceinline__ int expert(int64_t t, int j) const {
    const uint32_t* row = bm + t * W;
    for (int w = 0; w < W; ++w) {
      uint32_t x = row[w];
      const int c = __popc(x);
      if (j < c) {
        for (int i = 0; i < j; ++i) x &= x - 1u;
        return 32 * w + __ffs(x) - 1;
      }
      j -= c;
    }
    return -1;
  }
  // A token must have exactly k bits set.
  __device__ __forceinline__ bool count_ok(int64_t t) const {
    const uint32_t* row = bm + t * W;
    int c = 0;
    for (int w = 0; w < W; ++w) c += __popc(row[w]);
    return c == k;
  }
};

}  // namespace ep
