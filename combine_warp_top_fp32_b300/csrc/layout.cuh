// layout.cuh — the last step of the dispatch layout for a kernel that forms
// it within one CTA (the small-batch cluster kernel).
//
// From each expert's kept and dropped counts (cap already applied):
//   expert_off[e] = sum of kept counts of the experts before e  (E+1 entries),
//   rank_off[r]   = expert_off[r * E/R]                        (R+1 entries),
//   n_dropped     = sum of dropped counts.
// The NCCL EP article (§3.3) calls these the send counts' running-sum
// displacements; experts are contiguous per rank, so a rank's block starts at
// its first expert's offset.
#pragma once

#include "ep_device.cuh"

namespace ep {

// One warp (all 32 lanes call it): lane l sums experts [l*per, (l+1)*per),
// per = ceil(E/32), then a warp scan gives every expert's offset.
__device__ __forceinline__ void expert_offsets_warp(const int* kept_s, const int* drop_s, int E, int R,
                                                    int32_t* __restrict__ expert_off, int32_t* __restrict__ rank_off,
                                                    int32_t* __restrict__ n_dropped) {
  const int lane = threadIdx.x & 31;
  const int G = E / R;  // rank r starts at its first expert r*G
  const int per = (E + 31) / 32;
  const int e0 = lane * per;
  int kv = 0, dv = 0;
  for (int j = 0; j < per; ++j)
    if (e0 + j < E) {
      kv += kept_s[e0 + j];
      dv += drop_s[e0 + j];
    }
  const int ki = warp_inclusive_scan(kv);
  const int di = warp_inclusive_scan(dv);
  int run = ki - kv;
  for (int j = 0; j < per; ++j) {
    const int e = e0 + j;
    if (e < E) {
      expert_off[e] = run;
      if (e % G == 0) rank_off[e / G] = run;
      run += kept_s[e];
    }
  }
  if (lane == 31) {
    expert_off[E] = ki;
    rank_off[R] = ki;
    *n_dropped = di;
  }
}

}  // namespace ep
