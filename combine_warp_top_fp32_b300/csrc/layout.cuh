// layout.cuh — pieces for a kernel that finishes the dispatch layout inside
// one thread-block cluster (the small-batch route+layout kernel): barriers and
// stores across the cluster's shared memory, and the expert / rank offsets.
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

// Thread-block cluster helpers (distributed shared memory). Every thread of
// every CTA of the cluster must reach each barrier (the .aligned forms).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of `p` (this CTA's shared memory) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
  const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

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
