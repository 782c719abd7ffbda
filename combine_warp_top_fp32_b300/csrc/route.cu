// route.cu — the routing kernels: top-k gating with softmax weights over
// fp32 logits (the per-token steps are in route_device.cuh).
//
// Kernels: route_topk_kernel (ep_route: routing alone, a grid-stride loop
// over tokens); route_count_kernel (ep_route_dispatch: one CTA per tile of
// tokens routes the tile and writes its per-expert counts and in-tile ranks,
// the dispatch's count step); route_layout_cluster_kernel (ep_route_dispatch
// on batches of at most eight 32-token tiles: one thread-block cluster routes
// the batch and forms the whole layout, the count and scan steps together).
#include "ep_internal.h"
#include "layout.cuh"
#include "route_device.cuh"

namespace ep {
namespace {

using namespace routing;

template <int VPL, bool VEC4>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int lanes_log2, int renorm, int32_t* __restrict__ topk_idx,
                                                         float* __restrict__ topk_w) {
  const int L = 1 << lanes_log2;
  const int lane = threadIdx.x & 31;
  const int sub = lane & (L - 1);
  const int groups_per_warp = 32 >> lanes_log2;
  const int grp = lane >> lanes_log2;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  pdl_wait();  // the logits may come from the kernel before this one
  pdl_launch_dependents();

  if constexpr (VPL <= 8) {
    if (L == 32) {  // tokens w, w + n_warps, ...: NQ per warp at once, the next ones' logits loaded meanwhile
      constexpr int NQ = VPL <= 4 ? 2 : 1;
      route_warp<NQ, VPL, VEC4>(logits, 0, warp_id, NQ * n_warps, n_warps, T, E, k, lane, renorm,
                                [&](int64_t, int64_t t, int e, float w) {
                                  topk_idx[t * k + lane] = e;
                                  topk_w[t * k + lane] = w;
                                });
      return;
    }
  }
  for (int64_t tb = warp_id * groups_per_warp; tb < T; tb += n_warps * groups_per_warp) {
    const int64_t t = tb + grp;
    const bool active = t < T;
    int e;
    float w;
    route_token<VPL, VEC4>(logits, t, active, E, k, L, sub, renorm, &e, &w);
    if (active && sub < k) {
      topk_idx[t * k + sub] = e;
      topk_w[t * k + sub] = w;
    }
  }
}

// Routing fused with the per-tile count of the dispatch (the ThunderEP
// article's §5.2 suggestion to bucket by destination while routing): CTA b
// routes the tokens of tile b = [b*tile, (b+1)*tile), writes their slots,
// and builds the tile's per-expert bit masks in shared memory, from which it
// writes the tile's count per expert and each pair's rank within the tile in
// token order (the same tile_counts / lrank as the dispatch's count kernel).
template <int VPL, bool VEC4>
__global__ void __launch_bounds__(VPL >= 16 ? 256 : 512) route_count_kernel(
    const float* __restrict__ logits, int T, int E, int k, int lanes_log2, int renorm, int tile, int ntiles,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ tile_counts,
    int32_t* __restrict__ lrank, uint32_t* ticket) {
  extern __shared__ uint32_t smem[];
  const int TW = tile >> 5;
  uint32_t* mask = smem;          // [E][TW] bit b of word w: token 32*w+b of the tile chose e
  uint32_t* pre = smem + E * TW;  // [E][TW] set bits of e in the words before w
  const int b = blockIdx.x;
  const int64_t t0 = static_cast<int64_t>(b) * tile;
  const int nt = static_cast<int>(min(static_cast<int64_t>(tile), T - t0));
  for (int i = threadIdx.x; i < E * TW; i += blockDim.x) mask[i] = 0u;
  pdl_wait();  // the logits may come from the kernel before this one
  pdl_launch_dependents();
  if (b == 0 && threadIdx.x == 0) *ticket = 0u;  // the scan that follows counts its CTAs from 0
  __syncthreads();
  if (nt <= 0) return;  // an empty batch: only the ticket
  route_tile<VPL, VEC4>(logits, t0, nt, E, k, lanes_log2, renorm, TW, mask, topk_idx, topk_w);
  __syncthreads();

  tile_word_prefix(mask, pre, E, TW, tile_counts, ntiles, b);
  __syncthreads();

  const int64_t base = t0 * k;
  for (int p = threadIdx.x; p < nt * k; p += blockDim.x) {
    const int e = topk_idx[base + p];  // written above by this CTA
    const int tl = p / k;
    const int w = tl >> 5;
    lrank[base + p] = static_cast<int>(pre[e * TW + w]) + __popc(mask[e * TW + w] & ((1u << (tl & 31)) - 1u));
  }
}

// Small batches (at most kClusterTiles tiles of 32 tokens): one cluster of
// one CTA per tile, a warp per token. Each CTA routes its tile and ranks its
// pairs as route_count_kernel does, but pushes its per-expert tile counts
// into CTA 0's shared memory instead of global memory; after a cluster
// barrier CTA 0 alone forms what the scan kernel would from them (tile bases,
// raw and kept counts, expert and rank offsets, the number dropped), so the
// whole layout costs one launch. The outputs are those of route_count_kernel
// + scan_kernel, bit for bit.
template <int VPL, bool VEC4>
__global__ void __launch_bounds__(1024, 1) route_layout_cluster_kernel(
    const float* __restrict__ logits, int T, int E, int k, int lanes_log2, int renorm, int R, int cap,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ lrank,
    int32_t* __restrict__ tile_base, int32_t* __restrict__ expert_counts, int32_t* __restrict__ expert_raw,
    int32_t* __restrict__ expert_off, int32_t* __restrict__ rank_off, int32_t* __restrict__ n_dropped) {
  extern __shared__ uint32_t smem[];
  const int C = gridDim.x;  // tiles = CTAs = the cluster
  uint32_t* mask = smem;                                // [E] this tile's word per expert
  int* counts_s = reinterpret_cast<int*>(smem + E);    // [E][C] (CTA 0) every tile's count per expert
  int* kept_s = counts_s + E * C;                      // [E] (CTA 0)
  int* drop_s = kept_s + E;                            // [E] (CTA 0)
  const int warp = threadIdx.x >> 5;
  const int b = blockIdx.x;
  const int64_t t0 = static_cast<int64_t>(b) * 32;
  const int nt = min(32, T - static_cast<int>(t0));  // >= 1: the grid has ceil(T/32) CTAs
  for (int i = threadIdx.x; i < E; i += blockDim.x) mask[i] = 0u;
  cluster_arrive_relaxed();  // CTA 0 must be running before anyone writes into it
  pdl_wait();                // the logits may come from the kernel before this one
  pdl_launch_dependents();
  __syncthreads();
  route_tile<VPL, VEC4>(logits, t0, nt, E, k, lanes_log2, renorm, 1, mask, topk_idx, topk_w);
  __syncthreads();

  cluster_wait();
  const uint32_t counts0 = cluster_map(counts_s, 0);
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    st_cluster_u32(counts0 + 4u * static_cast<uint32_t>(e * C + b), static_cast<uint32_t>(__popc(mask[e])));
  const int64_t base = t0 * k;
  for (int p = threadIdx.x; p < nt * k; p += blockDim.x) {
    const int e = topk_idx[base + p];  // written above by this CTA
    const int tl = p / k;
    lrank[base + p] = __popc(mask[e] & ((1u << tl) - 1u));
  }
  cluster_sync();  // every tile's counts are in CTA 0
  if (b != 0) return;

  // one thread per (expert, tile), segments of Cp lanes (C rounded up to a
  // power of two, the padding lanes adding 0): a segmented scan gives the
  // tile bases, and the segment's last lane the expert's raw total
  int Cp = 1;
  while (Cp < C) Cp <<= 1;
  for (int i0 = 0; i0 < E * Cp; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    const int e = i / Cp, w = i & (Cp - 1);  // w == lane & (Cp - 1): i0 is a multiple of 32
    const bool ok = i < E * Cp && w < C;
    const int c = ok ? counts_s[e * C + w] : 0;
    int v = c;
    for (int o = 1; o < Cp; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (w >= o) v += u;
    }
    if (ok) tile_base[e * C + w] = v - c;
    if (i < E * Cp && w == Cp - 1) {
      const int kept = min(v, cap);
      expert_counts[e] = kept;
      if (expert_raw) expert_raw[e] = v;
      kept_s[e] = kept;
      drop_s[e] = v - kept;
    }
  }
  __syncthreads();
  if (warp != 0) return;

  expert_offsets_warp(kept_s, drop_s, E, R, expert_off, rank_off, n_dropped);
}

template <int VPL, bool VEC4>
cudaError_t launch_route_layout_cluster_t(const RouteCountArgs& r, const DispatchArgs& a, int lanes_log2,
                                          cudaStream_t s, bool dry) {
  constexpr int kBlock = 1024;  // a warp per token of the tile
  const int C = (r.T + 31) / 32;
  const int smem = (r.E + r.E * C + 2 * r.E) * static_cast<int>(sizeof(uint32_t));  // <= 11 KB
  static ClusterFits fits;
  return launch_cluster_pdl(route_layout_cluster_kernel<VPL, VEC4>, C, kBlock, static_cast<size_t>(smem), s, fits,
                            dry, r.logits, r.T, r.E, r.k, lanes_log2, r.renorm, a.R, a.cap, r.topk_idx, r.topk_w, a.lrank,
                            a.tile_base, a.expert_counts, a.expert_raw, a.expert_off, a.rank_off, a.n_dropped);
}

template <int VPL, bool VEC4>
cudaError_t launch_route_t(const float* logits, int T, int E, int k, int lanes_log2, int renorm, int32_t* idx,
                           float* w, int sms, cudaStream_t s) {
  const int groups_per_warp = 32 >> lanes_log2;
  const int64_t warps = (static_cast<int64_t>(T) + groups_per_warp - 1) / groups_per_warp;
  const int64_t blocks_needed = (warps + 7) / 8;
  static int occ[64];  // one cache per template instance
  const int64_t cap_blocks = static_cast<int64_t>(sms) * resident_ctas(route_topk_kernel<VPL, VEC4>, 256, 0, occ);
  const int grid = static_cast<int>(blocks_needed < cap_blocks ? blocks_needed : cap_blocks);
  return launch_pdl(route_topk_kernel<VPL, VEC4>, grid, 256, 0, s, logits, T, E, k, lanes_log2, renorm, idx, w);
}

template <int VPL, bool VEC4>
cudaError_t launch_route_count_t(const RouteCountArgs& r, int lanes_log2, cudaStream_t s) {
  constexpr int kBlock = VPL >= 16 ? 256 : 512;
  static int smem_set[64];  // per device: largest dynamic shared size already allowed
  const int smem = 2 * r.E * (r.tile / 32) * static_cast<int>(sizeof(uint32_t));
  if (smem > 48 * 1024) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 64 || cache_load(&smem_set[dev]) < smem) {
      err = cudaFuncSetAttribute(route_count_kernel<VPL, VEC4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (err != cudaSuccess) return err;
      if (dev < 64) cache_store(&smem_set[dev], smem);
    }
  }
  return launch_pdl(route_count_kernel<VPL, VEC4>, r.ntiles > 0 ? r.ntiles : 1, kBlock, static_cast<size_t>(smem),
                    s, r.logits, r.T, r.E, r.k, lanes_log2, r.renorm, r.tile, r.ntiles, r.topk_idx, r.topk_w,
                    r.tile_counts, r.lrank, r.ticket);
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w, int sms,
                         cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  int lanes_log2 = 0;
  while ((1 << lanes_log2) < E && lanes_log2 < 5) ++lanes_log2;
  const int L = 1 << lanes_log2;
  const int vpl = (E + L - 1) / L;
  const bool vec4 = (L == 32) && (E % 128 == 0);
  if (vec4) {
    switch (vpl) {
      case 4: return launch_route_t<4, true>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
      case 8: return launch_route_t<8, true>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
      case 16: return launch_route_t<16, true>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
      case 32: return launch_route_t<32, true>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
      default: break;
    }
  }
  if (vpl <= 1) return launch_route_t<1, false>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
  if (vpl <= 2) return launch_route_t<2, false>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
  if (vpl <= 4) return launch_route_t<4, false>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
  if (vpl <= 8) return launch_route_t<8, false>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
  if (vpl <= 16) return launch_route_t<16, false>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
  return launch_route_t<32, false>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
}

}  // namespace ep

namespace ep {

cudaError_t launch_route_count(const RouteCountArgs& r, cudaStream_t s) {
  int lanes_log2 = 0;
  while ((1 << lanes_log2) < r.E && lanes_log2 < 5) ++lanes_log2;
  const int L = 1 << lanes_log2;
  const int vpl = (r.E + L - 1) / L;
  const bool vec4 = (L == 32) && (r.E % 128 == 0);
  if (vec4) {
    switch (vpl) {
      case 4: return launch_route_count_t<4, true>(r, lanes_log2, s);
      case 8: return launch_route_count_t<8, true>(r, lanes_log2, s);
      case 16: return launch_route_count_t<16, true>(r, lanes_log2, s);
      case 32: return launch_route_count_t<32, true>(r, lanes_log2, s);
      default: break;
    }
  }
  if (vpl <= 1) return launch_route_count_t<1, false>(r, lanes_log2, s);
  if (vpl <= 2) return launch_route_count_t<2, false>(r, lanes_log2, s);
  if (vpl <= 4) return launch_route_count_t<4, false>(r, lanes_log2, s);
  if (vpl <= 8) return launch_route_count_t<8, false>(r, lanes_log2, s);
  if (vpl <= 16) return launch_route_count_t<16, false>(r, lanes_log2, s);
  return launch_route_count_t<32, false>(r, lanes_log2, s);
}

}  // namespace ep

namespace ep {

bool small_batch(int T, int E, int tile) {
  return T > 0 && T <= 32 * kClusterTiles && E <= kClusterExperts && tile == 32;
}

cudaError_t launch_route_layout_small(const RouteCountArgs& r, const DispatchArgs& a, cudaStream_t s, bool dry) {
  if (!small_batch(r.T, r.E, r.tile)) return cudaErrorNotSupported;
  int lanes_log2 = 0;
  while ((1 << lanes_log2) < r.E && lanes_log2 < 5) ++lanes_log2;
  const int L = 1 << lanes_log2;
  const int vpl = (r.E + L - 1) / L;  // <= 8 for E <= 256
  const bool vec4 = (L == 32) && (r.E % 128 == 0);
  if (vec4) return vpl == 4 ? launch_route_layout_cluster_t<4, true>(r, a, lanes_log2, s, dry)
                            : launch_route_layout_cluster_t<8, true>(r, a, lanes_log2, s, dry);
  if (vpl <= 1) return launch_route_layout_cluster_t<1, false>(r, a, lanes_log2, s, dry);
  if (vpl <= 2) return launch_route_layout_cluster_t<2, false>(r, a, lanes_log2, s, dry);
  if (vpl <= 4) return launch_route_layout_cluster_t<4, false>(r, a, lanes_log2, s, dry);
  return launch_route_layout_cluster_t<8, false>(r, a, lanes_log2, s, dry);
}

}  // namespace ep
