// ep_internal.h — launchers and the workspace layout behind the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "ep.h"
#include "ep_device.cuh"

namespace ep {

// Tokens per counting tile, a function of (T, E) alone so that the workspace
// size query and the dispatch agree: a power of two in [32, 1024] giving about
// 256 tiles (enough CTAs for 148 SMs), shrunk until the count kernel's two
// E x (tile/32) word arrays (bit masks and their prefix counts) fit in 96 KB.
inline int tile_tokens_for(int T, int E) {
  int tile = 32;
  while (tile < 1024 && static_cast<int64_t>(tile) * 256 < T) tile <<= 1;
  while (tile > 32 && static_cast<int64_t>(E) * (tile / 32) * 4 * 2 > 96 * 1024) tile >>= 1;
  return tile;
}

// The fused route+layout+scatter kernel (fused.cu): at most this many CTAs
// (one per SM) and experts (at most 8 logits per routing lane).
constexpr int kFusedMaxCTAs = 256;
constexpr int kFusedMaxExperts = 256;

// Workspace layout (each region 256-byte aligned):
//   [status word, scan ticket | barrier arrivals | barrier round | token counter | kept E |
//    dropped E | tile_counts E x max(ntiles, fused CTAs) | tile_base E x ntiles |
//    lrank T*k]
struct WsLayout {
  int tile;
  int ntiles;
  size_t status_off, ticket_off, bar_off, kept_off, drop_off, tile_counts_off, tile_base_off, lrank_off, total;
};

inline size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

inline WsLayout ws_layout(int T, int E, int k) {
  WsLayout L;
  L.tile = tile_tokens_for(T, E);
  L.ntiles = (T + L.tile - 1) / L.tile;
  const size_t counters = static_cast<size_t>(E) * static_cast<size_t>(L.ntiles) * sizeof(int32_t);
  const int fused_ctas = T < kFusedMaxCTAs ? T : kFusedMaxCTAs;
  const size_t count_slots = static_cast<size_t>(E) *
                             static_cast<size_t>(L.ntiles > fused_ctas ? L.ntiles : fused_ctas) * sizeof(int32_t);
  L.status_off = 0;
  L.ticket_off = 4;  // the combine's unit counter and its warps-done count at 64 and 68
  L.bar_off = 128;  // the grid barrier's arrivals at 128, its round at 256 and the fused scatter's token
                    // counter at 384, each on a 128-byte line of its own (the round is polled while the
                    // arrivals are counted, the counter taken from all the while)
  L.kept_off = 512;
  L.drop_off = L.kept_off + align256(static_cast<size_t>(E) * sizeof(int32_t));
  L.tile_counts_off = L.drop_off + align256(static_cast<size_t>(E) * sizeof(int32_t));
  L.tile_base_off = L.tile_counts_off + align256(count_slots);
  L.lrank_off = L.tile_base_off + align256(counters);
  L.total = L.lrank_off + align256(static_cast<size_t>(T) * static_cast<size_t>(k) * sizeof(int32_t));
  return L;
}

// Per-device caches of launch facts (occupancy, attributes already set,
// cluster residency) are shared by every host thread that calls the library;
// they are read and written with relaxed atomics, so concurrent first calls
// at worst repeat a query.
template <typename T>
inline T cache_load(const T* p) {
  return __atomic_load_n(p, __ATOMIC_RELAXED);
}
template <typename T>
inline void cache_store(T* p, T v) {
  __atomic_store_n(p, v, __ATOMIC_RELAXED);
}

// CTAs of `kernel` (at `block` threads, `smem` dynamic shared bytes) that fit
// on one SM at once, cached per device in cache[64]; 1 if the query fails. A
// grid-stride kernel launched with sms * this many CTAs runs in one wave: a
// larger grid would leave a second, partial wave that starts only when whole
// CTAs of the first one have finished all their work.
template <typename K>
inline int resident_ctas(K kernel, int block, int smem, int* cache) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev < 64) {
    const int c = cache_load(&cache[dev]);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, block, smem) != cudaSuccess || n < 1) n = 1;
  if (dev < 64) cache_store(&cache[dev], n);
  return n;
}

// Launches `kernel` on `s` with programmatic stream serialisation allowed
// (see pdl_wait / pdl_launch_dependents in ep_device.cuh).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// One thread-block cluster of `grid` CTAs (1..kMaxCluster) launched like
// launch_pdl. Whether such a cluster can be resident at all (it may not be,
// e.g. when the process is limited to a share of the SMs) is asked once per
// device and cluster size and kept in `fits` (0 unknown, 1 yes, -1 no); if it
// cannot, nothing is launched and cudaErrorNotSupported is returned, so that
// the caller can take its general path. Only an answer is kept: a query that
// fails is asked again next time. The key leaves out the dynamic shared
// memory, which for the one kernel launched this way is at most 11 KB (E <= 256
// experts, 8 tiles), far below what decides residency.
constexpr int kMaxCluster = 8;  // the portable cluster size
using ClusterFits = signed char[64][kMaxCluster + 1];
template <typename... KArgs, typename... Args>
inline cudaError_t launch_cluster_pdl(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t s,
                                      ClusterFits& fits, bool dry, Args&&... args) {
  if (grid < 1 || grid > kMaxCluster) return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(grid);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  signed char f = dev < 64 ? cache_load(&fits[dev][grid]) : static_cast<signed char>(0);
  if (f == 0) {
    cfg.numAttrs = 1;  // the cluster shape alone
    int clusters = 0;
    err = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
    if (err != cudaSuccess) {
      (void)cudaGetLastError();  // a refused query is not an error of this call: take the general path
      return cudaErrorNotSupported;
    }
    f = clusters > 0 ? 1 : -1;
    if (dev < 64) cache_store(&fits[dev][grid], f);
  }
  if (f < 0) return cudaErrorNotSupported;
  if (dry) return cudaSuccess;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w, int sms,
                         cudaStream_t s);

struct DispatchArgs {
  int T, H, E, k, R, cap;
  int fmt;  // payload format: kFmtBf16, kFmtInt8 or kFmtFp8
  const void* x;
  const int32_t* topk_idx;
  void* payload;
  float* scales;
  int32_t *row_slot, *slot_row, *expert_counts, *expert_raw, *expert_off, *rank_off, *n_dropped;
  // workspace regions
  uint32_t* status;
  uint32_t* ticket;
  unsigned *bar_count, *bar_round;  // the fused kernel's grid barrier
  unsigned* work;                   // the fused kernel's scatter token counter
  int32_t *kept, *dropped, *tile_counts, *tile_base, *lrank;
  int tile, ntiles;
  // 1 when the pair data (topk_idx, lrank) was written two or more launches
  // before the scatter, which may then read it before its dependency wait;
  // 0 when the kernel just before the scatter wrote it.
  int pairs_early = 1;
};

// Checks the arguments of a dispatch (before any launch: a status other than
// EP_OK means nothing was enqueued) and fills the kernel arguments, with the
// workspace ws carved into its regions; *sms_out is the device's SM count.
ep_status_t prepare_dispatch(const ep_config_t* cfg, const void* x, const int32_t* topk_idx, void* payload,
                             float* scales, int32_t* row_slot, int32_t* slot_row, int32_t* expert_counts,
                             int32_t* expert_raw, int32_t* expert_off, int32_t* rank_off, int32_t* n_dropped,
                             void* ws, size_t ws_bytes, DispatchArgs* out, int* sms_out);

// ep_dispatch: count kernel, then scan and scatter.
cudaError_t launch_dispatch(const DispatchArgs& a, int sms, cudaStream_t s);
// Counts and offsets from per-token expert bitmaps [T, words] (count + scan).
cudaError_t launch_layout_from_bitmap(const DispatchArgs& a, const uint32_t* bitmap, int words, cudaStream_t s);
// ep_bitmap_encode / ep_bitmap_layout.
cudaError_t launch_encode_bitmap(const int32_t* idx, int64_t T, int E, int k, uint32_t* bitmap, uint32_t* status,
                                 int sms, cudaStream_t s);
cudaError_t launch_bitmap_layout(const DispatchArgs& a, const uint32_t* bitmap, int32_t* row_token, int sms,
                                 cudaStream_t s);
// The scan and the scatter alone, once tile_counts / lrank are written (by
// the count kernel or the fused route+count kernel) and the ticket is clear.
cudaError_t launch_scan_scatter(const DispatchArgs& a, int sms, cudaStream_t s);
// The scatter alone, once lrank, tile_base and the offsets are written.
cudaError_t launch_scatter(const DispatchArgs& a, int sms, cudaStream_t s);

// Routing fused with the dispatch's per-tile count (ep_route_dispatch).
struct RouteCountArgs {
  const float* logits;
  int T, E, k, renorm, tile, ntiles;
  int32_t* topk_idx;
  float* topk_w;
  int32_t *tile_counts, *lrank;
  uint32_t* ticket;
};
cudaError_t launch_route_count(const RouteCountArgs& r, cudaStream_t s);

// Small batches (at most kClusterTiles tiles of 32 tokens, E <= 256): one
// thread-block cluster of one CTA per tile routes the batch and forms the
// whole layout (topk_idx / topk_w, lrank, tile_base and every layout output)
// in one launch; the scatter follows. Returns cudaErrorNotSupported, having
// launched nothing, when the batch is not small or such a cluster cannot be
// resident on the device.
constexpr int kClusterTiles = kMaxCluster;
constexpr int kClusterExperts = 256;  // experts per routing lane group of 32: at most 8 values per lane
bool small_batch(int T, int E, int tile);
cudaError_t launch_route_layout_small(const RouteCountArgs& r, const DispatchArgs& a, cudaStream_t s,
                                      bool dry = false);

// ep_route_dispatch in one cooperative launch of one CTA per SM (fused.cu):
// routing, layout and scatter with one bounded grid barrier. Returns
// cudaErrorNotSupported, having launched nothing, when the problem or the
// device does not suit it (E > kFusedMaxExperts, more than 1024 tokens per
// SM, x not 32-byte aligned, no cooperative launch); the caller then takes
// the kernel chain.
// dry: check only (the same checks, nothing launched): cudaSuccess when it would run.
cudaError_t launch_route_dispatch_fused(const RouteCountArgs& r, const DispatchArgs& a, int sms, cudaStream_t s,
                                        bool dry = false);
// Test hook (ep_debug_force_wait_timeout): the fused kernel's grid barrier
// waits for one CTA more than the grid, with a short limit, so that it runs
// out and reports EP_ERR_TIMEOUT.
void set_force_wait_timeout(int enable);

struct CombineArgs {
  int T, H, k;
  int out_fmt;  // expert-output format: kFmtBf16, kFmtInt8 or kFmtFp8
  int slices;  // work units per token (set by the launcher)
  int64_t max_rows;
  const void* expert_out;
  const float* out_scales;
  const int32_t* slot_row;
  const float* topk_w;
  void* y;
  uint32_t* status;
  unsigned* counter;  // two words of the workspace (zero between calls): a unit counter and the warps done; or null
  int static_rounds;  // with counter: units each warp takes in the static order before the shared ones (>= 1)
};

cudaError_t launch_combine(const CombineArgs& a, int sms, cudaStream_t s);

cudaError_t launch_quantize_rows(const void* in, int64_t n, int H, int fmt, void* q, float* scales, int sms,
                                 cudaStream_t s);

}  // namespace ep
