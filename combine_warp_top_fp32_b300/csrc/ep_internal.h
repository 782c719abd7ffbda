// ep_internal.h — launchers and the workspace layout behind the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ep_device.cuh"

namespace ep {

// Tokens per counting tile, a function of E alone so that the workspace size
// query and the dispatch agree. The count kernel keeps two E x (tile/32)
// word arrays in shared memory (bit masks and their prefix counts).
inline int tile_tokens_for(int E) {
  if (static_cast<int64_t>(E) * (1024 / 32) * 4 * 2 <= 96 * 1024) return 1024;
  if (static_cast<int64_t>(E) * (512 / 32) * 4 * 2 <= 96 * 1024) return 512;
  return 256;
}

// Workspace layout (each region 256-byte aligned):
//   [status word | tile_counts E x ntiles | tile_base E x ntiles | lrank T*k]
struct WsLayout {
  int tile;
  int ntiles;
  size_t status_off, tile_counts_off, tile_base_off, lrank_off, total;
};

inline size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

inline WsLayout ws_layout(int T, int E, int k) {
  WsLayout L;
  L.tile = tile_tokens_for(E);
  L.ntiles = (T + L.tile - 1) / L.tile;
  const size_t counters = static_cast<size_t>(E) * static_cast<size_t>(L.ntiles) * sizeof(int32_t);
  L.status_off = 0;
  L.tile_counts_off = 256;
  L.tile_base_off = L.tile_counts_off + align256(counters);
  L.lrank_off = L.tile_base_off + align256(counters);
  L.total = L.lrank_off + align256(static_cast<size_t>(T) * static_cast<size_t>(k) * sizeof(int32_t));
  return L;
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w, int sms,
                         cudaStream_t s);

struct DispatchArgs {
  int T, H, E, k, R, cap, int8;
  const void* x;
  const int32_t* topk_idx;
  void* payload;
  float* scales;
  int32_t *row_slot, *slot_row, *expert_counts, *expert_raw, *expert_off, *rank_off, *n_dropped;
  // workspace regions
  uint32_t* status;
  int32_t *tile_counts, *tile_base, *lrank;
  int tile, ntiles;
};

cudaError_t launch_dispatch(const DispatchArgs& a, int sms, cudaStream_t s);

struct CombineArgs {
  int T, H, k, int8_out;
  int64_t max_rows;
  const void* expert_out;
  const float* out_scales;
  const int32_t* slot_row;
  const float* topk_w;
  void* y;
  uint32_t* status;
};

cudaError_t launch_combine(const CombineArgs& a, int sms, cudaStream_t s);

cudaError_t launch_quantize_rows(const void* in, int64_t n, int H, int8_t* q, float* scales, int sms,
                                 cudaStream_t s);

}  // namespace ep
