// ep_static.cu — ep_dispatch_static: the dispatch for callers that cannot
// allocate device memory.
//
// ep_dispatch needs a scratch workspace (per-tile counters, the scan's ticket
// and status word, per-pair ranks). Most callers allocate it once with
// cudaMalloc or their framework's allocator. Some callers cannot: a plugin or
// custom-op host that hands an operator only its input and output buffers
// and forbids allocation inside the enqueue call, a runtime that plans all
// device memory ahead of time in a fixed arena, or a latency-critical path
// where cudaMalloc's implicit device-wide synchronisation is not acceptable.
// For them this entry point keeps the scratch in a file-scope device array of
// fixed size, EP_STATIC_SCRATCH_BYTES, which every GPU that loads the library
// holds until the process exits. It runs the same kernels as ep_dispatch.
//
// The array's name in host code is only a host-side handle, not a device
// address. The device address is obtained once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// that device; that first call should therefore come before any stream
// capture begins. All calls share the one array: two calls whose work
// overlaps on the GPU (different streams, or different host threads on the
// same device) race on it and must be serialised by the caller.
#include <stdint.h>

#include "ep.h"
#include "ep_internal.h"

// The scratch area itself: file scope, one copy per device.
static __device__ __align__(256) unsigned char g_dispatch_scratch[EP_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];  // device address of g_dispatch_scratch, per device
int g_scratch_sms[kMaxDevices];

bool is_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device address of the static scratch on the current device (set up on the
// first call per device). Returns nullptr and sets *err on failure.
void* static_scratch(int* sms, cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (*err != cudaSuccess) return nullptr;
    int n = 0;
    *err = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (*err != cudaSuccess) return nullptr;
    g_scratch_sms[dev] = n;
    g_scratch_ptr[dev] = p;
  }
  *sms = g_scratch_sms[dev];
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" ep_status_t ep_dispatch_static(const ep_config_t* cfg, const void* x, const int32_t* topk_idx,
                                          void* payload, float* scales, int32_t* row_slot, int32_t* slot_row,
                                          int32_t* expert_counts, int32_t* expert_raw, int32_t* expert_off,
                                          int32_t* rank_off, int32_t* n_dropped, cudaStream_t stream) {
  if (ep_config_check(cfg) != EP_OK) return EP_ERR_INVALID_ARG;
  const bool coded = cfg->payload != EP_PAYLOAD_BF16;  // int8 or FP8 code + per-row scale
  if (!expert_counts || !expert_off || !rank_off || !n_dropped) return EP_ERR_INVALID_ARG;
  if (cfg->T > 0) {
    if (!x || !topk_idx || !payload || !row_slot || !slot_row) return EP_ERR_INVALID_ARG;
    if (coded && !scales) return EP_ERR_INVALID_ARG;
    if (!is_aligned(x, 16) || !is_aligned(payload, 16)) return EP_ERR_INVALID_ARG;
  }
  if (!is_aligned(topk_idx, 4) || !is_aligned(row_slot, 4) || !is_aligned(slot_row, 4) ||
      !is_aligned(expert_counts, 4) || !is_aligned(expert_raw, 4) || !is_aligned(expert_off, 4) ||
      !is_aligned(rank_off, 4) || !is_aligned(n_dropped, 4) || !is_aligned(scales, 4))
    return EP_ERR_INVALID_ARG;
  // The problem's scratch must fit the fixed array; larger problems are
  // refused here, before anything is enqueued.
  const ep::WsLayout L = ep::ws_layout(cfg->T, cfg->E, cfg->k);
  if (L.total > static_cast<size_t>(EP_STATIC_SCRATCH_BYTES)) return EP_ERR_WORKSPACE;

  int sms = 0;
  cudaError_t err = cudaSuccess;
  char* w = static_cast<char*>(static_scratch(&sms, &err));
  if (w == nullptr || sms <= 0) return EP_ERR_CUDA;
  // The array keeps the previous call's contents: clear the status word and
  // the scan ticket, the only parts read before this call writes them.
  if (cudaMemsetAsync(w, 0, 256, stream) != cudaSuccess) return EP_ERR_CUDA;

  ep::DispatchArgs a;
  a.T = cfg->T;
  a.H = cfg->H;
  a.E = cfg->E;
  a.k = cfg->k;
  a.R = cfg->R;
  int32_t cap = 0;
  if (ep_capacity(cfg, &cap) != EP_OK) return EP_ERR_INVALID_ARG;
  a.cap = cap;
  a.fmt = cfg->payload;
  a.x = x;
  a.topk_idx = topk_idx;
  a.payload = payload;
  a.scales = scales;
  a.row_slot = row_slot;
  a.slot_row = slot_row;
  a.expert_counts = expert_counts;
  a.expert_raw = expert_raw;
  a.expert_off = expert_off;
  a.rank_off = rank_off;
  a.n_dropped = n_dropped;
  a.status = reinterpret_cast<uint32_t*>(w + L.status_off);
  a.ticket = reinterpret_cast<uint32_t*>(w + L.ticket_off);
  a.kept = reinterpret_cast<int32_t*>(w + L.kept_off);
  a.dropped = reinterpret_cast<int32_t*>(w + L.drop_off);
  a.tile_counts = reinterpret_cast<int32_t*>(w + L.tile_counts_off);
  a.tile_base = reinterpret_cast<int32_t*>(w + L.tile_base_off);
  a.lrank = reinterpret_cast<int32_t*>(w + L.lrank_off);
  a.tile = L.tile;
  a.ntiles = L.ntiles;
  return ep::launch_dispatch(a, sms, stream) == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}
