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
// Device address of g_dispatch_scratch, per device: one pointer, read and
// written with relaxed atomics, so concurrent first calls on a device at
// worst both look the address up (and store the same value).
void* g_scratch_ptr[kMaxDevices];

// Device address of the static scratch on the current device (looked up on
// the first call per device). Returns nullptr and sets *err on failure.
void* static_scratch(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  void* p = ep::cache_load(&g_scratch_ptr[dev]);
  if (p == nullptr) {
    *err = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (*err != cudaSuccess) return nullptr;
    ep::cache_store(&g_scratch_ptr[dev], p);
  }
  return p;
}

}  // namespace

extern "C" ep_status_t ep_dispatch_static(const ep_config_t* cfg, const void* x, const int32_t* topk_idx,
                                          void* payload, float* scales, int32_t* row_slot, int32_t* slot_row,
                                          int32_t* expert_counts, int32_t* expert_raw, int32_t* expert_off,
                                          int32_t* rank_off, int32_t* n_dropped, cudaStream_t stream) {
  // The size check comes first and needs no device: a problem whose scratch
  // does not fit the fixed array is refused before anything is enqueued.
  if (ep_config_check(cfg) != EP_OK) return EP_ERR_INVALID_ARG;
  const ep::WsLayout L = ep::ws_layout(cfg->T, cfg->E, cfg->k);
  if (L.total > static_cast<size_t>(EP_STATIC_SCRATCH_BYTES)) return EP_ERR_WORKSPACE;

  cudaError_t err = cudaSuccess;
  void* w = static_scratch(&err);
  if (w == nullptr) return EP_ERR_CUDA;
  // The same argument checks and workspace carving as ep_dispatch, over the
  // static array (nothing is enqueued unless they pass).
  ep::DispatchArgs a;
  int sms = 0;
  const ep_status_t st = ep::prepare_dispatch(cfg, x, topk_idx, payload, scales, row_slot, slot_row, expert_counts,
                                              expert_raw, expert_off, rank_off, n_dropped, w,
                                              static_cast<size_t>(EP_STATIC_SCRATCH_BYTES), &a, &sms);
  if (st != EP_OK) return st;
  // The array keeps the previous call's contents: clear the status word and
  // the scan ticket, the only parts read before this call writes them.
  if (cudaMemsetAsync(w, 0, 256, stream) != cudaSuccess) return EP_ERR_CUDA;
  return ep::launch_dispatch(a, sms, stream) == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}
