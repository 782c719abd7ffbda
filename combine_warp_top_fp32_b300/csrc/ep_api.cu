// ep_api.cu — the extern "C" entry points of libep_b300 (declared in ep.h):
// host-side argument checks, workspace carving and kernel launches.
//
// Every check runs before the first launch, so a call that returns
// EP_ERR_INVALID_ARG or EP_ERR_WORKSPACE has enqueued nothing. The library
// never synchronises a stream except in ep_get_error().
#include <math.h>
#include <string.h>

#include "ep.h"
#include "ep_internal.h"

namespace {

constexpr int kMaxH = 16384;
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kMaxDevices = 64;

int g_sm_count[kMaxDevices];  // per-device SM count, filled on first use

// A device attribute of the current device, cached per device (relaxed
// atomics: concurrent first calls at worst repeat the query); 0 on failure.
int current_attribute(cudaDeviceAttr attr, int* cache) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < kMaxDevices) {
    const int v = ep::cache_load(&cache[dev]);
    if (v > 0) return v;
  }
  int v = 0;
  if (cudaDeviceGetAttribute(&v, attr, dev) != cudaSuccess) return 0;
  if (dev < kMaxDevices && v > 0) ep::cache_store(&cache[dev], v);
  return v;
}

// SM count of the current device; 0 on failure.
int current_sm_count() { return current_attribute(cudaDevAttrMultiProcessorCount, g_sm_count); }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool config_ok(const ep_config_t* c) {
  if (c == nullptr) return false;
  if (c->T < 0) return false;
  if (c->H < 16 || c->H > kMaxH || c->H % 16 != 0) return false;
  if (c->E < 1 || c->E > kMaxE) return false;
  if (c->k < 1 || c->k > c->E || c->k > kMaxK) return false;
  if (c->R < 1 || c->E % c->R != 0) return false;
  if (isnan(c->capacity_factor) || isinf(c->capacity_factor)) return false;
  if (c->renormalize != 0 && c->renormalize != 1) return false;
  if (c->payload < EP_PAYLOAD_BF16 || c->payload > EP_PAYLOAD_INT4) return false;
  if (c->payload == EP_PAYLOAD_INT4 && c->H % 32 != 0) return false;  // rows of H/2 bytes, 16-byte aligned
  if (static_cast<int64_t>(c->T) * c->k > INT32_MAX) return false;
  return true;
}

// ceil(cf * T * k / E) in double, in that order, clipped to T (an expert can
// receive at most one copy per token); T when dropless.
int32_t capacity_of(const ep_config_t* c) {
  if (!(c->capacity_factor > 0.0f)) return c->T;
  const double v = ceil(static_cast<double>(c->capacity_factor) * c->T * c->k / c->E);
  return v >= static_cast<double>(c->T) ? c->T : static_cast<int32_t>(v);
}

int64_t max_rows_of(const ep_config_t* c) {
  const int64_t tk = static_cast<int64_t>(c->T) * c->k;
  if (!(c->capacity_factor > 0.0f)) return tk;
  const int64_t ecap = static_cast<int64_t>(c->E) * capacity_of(c);
  return tk < ecap ? tk : ecap;
}

ep_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? EP_OK : EP_ERR_CUDA; }

int g_route_dispatch_form = EP_FORM_AUTO;  // ep_debug_set(EP_DEBUG_ROUTE_DISPATCH_FORM, ...)

// Whether the single launch beats the chain by default (measured on the
// B300): with E >= 32 at every batch size measured (128 to 131,072 tokens;
// e.g. 4,096 tokens, E = 64: 49-50 against 56 us a step with bf16
// payloads), and with large batches (T >= 8192) at any E; with E < 32 on
// small batches the cluster form of the chain is quicker.
bool single_launch_pays(const ep_config_t* c) { return c->T >= 8192 || c->E >= 32; }

// The form ep_route_dispatch takes for a call whose arguments passed the
// checks: the single launch (if chosen and it can run here), the cluster form
// of the chain for small batches (if such a cluster can be resident), else
// the three-kernel chain. The checks launch nothing.
enum class Form { kSingle, kCluster, kChain };
Form choose_form(const ep_config_t* cfg, const ep::RouteCountArgs& r, const ep::DispatchArgs& a, int sms) {
  const int form = ep::cache_load(&g_route_dispatch_form);
  if ((form == EP_FORM_SINGLE || (form == EP_FORM_AUTO && single_launch_pays(cfg))) &&
      ep::launch_route_dispatch_fused(r, a, sms, nullptr, true) == cudaSuccess)
    return Form::kSingle;
  if (ep::small_batch(r.T, r.E, r.tile) && ep::launch_route_layout_small(r, a, nullptr, true) == cudaSuccess)
    return Form::kCluster;
  return Form::kChain;
}

// The routing arguments of ep_route_dispatch (from the checked dispatch ones).
ep::RouteCountArgs route_count_args(const ep_config_t* cfg, const float* logits, int32_t* topk_idx, float* topk_w,
                                    const ep::DispatchArgs& a) {
  ep::RouteCountArgs r;
  r.logits = logits;
  r.T = cfg->T;
  r.E = cfg->E;
  r.k = cfg->k;
  r.renorm = cfg->renormalize;
  r.tile = a.tile;
  r.ntiles = a.ntiles;
  r.topk_idx = topk_idx;
  r.topk_w = topk_w;
  r.tile_counts = a.tile_counts;
  r.lrank = a.lrank;
  r.ticket = a.ticket;
  return r;
}

ep_status_t carve_layout(const ep_config_t* cfg, int32_t* expert_counts, int32_t* expert_raw, int32_t* expert_off,
                         int32_t* rank_off, int32_t* n_dropped, void* ws, size_t ws_bytes, ep::DispatchArgs* out,
                         int* sms_out);

}  // namespace

// Checks the dispatch arguments (before any launch) and fills the kernel
// arguments, with the workspace carved into its regions.
ep_status_t ep::prepare_dispatch(const ep_config_t* cfg, const void* x, const int32_t* topk_idx, void* payload,
                                 float* scales, int32_t* row_slot, int32_t* slot_row, int32_t* expert_counts,
                                 int32_t* expert_raw, int32_t* expert_off, int32_t* rank_off, int32_t* n_dropped,
                                 void* ws, size_t ws_bytes, ep::DispatchArgs* out, int* sms_out) {
  if (!config_ok(cfg)) return EP_ERR_INVALID_ARG;
  const bool coded = cfg->payload != EP_PAYLOAD_BF16;  // int8 or FP8 code + per-row scale
  if (!expert_counts || !expert_off || !rank_off || !n_dropped) return EP_ERR_INVALID_ARG;
  if (cfg->T > 0) {
    if (!x || !topk_idx || !payload || !row_slot || !slot_row) return EP_ERR_INVALID_ARG;
    if (coded && !scales) return EP_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(payload, 16)) return EP_ERR_INVALID_ARG;
  }
  if (!aligned(topk_idx, 4) || !aligned(row_slot, 4) || !aligned(slot_row, 4) || !aligned(expert_counts, 4) ||
      !aligned(expert_raw, 4) || !aligned(expert_off, 4) || !aligned(rank_off, 4) || !aligned(n_dropped, 4) ||
      !aligned(scales, 4))
    return EP_ERR_INVALID_ARG;
  const ep_status_t st = carve_layout(cfg, expert_counts, expert_raw, expert_off, rank_off, n_dropped, ws, ws_bytes,
                                      out, sms_out);
  if (st != EP_OK) return st;
  ep::DispatchArgs& a = *out;
  a.x = x;
  a.topk_idx = topk_idx;
  a.payload = payload;
  a.scales = scales;
  a.row_slot = row_slot;
  a.slot_row = slot_row;
  return EP_OK;
}

namespace {

// The layout part of the kernel arguments (sizes, cap, the layout outputs and
// the workspace regions), after the workspace check.
ep_status_t carve_layout(const ep_config_t* cfg, int32_t* expert_counts, int32_t* expert_raw, int32_t* expert_off,
                         int32_t* rank_off, int32_t* n_dropped, void* ws, size_t ws_bytes, ep::DispatchArgs* out,
                         int* sms_out) {
  const ep::WsLayout L = ep::ws_layout(cfg->T, cfg->E, cfg->k);
  if (ws == nullptr || ws_bytes < L.total || !aligned(ws, 256)) return EP_ERR_WORKSPACE;
  const int sms = current_sm_count();
  if (sms <= 0) return EP_ERR_CUDA;

  char* w = static_cast<char*>(ws);
  ep::DispatchArgs& a = *out;
  a.T = cfg->T;
  a.H = cfg->H;
  a.E = cfg->E;
  a.k = cfg->k;
  a.R = cfg->R;
  a.cap = capacity_of(cfg);
  a.fmt = cfg->payload;  // EP_PAYLOAD_* values are the kernels' format numbers
  a.x = nullptr;
  a.topk_idx = nullptr;
  a.payload = nullptr;
  a.scales = nullptr;
  a.row_slot = nullptr;
  a.slot_row = nullptr;
  a.expert_counts = expert_counts;
  a.expert_raw = expert_raw;
  a.expert_off = expert_off;
  a.rank_off = rank_off;
  a.n_dropped = n_dropped;
  a.status = reinterpret_cast<uint32_t*>(w + L.status_off);
  a.ticket = reinterpret_cast<uint32_t*>(w + L.ticket_off);
  a.bar_count = reinterpret_cast<unsigned*>(w + L.bar_off);
  a.bar_round = reinterpret_cast<unsigned*>(w + L.bar_off + 128);
  a.work = reinterpret_cast<unsigned*>(w + L.bar_off + 256);
  a.kept = reinterpret_cast<int32_t*>(w + L.kept_off);
  a.dropped = reinterpret_cast<int32_t*>(w + L.drop_off);
  a.tile_counts = reinterpret_cast<int32_t*>(w + L.tile_counts_off);
  a.tile_base = reinterpret_cast<int32_t*>(w + L.tile_base_off);
  a.lrank = reinterpret_cast<int32_t*>(w + L.lrank_off);
  a.tile = L.tile;
  a.ntiles = L.ntiles;
  *sms_out = sms;
  return EP_OK;
}

// int8 or FP8 per-row code of n rows (ep_quantize_rows, ep_quantize_rows_fp8).
ep_status_t quantize_rows(const void* in, int64_t n, int32_t H, int fmt, void* q, float* scales,
                          cudaStream_t stream) {
  if (n < 0 || H < 16 || H > kMaxH || H % 16 != 0) return EP_ERR_INVALID_ARG;
  if (fmt == ep::kFmtInt4 && H % 32 != 0) return EP_ERR_INVALID_ARG;
  if (n == 0) return EP_OK;
  if (!in || !q || !scales || !aligned(in, 16) || !aligned(q, 16) || !aligned(scales, 4)) return EP_ERR_INVALID_ARG;
  const int sms = current_sm_count();
  if (sms <= 0) return EP_ERR_CUDA;
  return from_cuda(ep::launch_quantize_rows(in, n, H, fmt, q, scales, sms, stream));
}

}  // namespace

extern "C" {

const char* ep_status_string(ep_status_t s) {
  switch (s) {
    case EP_OK: return "ok";
    case EP_ERR_INVALID_ARG: return "invalid argument";
    case EP_ERR_WORKSPACE: return "workspace missing or too small";
    case EP_ERR_CUDA: return "CUDA runtime error";
    case EP_ERR_TIMEOUT: return "bounded device wait timed out";
    case EP_ERR_DEVICE_INDEX: return "index input out of range or repeated";
  }
  return "unknown status";
}

ep_status_t ep_config_check(const ep_config_t* cfg) { return config_ok(cfg) ? EP_OK : EP_ERR_INVALID_ARG; }

ep_status_t ep_capacity(const ep_config_t* cfg, int32_t* cap) {
  if (!config_ok(cfg) || cap == nullptr) return EP_ERR_INVALID_ARG;
  *cap = capacity_of(cfg);
  return EP_OK;
}

int64_t ep_max_rows(const ep_config_t* cfg) { return config_ok(cfg) ? max_rows_of(cfg) : 0; }

ep_status_t ep_workspace_size(const ep_config_t* cfg, size_t* bytes) {
  if (!config_ok(cfg) || bytes == nullptr) return EP_ERR_INVALID_ARG;
  *bytes = ep::ws_layout(cfg->T, cfg->E, cfg->k).total;
  return EP_OK;
}

ep_status_t ep_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (ws == nullptr || ws_bytes < 256 || !aligned(ws, 256)) return EP_ERR_WORKSPACE;
  return from_cuda(cudaMemsetAsync(ws, 0, ws_bytes, stream));
}

ep_status_t ep_route(const ep_config_t* cfg, const float* logits, int32_t* topk_idx, float* topk_w,
                     cudaStream_t stream) {
  if (!config_ok(cfg)) return EP_ERR_INVALID_ARG;
  if (cfg->T == 0) return EP_OK;
  if (!logits || !topk_idx || !topk_w) return EP_ERR_INVALID_ARG;
  if (!aligned(logits, 16) || !aligned(topk_idx, 4) || !aligned(topk_w, 4)) return EP_ERR_INVALID_ARG;
  const int sms = current_sm_count();
  if (sms <= 0) return EP_ERR_CUDA;
  return from_cuda(ep::launch_route(logits, cfg->T, cfg->E, cfg->k, cfg->renormalize, topk_idx, topk_w, sms, stream));
}

ep_status_t ep_dispatch(const ep_config_t* cfg, const void* x, const int32_t* topk_idx, void* payload,
                        float* scales, int32_t* row_slot, int32_t* slot_row, int32_t* expert_counts,
                        int32_t* expert_raw, int32_t* expert_off, int32_t* rank_off, int32_t* n_dropped,
                        void* ws, size_t ws_bytes, cudaStream_t stream) {
  ep::DispatchArgs a;
  int sms = 0;
  const ep_status_t st = ep::prepare_dispatch(cfg, x, topk_idx, payload, scales, row_slot, slot_row, expert_counts,
                                          expert_raw, expert_off, rank_off, n_dropped, ws, ws_bytes, &a, &sms);
  if (st != EP_OK) return st;
  return from_cuda(ep::launch_dispatch(a, sms, stream));
}

ep_status_t ep_route_dispatch(const ep_config_t* cfg, const float* logits, const void* x, int32_t* topk_idx,
                              float* topk_w, void* payload, float* scales, int32_t* row_slot, int32_t* slot_row,
                              int32_t* expert_counts, int32_t* expert_raw, int32_t* expert_off, int32_t* rank_off,
                              int32_t* n_dropped, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!config_ok(cfg)) return EP_ERR_INVALID_ARG;
  if (cfg->T > 0) {
    if (!logits || !topk_idx || !topk_w) return EP_ERR_INVALID_ARG;
    if (!aligned(logits, 16) || !aligned(topk_w, 4)) return EP_ERR_INVALID_ARG;
  }
  ep::DispatchArgs a;
  int sms = 0;
  const ep_status_t st = ep::prepare_dispatch(cfg, x, topk_idx, payload, scales, row_slot, slot_row, expert_counts,
                                          expert_raw, expert_off, rank_off, n_dropped, ws, ws_bytes, &a, &sms);
  if (st != EP_OK) return st;
  ep::RouteCountArgs r = route_count_args(cfg, logits, topk_idx, topk_w, a);
  switch (choose_form(cfg, r, a, sms)) {
    case Form::kSingle:  // one cooperative launch routes, lays out and scatters the batch
      return from_cuda(ep::launch_route_dispatch_fused(r, a, sms, stream));
    case Form::kCluster: {  // one cluster routes and lays out the batch, then the scatter
      const cudaError_t e = ep::launch_route_layout_small(r, a, stream);
      if (e != cudaSuccess) return EP_ERR_CUDA;
      a.pairs_early = 0;  // the routing kernel just before wrote topk_idx and lrank
      return from_cuda(ep::launch_scatter(a, sms, stream));
    }
    case Form::kChain:
      break;
  }
  const cudaError_t err = ep::launch_route_count(r, stream);
  if (err != cudaSuccess) return EP_ERR_CUDA;
  return from_cuda(ep::launch_scan_scatter(a, sms, stream));
}

ep_status_t ep_bitmap_encode(const ep_config_t* cfg, const int32_t* topk_idx, uint32_t* bitmap, void* ws,
                             size_t ws_bytes, cudaStream_t stream) {
  if (!config_ok(cfg)) return EP_ERR_INVALID_ARG;
  if (ws == nullptr || ws_bytes < 256 || !aligned(ws, 256)) return EP_ERR_WORKSPACE;
  if (cfg->T == 0) return EP_OK;
  if (!topk_idx || !bitmap || !aligned(topk_idx, 4) || !aligned(bitmap, 4)) return EP_ERR_INVALID_ARG;
  const int sms = current_sm_count();
  if (sms <= 0) return EP_ERR_CUDA;
  return from_cuda(ep::launch_encode_bitmap(topk_idx, cfg->T, cfg->E, cfg->k, bitmap, static_cast<uint32_t*>(ws), sms,
                                            stream));
}

ep_status_t ep_bitmap_layout(const ep_config_t* cfg, const uint32_t* bitmap, int32_t* row_token,
                             int32_t* expert_counts, int32_t* expert_raw, int32_t* expert_off, int32_t* rank_off,
                             int32_t* n_dropped, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!config_ok(cfg)) return EP_ERR_INVALID_ARG;
  if (!expert_counts || !expert_off || !rank_off || !n_dropped) return EP_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!bitmap || !row_token)) return EP_ERR_INVALID_ARG;
  if (!aligned(bitmap, 4) || !aligned(row_token, 4) || !aligned(expert_counts, 4) || !aligned(expert_raw, 4) ||
      !aligned(expert_off, 4) || !aligned(rank_off, 4) || !aligned(n_dropped, 4))
    return EP_ERR_INVALID_ARG;
  ep::DispatchArgs a;
  int sms = 0;
  const ep_status_t st =
      carve_layout(cfg, expert_counts, expert_raw, expert_off, rank_off, n_dropped, ws, ws_bytes, &a, &sms);
  if (st != EP_OK) return st;
  return from_cuda(ep::launch_bitmap_layout(a, bitmap, row_token, sms, stream));
}

ep_status_t ep_combine(const ep_config_t* cfg, const void* expert_out, const float* out_scales,
                       int32_t out_payload, const int32_t* slot_row, const float* topk_w, void* y, void* ws,
                       size_t ws_bytes, cudaStream_t stream) {
  if (!config_ok(cfg)) return EP_ERR_INVALID_ARG;
  if (out_payload < EP_PAYLOAD_BF16 || out_payload > EP_PAYLOAD_INT4) return EP_ERR_INVALID_ARG;
  if (out_payload == EP_PAYLOAD_INT4 && cfg->H % 32 != 0) return EP_ERR_INVALID_ARG;
  if (ws == nullptr || ws_bytes < 256 || !aligned(ws, 256)) return EP_ERR_WORKSPACE;
  if (cfg->T == 0) return EP_OK;
  const bool coded = out_payload != EP_PAYLOAD_BF16;
  if (!expert_out || !slot_row || !topk_w || !y || (coded && !out_scales)) return EP_ERR_INVALID_ARG;
  if (!aligned(expert_out, 16) || !aligned(y, 16) || !aligned(slot_row, 4) || !aligned(topk_w, 4) ||
      !aligned(out_scales, 4))
    return EP_ERR_INVALID_ARG;
  const int sms = current_sm_count();
  if (sms <= 0) return EP_ERR_CUDA;
  ep::CombineArgs a;
  a.T = cfg->T;
  a.H = cfg->H;
  a.k = cfg->k;
  a.out_fmt = out_payload;
  a.max_rows = max_rows_of(cfg);
  a.expert_out = expert_out;
  a.out_scales = out_scales;
  a.slot_row = slot_row;
  a.topk_w = topk_w;
  a.y = y;
  a.status = static_cast<uint32_t*>(ws);
  a.counter = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + 64);  // the launcher may not use it
  a.static_rounds = 1;
  return from_cuda(ep::launch_combine(a, sms, stream));
}

ep_status_t ep_quantize_rows(const void* in, int64_t n, int32_t H, int8_t* q, float* scales, cudaStream_t stream) {
  return quantize_rows(in, n, H, ep::kFmtInt8, q, scales, stream);
}

ep_status_t ep_quantize_rows_fp8(const void* in, int64_t n, int32_t H, uint8_t* q, float* scales,
                                 cudaStream_t stream) {
  return quantize_rows(in, n, H, ep::kFmtFp8, q, scales, stream);
}

ep_status_t ep_quantize_rows_int4(const void* in, int64_t n, int32_t H, uint8_t* q, float* scales,
                                  cudaStream_t stream) {
  return quantize_rows(in, n, H, ep::kFmtInt4, q, scales, stream);
}

ep_status_t ep_get_error(void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (ws == nullptr || ws_bytes < 256 || !aligned(ws, 256)) return EP_ERR_WORKSPACE;
  uint32_t flags = 0;
  if (cudaMemcpyAsync(&flags, ws, sizeof flags, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return EP_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return EP_ERR_CUDA;
  if (flags == 0) return EP_OK;
  // clear the status word; after a timed-out wait also the grid barrier's
  // words, which a wait that gave up leaves behind
  const size_t header = ws_bytes < 512 ? ws_bytes : 512;  // status, ticket, barrier words, counter
  const size_t clear = (flags & ep::kStatusTimeout) ? header : sizeof flags;
  if (cudaMemsetAsync(ws, 0, clear, stream) != cudaSuccess) return EP_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return EP_ERR_CUDA;
  if (flags & ep::kStatusTimeout) return EP_ERR_TIMEOUT;
  return EP_ERR_DEVICE_INDEX;
}

ep_status_t ep_route_dispatch_kernels(const ep_config_t* cfg, int32_t* kernels) {
  if (!config_ok(cfg) || kernels == nullptr) return EP_ERR_INVALID_ARG;
  const ep::WsLayout L = ep::ws_layout(cfg->T, cfg->E, cfg->k);
  ep::DispatchArgs a;
  int sms = 0;
  // no buffers: carve a workspace-sized range at address 0 (nothing is read
  // or launched; x is taken as 32-byte aligned)
  const ep_status_t st = carve_layout(cfg, nullptr, nullptr, nullptr, nullptr, nullptr,
                                      reinterpret_cast<void*>(static_cast<uintptr_t>(256)), L.total, &a, &sms);
  if (st != EP_OK) return st;
  const ep::RouteCountArgs r = route_count_args(cfg, nullptr, nullptr, nullptr, a);
  switch (choose_form(cfg, r, a, sms)) {
    case Form::kSingle: *kernels = 1; break;
    case Form::kCluster: *kernels = 2; break;
    case Form::kChain: *kernels = cfg->T > 0 ? 3 : 2; break;  // route+count, scan, scatter (none when empty)
  }
  return EP_OK;
}

ep_status_t ep_debug_set(int32_t option, int32_t value) {
  switch (option) {
    case EP_DEBUG_FORCE_WAIT_TIMEOUT:
      ep::set_force_wait_timeout(value);
      return EP_OK;
    case EP_DEBUG_ROUTE_DISPATCH_FORM:
      if (value < EP_FORM_AUTO || value > EP_FORM_CHAIN) return EP_ERR_INVALID_ARG;
      ep::cache_store(&g_route_dispatch_form, value);
      return EP_OK;
  }
  return EP_ERR_INVALID_ARG;
}

ep_status_t ep_load_stats(const int32_t* host_counts, int32_t E, ep_load_stats_t* out) {
  if (host_counts == nullptr || out == nullptr || E < 1) return EP_ERR_INVALID_ARG;
  int64_t total = 0;
  int32_t mn = host_counts[0], mx = host_counts[0];
  for (int32_t e = 0; e < E; ++e) {
    total += host_counts[e];
    if (host_counts[e] < mn) mn = host_counts[e];
    if (host_counts[e] > mx) mx = host_counts[e];
  }
  const double mean = static_cast<double>(total) / E;
  double var = 0.0;
  for (int32_t e = 0; e < E; ++e) {
    const double d = host_counts[e] - mean;
    var += d * d;
  }
  var /= E;
  out->mean = mean;
  out->stddev = sqrt(var);
  out->cv = mean > 0.0 ? out->stddev / mean : 0.0;
  out->min = mn;
  out->max = mx;
  out->total = total;
  return EP_OK;
}

}  // extern "C"
