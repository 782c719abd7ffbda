/*
 * ep.h — C ABI of libep_b300: MoE expert-parallel token dispatch and combine
 * on one NVIDIA B300 (sm_103a).
 *
 * The path (pages cited by title and section):
 *   ep_route     top-k gating with softmax weights over fp32 router logits
 *                (MoE sparse-communication article, intelliparadigm.com, §2.1
 *                 Router listing: softmax over the logits, then topk)
 *   ep_dispatch  group every (token, slot) copy by destination into one
 *                contiguous rank-major buffer — "aggregate by target card"
 *                (ThunderEP on consumer GPUs, bjdmk.com.cn, §2.1) with the
 *                flat [rank0_data, rank1_data, ...] layout whose segments
 *                start at running sums of the counts (NCCL EP article,
 *                hotelren.com, §3.3) — fused with optional per-token dynamic
 *                int8 compression (ThunderEP §2.3)
 *   ep_combine   gate-weighted sum of each token's k expert outputs at its
 *                source (ThunderEP §1.3 steps 3-4; §3.3 combine), fp32
 *                accumulate in fixed slot order
 * The R expert-parallel ranks are virtual: expert e belongs to rank e/(E/R)
 * (MoE communication-wall explainer, juhe.plus, "64 experts on 8 GPUs"), and
 * rank r's send block is payload rows [rank_off[r], rank_off[r+1]).
 *
 * Conventions for every call:
 *   - All array pointers are caller-owned device memory unless stated; the
 *     library allocates nothing and keeps no state between calls apart from
 *     per-device launch settings. Scratch comes from a caller-provided
 *     workspace sized by ep_workspace_size(). Its counters and wait words
 *     need no reset between calls (each call leaves them as the next one
 *     expects); calls that share a workspace must not run at the same time
 *     on the GPU (issue them on one stream, or order them with events).
 *   - Calls are asynchronous on the given stream (0 = legacy default stream)
 *     and never synchronise it, except ep_get_error().
 *   - Errors are returned, never raised by exit/abort (the NCCL EP article,
 *     §4.2-4.3, on returning errors instead of hanging or exiting). Argument
 *     checks run on the host before any launch: a call that returns
 *     EP_ERR_INVALID_ARG or EP_ERR_WORKSPACE has enqueued nothing.
 *   - Index inputs that come from the caller (topk_idx, slot_row) are checked
 *     on the device too: an out-of-range or repeated entry is never used as an
 *     address; it sets EP_ERR_DEVICE_INDEX in the workspace's status word,
 *     which ep_get_error() reports.
 *   - Alignment: float and bf16 arrays 16-byte aligned; int32 arrays 4-byte.
 *   - Layouts are row-major and dense (no strides).
 */
#ifndef EP_B300_H_
#define EP_B300_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EP_OK = 0,
  EP_ERR_INVALID_ARG = 1,  /* bad config, null or misaligned pointer      */
  EP_ERR_WORKSPACE = 2,    /* workspace missing or smaller than required */
  EP_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed        */
  EP_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up          */
  EP_ERR_DEVICE_INDEX = 5  /* an index input was out of range or repeated */
} ep_status_t;

typedef enum {
  EP_PAYLOAD_BF16 = 0,     /* rows are the token's bf16 bytes, unchanged                   */
  EP_PAYLOAD_INT8 = 1,     /* rows are the token's int8 code + one fp32 scale per row      */
  EP_PAYLOAD_FP8_E4M3 = 2, /* rows are the token's FP8 E4M3 code + one fp32 scale per row  */
  EP_PAYLOAD_INT4 = 3      /* rows of H/2 bytes: the token's 4-bit code, two per byte, + one
                              fp32 scale per row (H % 32 == 0)                              */
} ep_payload_t;

/*
 * Problem statement (ThunderEP §1.3: T tokens, hidden size, E experts, top-k,
 * N cards; juhe.plus all-to-all volume 2*T*k*H*b).
 *   T                tokens in the batch, >= 0
 *   H                hidden size, 16 <= H <= 16384, H % 16 == 0 (H % 32 == 0
 *                    with the int4 payload)
 *   E                experts, 1 <= E <= 1024
 *   k                experts per token, 1 <= k <= min(E, 32)
 *   R                virtual ranks, R >= 1, E % R == 0
 *   capacity_factor  <= 0: dropless. > 0: each expert keeps at most
 *                    cap = ceil(capacity_factor * T * k / E) copies (evaluated
 *                    in double, in that order); further (token, slot) pairs
 *                    are dropped in (token, slot) order and their weight is
 *                    excluded from the combine (intelliparadigm §2.1 capacity
 *                    factor, typical 1.0-1.25)
 *   renormalize      0: w = full softmax probability of the chosen expert;
 *                    1: the k chosen weights are rescaled to sum to one
 *   payload          EP_PAYLOAD_BF16, EP_PAYLOAD_INT8 or EP_PAYLOAD_FP8_E4M3 for
 *                    ep_dispatch
 * The per-token codes (ThunderEP §2.3 per-token dynamic quantisation; §5.2
 * and the NCCL EP article §6.3 for FP8):
 *   int8  scale = amax/127.0f, q = clamp(rint(x/scale), -127, 127)
 *   FP8   scale = amax/448.0f, q = E4M3 round-to-nearest-even of x/scale,
 *         saturated to +-448 (OCP E4M3: bias 7, 3 mantissa bits, no inf)
 *   int4  scale = amax/7.0f, q = clamp(rint(x/scale), -7, 7) as a
 *         two's-complement nibble; byte i of a row holds elements 2i (low
 *         nibble) and 2i+1 (high nibble)
 * with IEEE fp32 division and amax = 0 giving scale 0 and all-zero codes.
 */
typedef struct {
  int32_t T, H, E, k, R;
  float capacity_factor;
  int32_t renormalize;
  int32_t payload; /* ep_payload_t */
} ep_config_t;

/* Human-readable name of a status code (static storage). */
const char* ep_status_string(ep_status_t s);

/* Checks a config against the limits above (host only). */
ep_status_t ep_config_check(const ep_config_t* cfg);

/* Per-expert cap (T when dropless). Host only. */
ep_status_t ep_capacity(const ep_config_t* cfg, int32_t* cap);

/* Rows the dispatch buffers must hold: T*k dropless, else min(T*k, E*cap).
 * Returns 0 for an invalid config. Host only. */
int64_t ep_max_rows(const ep_config_t* cfg);

/* Workspace bytes needed by ep_dispatch / ep_combine for this config. The
 * size grows with T*k (a 4-byte rank per pair) plus E*ceil(T/tile) counters.
 * Host only. */
ep_status_t ep_workspace_size(const ep_config_t* cfg, size_t* bytes);

/* Zero a freshly allocated workspace (its status word must start clear).
 * Enqueued on `stream`. Needed once per allocation, not per call. */
ep_status_t ep_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * ep_route — top-k gating (intelliparadigm §2.1 Router; NCCL EP §3.4 step 1).
 *   logits    [T, E] fp32 in   router scores (kept in fp32: the NCCL EP
 *                              article, §6.3, warns that low-precision scores
 *                              distort top-k)
 *   topk_idx  [T, k] int32 out expert ids, slot j = j-th by (logit desc,
 *                              expert id asc); ties go to the lower id
 *   topk_w    [T, k] fp32 out  softmax weight of each chosen expert (see
 *                              ep_config_t.renormalize); within 1e-6 relative
 *                              of the exactly rounded value
 * NaN/Inf logits are outside the contract (they are never used as addresses).
 */
ep_status_t ep_route(const ep_config_t* cfg, const float* logits, int32_t* topk_idx, float* topk_w,
                     cudaStream_t stream);

/*
 * ep_dispatch — rank-major send layout plus its inverse (ThunderEP §2.1 and
 * §2.3; NCCL EP §3.3 sendcounts/flat sendbuff).
 *   x              [T, H] bf16 in     token hidden states
 *   topk_idx       [T, k] int32 in    k distinct expert ids per token
 *   payload        [max_rows, H] out  bf16 (EP_PAYLOAD_BF16), int8
 *                                     (EP_PAYLOAD_INT8) or E4M3 bytes
 *                                     (EP_PAYLOAD_FP8_E4M3), or [max_rows,
 *                                     H/2] packed int4 (EP_PAYLOAD_INT4);
 *                                     rows [0, N) are
 *                                     written, N = T*k - dropped; row order is
 *                                     (expert, token), so rank r's block is
 *                                     rows [rank_off[r], rank_off[r+1])
 *   scales         [max_rows] fp32 out one scale per row (int8 and FP8; NULL
 *                                     in bf16 mode), codes as in ep_config_t
 *   row_slot       [max_rows] int32 out row -> t*k + j, rows [0, N)
 *   slot_row       [T*k] int32 out    (t, j) -> row, or -1 if dropped
 *   expert_counts  [E] int32 out      kept copies per expert
 *   expert_raw     [E] int32 out      copies per expert before the cap (may be NULL)
 *   expert_off     [E+1] int32 out    exclusive running sum of expert_counts
 *   rank_off       [R+1] int32 out    rank_off[r] = expert_off[r*E/R] (the
 *                                     send displacements; rank_off[R] = N)
 *   n_dropped      [1] int32 out      pairs dropped by the cap
 *   ws, ws_bytes   workspace from ep_workspace_size(), initialised once
 * Counts and offsets stay on the device; copy rank_off back if the host needs N.
 */
ep_status_t ep_dispatch(const ep_config_t* cfg, const void* x, const int32_t* topk_idx, void* payload,
                        float* scales, int32_t* row_slot, int32_t* slot_row, int32_t* expert_counts,
                        int32_t* expert_raw, int32_t* expert_off, int32_t* rank_off, int32_t* n_dropped,
                        void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * ep_route_dispatch — ep_route followed by ep_dispatch in one call, with the
 * routing fused into the dispatch (ThunderEP on consumer GPUs, bjdmk.com.cn,
 * §5.2: do the bucketing by destination while routing, saving a pass; the
 * Perseus summary, itsolotime.com, §1.3: one persistent kernel for the whole
 * exchange). Every output is bit-for-bit what
 *   ep_route(cfg, logits, topk_idx, topk_w, stream);
 *   ep_dispatch(cfg, x, topk_idx, payload, ..., ws, ws_bytes, stream);
 * would write; the arguments mean what they mean there (logits [T, E] fp32
 * in, 16-byte aligned; topk_idx / topk_w [T, k] out).
 * Single-launch form (by default when 32 <= E <= 256, or T >= 8192 with
 * E <= 256; at most 1024 tokens per SM, x 32-byte aligned, cooperative
 * launch available): one cooperative launch of one CTA per SM does it all.
 * Each CTA routes its own tile of ceil(T / SMs) tokens; one device-wide wait;
 * each CTA forms its tile's positions from every tile's counts (small
 * batches: from all the routed ids) and writes its pairs' rows; then it
 * scatters the first tokens of its own tile and, after a second device-wide
 * wait, takes the rest of every tile from a shared counter (small batches:
 * each CTA its whole tile, nothing shared). Those waits are bounded (about a
 * second); if one runs out the call's outputs are not valid and
 * ep_get_error() reports EP_ERR_TIMEOUT (and resets the waits' words in the
 * workspace, so the workspace can be used again).
 * Otherwise three kernels run: a CTA routes one tile of tokens and counts its
 * per-expert copies in shared memory, then the scan and the scatter of
 * ep_dispatch; a batch of at most 256 tokens with E <= 256 then takes two
 * (one thread-block cluster routes it and forms the whole layout, then the
 * scatter).
 */
ep_status_t ep_route_dispatch(const ep_config_t* cfg, const float* logits, const void* x, int32_t* topk_idx,
                              float* topk_w, void* payload, float* scales, int32_t* row_slot, int32_t* slot_row,
                              int32_t* expert_counts, int32_t* expert_raw, int32_t* expert_off, int32_t* rank_off,
                              int32_t* n_dropped, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * ep_route_dispatch_kernels — how many kernels ep_route_dispatch launches for
 * `cfg` on the current device (1: the single cooperative launch; 2: the
 * cluster form; 3: the chain, or 2 for an empty batch), taking x as 32-byte
 * aligned; host only, launches nothing. *kernels out.
 */
ep_status_t ep_route_dispatch_kernels(const ep_config_t* cfg, int32_t* kernels);

/*
 * ep_bitmap_encode — compact routing metadata (MoE sparse-communication
 * article, intelliparadigm.com, §4.1: the index of [expert, position] entries
 * sent with each copy becomes one bitmap per token).
 *   topk_idx  [T, k] int32 in    k distinct expert ids per token
 *   bitmap    [T, W] uint32 out  W = (E + 31) / 32; bit e % 32 of word e / 32
 *                                is set iff the token chose expert e
 *   ws        workspace (its status word records out-of-range or repeated ids)
 * 4*W bytes per token take the place of k (expert id, position) pairs of
 * 4 + 4 bytes (E = 128, k = 8: 16 bytes against 64).
 */
ep_status_t ep_bitmap_encode(const ep_config_t* cfg, const int32_t* topk_idx, uint32_t* bitmap, void* ws,
                             size_t ws_bytes, cudaStream_t stream);

/*
 * ep_bitmap_layout — what a receiving rank rebuilds from the bitmaps alone:
 * the same expert_counts, expert_raw (may be NULL), expert_off, rank_off and
 * n_dropped as ep_dispatch, and row_token[row] = the source token of each of
 * the rows [0, N) of the rank-major buffer (ep_dispatch's row_slot[row] / k).
 * The layout depends only on which experts each token chose (rows within an
 * expert are in token order, the cap drops the latest tokens), not on the
 * slot order, so nothing else has to travel with the data.
 *   bitmap     [T, W] uint32 in   each token with exactly k bits set (fewer,
 *                                 more, or bits at or above E set
 *                                 EP_ERR_DEVICE_INDEX in the status word)
 *   row_token  [max_rows] int32 out
 *   ws         workspace from ep_workspace_size(), initialised once
 */
ep_status_t ep_bitmap_layout(const ep_config_t* cfg, const uint32_t* bitmap, int32_t* row_token,
                             int32_t* expert_counts, int32_t* expert_raw, int32_t* expert_off, int32_t* rank_off,
                             int32_t* n_dropped, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * ep_dispatch_static — ep_dispatch for callers that cannot allocate device
 * memory. The pages have no counterpart to this call: it exists only for
 * this library's users.
 *
 * Some callers cannot provide the workspace ep_dispatch needs: a plugin or
 * custom-op host that passes an operator only its inputs and outputs and
 * forbids allocation inside the enqueue call, a runtime that plans every
 * device allocation ahead of time, or a latency-critical path that cannot
 * afford cudaMalloc's implicit synchronisation. This call takes the same
 * arguments as ep_dispatch minus the workspace, runs the same kernels, and
 * keeps its scratch in a fixed device array of EP_STATIC_SCRATCH_BYTES inside
 * the library, which every GPU that loads the library holds until exit. It
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Limit: a problem whose ep_workspace_size() exceeds
 *     EP_STATIC_SCRATCH_BYTES is refused with EP_ERR_WORKSPACE before
 *     anything is enqueued (the scratch is about 4*T*k + 8*E*ceil(T/tile)
 *     bytes plus 2 KB: T=131072, k=8, E=256 needs about 4.6 MB).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture starts.
 *   - All calls share the one array and each call starts by clearing the part
 *     that must begin at zero. Calls whose work overlaps on the GPU (other
 *     streams, other host threads on the same device) race on it: serialise
 *     them.
 *   - Device-side index checks still guard every access, but their status
 *     word lives in the shared array, so ep_get_error cannot report them;
 *     diagnose bad indices with ep_dispatch and a workspace.
 */
#define EP_STATIC_SCRATCH_BYTES (8u * 1024u * 1024u)

ep_status_t ep_dispatch_static(const ep_config_t* cfg, const void* x, const int32_t* topk_idx, void* payload,
                               float* scales, int32_t* row_slot, int32_t* slot_row, int32_t* expert_counts,
                               int32_t* expert_raw, int32_t* expert_off, int32_t* rank_off, int32_t* n_dropped,
                               cudaStream_t stream);

/*
 * ep_combine — weighted top-k recombination (ThunderEP §1.3 steps 3-4).
 *   expert_out   [max_rows, H] in  bf16 (out_payload = EP_PAYLOAD_BF16), int8
 *                                  (EP_PAYLOAD_INT8) or E4M3 bytes
 *                                  (EP_PAYLOAD_FP8_E4M3), or [max_rows, H/2]
 *                                  packed int4 (EP_PAYLOAD_INT4) expert
 *                                  outputs, row-aligned with the dispatch
 *                                  payload
 *   out_scales   [max_rows] fp32   per-row scales for int8 / FP8 / int4 rows,
 *                                  else NULL
 *   slot_row     [T*k] int32 in    from ep_dispatch (-1 = dropped slot)
 *   topk_w       [T, k] fp32 in    from ep_route
 *   y            [T, H] bf16 out   y[t] = bf16_rne(sum over j = 0..k-1 in
 *                                  order, slot not dropped, of
 *                                  fmaf(w[t,j], v_j, acc)), acc starting at 0,
 *                                  v_j = float(bf16) or (float)q * scale
 *                                  (q the int8, E4M3 or int4 code, widened
 *                                  exactly)
 *   ws, ws_bytes workspace, at least 256 bytes (its status word records bad
 *                slot_row entries; two words at byte 64 count the units of
 *                work that the warps take, and are zero again on return)
 * A token whose k slots were all dropped gets y = 0. The E4M3 NaN codes (0x7F,
 * 0xFF), which no encoder of this library writes, are outside the contract
 * (they read as +-480).
 */
ep_status_t ep_combine(const ep_config_t* cfg, const void* expert_out, const float* out_scales,
                       int32_t out_payload, const int32_t* slot_row, const float* topk_w, void* y,
                       void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * ep_quantize_rows — the per-token int8 code applied to n rows of width H
 * (ThunderEP §2.3), for an expert side that returns int8 outputs.
 *   in      [n, H] bf16 in;  q [n, H] int8 out;  scales [n] fp32 out.
 *   H % 16 == 0, 16 <= H <= 16384.
 */
ep_status_t ep_quantize_rows(const void* in, int64_t n, int32_t H, int8_t* q, float* scales,
                             cudaStream_t stream);

/*
 * ep_quantize_rows_fp8 — the per-token FP8 E4M3 code (scale = amax/448) of n
 * rows, for an expert side that returns FP8 outputs; as ep_quantize_rows
 * otherwise (q [n, H] E4M3 bytes out, 16-byte aligned).
 */
ep_status_t ep_quantize_rows_fp8(const void* in, int64_t n, int32_t H, uint8_t* q, float* scales,
                                 cudaStream_t stream);

/*
 * ep_quantize_rows_int4 — the per-token 4-bit code (scale = amax/7) of n rows,
 * for an expert side that returns 4-bit outputs: q [n, H/2] packed nibbles
 * out (16-byte aligned), H % 32 == 0; as ep_quantize_rows otherwise.
 */
ep_status_t ep_quantize_rows_int4(const void* in, int64_t n, int32_t H, uint8_t* q, float* scales,
                                  cudaStream_t stream);

/*
 * ep_get_error — synchronises `stream`, reads the workspace's status word,
 * clears it, and returns EP_OK, EP_ERR_DEVICE_INDEX or EP_ERR_TIMEOUT (or
 * EP_ERR_CUDA if the stream itself failed). The one call that blocks. After
 * EP_ERR_TIMEOUT it also resets the words of the device-wide waits.
 */
ep_status_t ep_get_error(void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * ep_debug_set — process-wide test hooks (not for production use); returns
 * EP_OK, or EP_ERR_INVALID_ARG for an unknown option.
 *   EP_DEBUG_FORCE_WAIT_TIMEOUT (value 0/1): while set, the device-wide wait
 *     of ep_route_dispatch's single-launch form counts one CTA more than the
 *     launch has and gives up after about a millisecond, so every such call
 *     made meanwhile reports EP_ERR_TIMEOUT through ep_get_error() and leaves
 *     its outputs invalid (the NCCL EP article, §4.2-4.3: a wait that cannot
 *     complete must end in an error, not a hang).
 *   EP_DEBUG_ROUTE_DISPATCH_FORM (value EP_FORM_*): which form of
 *     ep_route_dispatch runs: the library's choice by batch shape (AUTO), the
 *     single cooperative launch wherever it can run (SINGLE), or the kernel
 *     chain (CHAIN). Every form writes the same bytes.
 */
typedef enum { EP_DEBUG_FORCE_WAIT_TIMEOUT = 1, EP_DEBUG_ROUTE_DISPATCH_FORM = 2 } ep_debug_option_t;
typedef enum { EP_FORM_AUTO = 0, EP_FORM_SINGLE = 1, EP_FORM_CHAIN = 2 } ep_route_dispatch_form_t;
ep_status_t ep_debug_set(int32_t option, int32_t value);

/*
 * Load statistics over per-expert counts already copied to the host
 * (intelliparadigm §2.1: watch the spread of expert calls; coefficient of
 * variation below 0.3 is the healthy range; NCCL EP §5.3 ncclEpStats_t idea).
 */
typedef struct {
  double mean, stddev, cv; /* population standard deviation; cv = stddev/mean */
  int32_t min, max;
  int64_t total;
} ep_load_stats_t;

ep_status_t ep_load_stats(const int32_t* host_counts, int32_t E, ep_load_stats_t* out);

#ifdef __cplusplus
}
#endif

#endif /* EP_B300_H_ */
