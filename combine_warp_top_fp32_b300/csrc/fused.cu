// fused.cu — ep_route_dispatch in one cooperative launch: route, lay out and
// scatter a batch with one CTA per SM.
//
// The ThunderEP article (bjdmk.com.cn, §5.2) suggests fusing the bucketing by
// destination with the routing; the Perseus summary (itsolotime.com, §1.3)
// runs the whole exchange as one persistent kernel. Here, on one GPU, one
// cooperative launch of G CTAs (one per SM) does the three steps of the
// dispatch, each CTA routing its own tile of consecutive tokens
// (tile = ceil(T / G), so every SM routes the same number of tokens):
//
//   A  route the tile (route_device.cuh): topk_idx / topk_w, and per-expert
//      bit masks of the tile's tokens in shared memory, whose popcounts give
//      the tile's count per expert (written to counts[b][e]) and every pair's
//      rank within the tile in token order. Small batches only: meanwhile the
//      copy engine brings the tile's x rows into shared memory.
//   -- grid barrier 1 (grid_sync.cuh): every tile's routing is written --
//   B  every CTA forms, for each expert, the number of its pairs in earlier
//      tiles (this tile's first position within the expert) and its total:
//      from all G x E tile counts, or, for small batches, from all T*k routed
//      ids. The capacity clip and the expert and rank offsets follow (NCCL EP
//      article, hotelren.com, §3.3: running sums of the send counts); CTA 0
//      writes the layout outputs; each CTA writes its own pairs' rows
//      (slot_row / row_slot).
//   -- grid barrier 2, split: each CTA arrives when its pairs' rows are
//      written and waits only before it takes another tile's tokens --
//   C  scatter the payload: bf16 copies (a warp per token) or the per-token
//      int8 / FP8 / int4 code (ThunderEP §2.3; a group of warps per token with
//      its own named barrier). First the first tokens of the CTA's own tile,
//      then (after barrier 2) the rest of every tile from one shared counter,
//      so that the SMs, which move data at different speeds, and the tokens,
//      whose kept rows differ (capacity drops fall on the later ones), even
//      out. Small batches: each CTA its own tile, x from shared memory, and
//      nothing shared.
//
// Both barriers count arrivals on one word (count_barrier, split_arrive): the
// first completes at G arrivals, the second at 2G, whose last arrival zeroes
// the words for the next launch.
//
// Every output equals that of route_count_kernel + scan_kernel + the scatter
// kernels, bit for bit (the same routing, the same row rule, the same codes).
#include "ep_internal.h"
#include "grid_sync.cuh"
#include "route_device.cuh"


namespace ep {
namespace {

using namespace routing;

constexpr int kFusedBlock = 768;  // one CTA per SM; 24 warps leave 85 registers a thread, so neither phase spills
constexpr int kFusedMaxGroups = 15;     // named barriers 1..15: at most 15 token groups
constexpr long long kBarrierPolls = 1ll << 20;  // about a second of polling before a wait gives up
constexpr long long kCopyPolls = 1ll << 22;
// The scatter's own part is kOwnPerGroup tokens for each token group of the
// CTA in the coded scatter and kOwnPerWarp for each warp in the bf16 one (at
// most the tile): enough work that a group rarely finds the second grid
// barrier incomplete (every group's first thread polls it then), and little
// enough on large tiles that the shared part, whose concurrent tokens are
// neighbours in the batch (so are the payload rows they write), does most
// of the work.
constexpr int kOwnPerGroup = 8;
constexpr int kOwnPerWarp = 4;

// Warps per token in the coded scatter (each thread codes 32 elements) and
// token groups per CTA.
__host__ __device__ constexpr int coded_group_warps(int H) { return ((((H >> 4) + 1) >> 1) + 31) >> 5; }
__host__ __device__ constexpr int coded_groups(int H) {
  return (kFusedBlock / 32) / coded_group_warps(H) < kFusedMaxGroups ? (kFusedBlock / 32) / coded_group_warps(H)
                                                                      : kFusedMaxGroups;
}
// x rows are preloaded into shared memory only when a whole tile's rows fit in
// kPreloadBytes (small batches: each CTA then scatters exactly its own tile,
// with no wait on any other CTA). Otherwise nothing is preloaded: the SM's
// unified L1 / shared storage then stays L1, through which every global load
// in flight passes, and a large preload costs the scatter more than it saves.
constexpr int64_t kPreloadBytes = 64 * 1024;
// At most this many (token, slot) pairs: each CTA forms the layout from the
// routed expert ids of the whole batch (T*k ids, one coalesced read) instead
// of from every tile's per-expert counts (G*E values, most of them zero).
constexpr int64_t kSmallLayoutPairs = 8192;

struct FusedArgs {
  const float* logits;
  const void* x;
  int T, H, E, k, R, cap, renorm, lanes_log2;
  int tile, TW;        // tokens per tile, mask words per expert (a power of two)
  int npre;            // x rows preloaded per CTA (its own tile's), 0 for none
  int own_tile;        // 1: each CTA scatters its whole tile (nothing shared, no wait at the second barrier)
  int small_layout;    // 1: the layout comes from the routed ids, not the tile counts
  int32_t* topk_idx;
  float* topk_w;
  void* payload;
  float* scales;
  int32_t *row_slot, *slot_row, *expert_counts, *expert_raw, *expert_off, *rank_off, *n_dropped;
  int32_t* counts;  // workspace: [G][E] per-tile counts
  uint32_t* status;
  GridBarrier bar;
  unsigned* work;  // the scatter's shared token counter, zeroed by the second barrier's last arrival
  int extra_arrivals;  // > 0 only when a test forces the barrier to time out
  long long barrier_polls;
};

// Shared memory of the fused kernel (dynamic, carved in this order).
struct FusedSmem {
  unsigned char* xpre;  // [npre][2H] preloaded x rows (128-byte aligned)
  uint32_t* mask;       // [E][TW] bit b of word w: tile token 32w+b chose e
  uint32_t* pre;        // [E][TW] set bits of e in the words before w
  int* base;            // [E] pairs of e in earlier tiles
  int* kept;            // [E] kept pairs of e (then the expert offsets)
  uint8_t* ids;         // [32 TW][k] the expert of each pair of the tile (E <= 256), from the routing
};

__host__ __device__ inline size_t fused_smem_fixed(int E, int TW, int k) {
  return static_cast<size_t>(E) * TW * 8 + static_cast<size_t>(E) * 8 + ((static_cast<size_t>(32) * TW * k + 15) & ~15ull) +
         64;
}

__device__ __forceinline__ FusedSmem carve_fused(unsigned char* smem, int E, int TW, int npre, int H) {
  FusedSmem s;
  s.xpre = smem;
  unsigned char* p = smem + static_cast<size_t>(npre) * 2 * H;
  s.mask = reinterpret_cast<uint32_t*>(p);
  s.pre = s.mask + E * TW;
  s.base = reinterpret_cast<int*>(s.pre + E * TW);
  s.kept = s.base + E;
  s.ids = reinterpret_cast<uint8_t*>(s.kept + E);
  return s;
}

__device__ __forceinline__ void group_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Destination row of tile token tl's slot j (expert e): this tile's first
// position within e, plus the token's rank among the tile's tokens that chose
// e, placed at e's offset; -1 past the capacity. Writes slot_row / row_slot.
__device__ __forceinline__ int fused_row(const FusedArgs& a, const FusedSmem& s, int64_t t, int tl, int j) {
  const int64_t p = t * a.k + j;
  const int e = s.ids[tl * a.k + j];  // the routed expert, kept in shared memory by this CTA
  const int w = tl >> 5;
  const int r = static_cast<int>(s.pre[e * a.TW + w]) + __popc(s.mask[e * a.TW + w] & ((1u << (tl & 31)) - 1u));
  const int pos = s.base[e] + r;
  const int row = pos < a.cap ? s.kept[e] + pos : -1;
  a.slot_row[p] = row;
  if (row >= 0) a.row_slot[row] = static_cast<int32_t>(p);
  return row;
}

// 32 bytes (16 bf16) of x per thread, from global memory (evict-first in L2).
__device__ __forceinline__ void ld_x32_global(const char* p, uint4& lo, uint4& hi) {
  asm volatile("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
               : "l"(p));
}

// Per-tile mask word prefixes (as tile_word_prefix) with the tile's count of
// expert e written to counts_b[e].
__device__ __forceinline__ void tile_word_prefix_row(const uint32_t* mask, uint32_t* pre, int E, int TW,
                                                     int32_t* __restrict__ counts_b) {
  const int lane = threadIdx.x & 31;
  const int n = E * TW;
  for (int i0 = 0; i0 < n; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    const bool ok = i < n;
    const int c = ok ? __popc(mask[i]) : 0;
    int v = c;
    for (int o = 1; o < TW; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if ((lane & (TW - 1)) >= o) v += u;
    }
    if (ok) {
      pre[i] = static_cast<uint32_t>(v - c);
      if ((i & (TW - 1)) == TW - 1) counts_b[i / TW] = v;
    }
  }
}

// Per-expert sums over every tile's counts for this CTA's tile b: base[e] =
// pairs of e in tiles before b, total[e] = all pairs of e (both zeroed by the
// caller). Warp w reads whole count rows g = w, w + 32, ... (lane l holds
// experts 4l..4l+3, 4(l+32).., so a row is one coalesced read), four rows'
// loads in flight before any is added; the 32 warps' partial sums meet in
// shared memory by atomic adds. E % 4 == 0 reads int4, else one int per lane.
__device__ __forceinline__ void tile_bases(const int32_t* __restrict__ counts, int G, int E, int b, int* base,
                                           int* total) {
  constexpr int NW = kFusedBlock / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((E & 3) == 0) {
    const int C4 = E >> 2;  // <= 64 int4 columns (E <= 256)
    int4 bf[2] = {make_int4(0, 0, 0, 0), make_int4(0, 0, 0, 0)};
    int4 tt[2] = {make_int4(0, 0, 0, 0), make_int4(0, 0, 0, 0)};
    if (C4 <= 32) {  // E <= 128: one int4 per lane per row, all of a warp's rows in flight at once
      constexpr int RW = (kFusedMaxCTAs + NW - 1) / NW;
      int4 v[RW];
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        const int g = warp + r * NW;
        v[r] = (g < G && lane < C4) ? __ldcg(reinterpret_cast<const int4*>(counts + static_cast<int64_t>(g) * E) + lane)
                                    : make_int4(0, 0, 0, 0);
      }
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        tt[0].x += v[r].x; tt[0].y += v[r].y; tt[0].z += v[r].z; tt[0].w += v[r].w;
        if (warp + r * NW < b) { bf[0].x += v[r].x; bf[0].y += v[r].y; bf[0].z += v[r].z; bf[0].w += v[r].w; }
      }
    } else
    for (int g0 = warp; g0 < G; g0 += 4 * NW) {
      int4 v[4][2];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int g = g0 + r * NW;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = lane + 32 * h;
          v[r][h] = (g < G && c < C4)
                        ? __ldcg(reinterpret_cast<const int4*>(counts + static_cast<int64_t>(g) * E) + c)
                        : make_int4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const bool before = g0 + r * NW < b;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          tt[h].x += v[r][h].x; tt[h].y += v[r][h].y; tt[h].z += v[r][h].z; tt[h].w += v[r][h].w;
          if (before) { bf[h].x += v[r][h].x; bf[h].y += v[r][h].y; bf[h].z += v[r][h].z; bf[h].w += v[r][h].w; }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = lane + 32 * h;
      if (c < C4) {
        atomicAdd(&base[4 * c], bf[h].x); atomicAdd(&base[4 * c + 1], bf[h].y);
        atomicAdd(&base[4 * c + 2], bf[h].z); atomicAdd(&base[4 * c + 3], bf[h].w);
        atomicAdd(&total[4 * c], tt[h].x); atomicAdd(&total[4 * c + 1], tt[h].y);
        atomicAdd(&total[4 * c + 2], tt[h].z); atomicAdd(&total[4 * c + 3], tt[h].w);
      }
    }
  } else {
    int bf[8] = {0, 0, 0, 0, 0, 0, 0, 0}, tt[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // experts lane + 32 h
    for (int g = warp; g < G; g += NW) {
      const bool before = g < b;
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const int e = lane + 32 * h;
        const int v = e < E ? __ldcg(counts + static_cast<int64_t>(g) * E + e) : 0;
        tt[h] += v;
        if (before) bf[h] += v;
      }
    }
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const int e = lane + 32 * h;
      if (e < E) {
        atomicAdd(&base[e], bf[h]);
        atomicAdd(&total[e], tt[h]);
      }
    }
  }
}

// The scatter's tokens, in two parts. Own part: the first `own` tokens of
// each tile (the same number in every tile), scattered by the tile's CTA
// straight after it has written its rows, its groups (warps) taking them in
// turn: no atomic, and no wait on any other CTA. Shared part: the rest of
// every tile, handed out by one counter to every group of every CTA (so that
// SMs that run faster, and tiles with fewer kept rows, even out: capacity
// drops fall on the batch's later tokens). A group takes from the counter
// only after the second grid barrier, which each CTA arrives at when its rows
// are written and waits for only once its own part is done, by when the
// barrier has normally completed. Counter value p is token
// (p / (tile - own)) * tile + own + p % (tile - own); values past the batch
// end the sequence. A value is asked for (issue) one token before it is read
// (resolve), so no group waits on the atomic. One thread per group calls
// these.
struct TokenPlan {
  unsigned* work;           // the shared counter (zeroed when the second barrier completes)
  const unsigned* round;    // the grid barrier's round word
  uint32_t* status;
  unsigned round_before;    // the round while the second barrier is incomplete
  int T, tile, own, t0, own_end;
};

// ticket >= 0: a token of the own part; < 0: -(counter value + 1).
__device__ __forceinline__ int plan_issue(const TokenPlan& tp, int& own_next, int step, bool& shared_ok) {
  if (own_next < tp.own_end) {
    const int t = own_next;
    own_next += step;
    return t;
  }
  if (tp.own >= tp.tile) return -1;  // own-tile mode: no shared part (resolves past the batch)
  if (!shared_ok) {  // the second barrier: every tile's rows are written
    long long polls = 0;
    while (ld_acquire_gpu(tp.round) == tp.round_before) {
      if (++polls > kBarrierPolls) {
        raise_status(tp.status, kStatusTimeout);
        return -1 - 0x3fffffff;  // past every token: ends the sequence
      }
      __nanosleep(16);
    }
    shared_ok = true;
  }
  return -1 - static_cast<int>(atomicAdd(tp.work, 1u));
}

__device__ __forceinline__ int plan_resolve(const TokenPlan& tp, int ticket) {
  if (ticket >= 0) return ticket;
  const int p = -1 - ticket;
  const int per = tp.tile - tp.own;
  if (per <= 0) return tp.T;
  const int64_t t = static_cast<int64_t>(p / per) * tp.tile + tp.own + p % per;
  return t < tp.T ? static_cast<int>(t) : tp.T;
}

template <int VPL, bool VEC4, int FMT>
__global__ void __launch_bounds__(kFusedBlock, 1) route_dispatch_fused_kernel(const FusedArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t xbar;  // the preloaded rows' bulk copies
  __shared__ int32_t rows_s[kFusedMaxGroups][3][32];  // per token group: its next tokens' rows (three deep)
  __shared__ float amax_s[kFusedMaxGroups][2][16];    // per token group: its warps' amax
  __shared__ int ids_s[kFusedMaxGroups][2];           // per token group: the token after next
  __shared__ int scan_s[16];                          // the offsets' warp sums and drops
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x, G = gridDim.x;
  const int64_t t0 = static_cast<int64_t>(b) * a.tile;
  const int nt = static_cast<int>(min(static_cast<int64_t>(a.tile), a.T - t0));  // >= 1: G = ceil(T / tile)
  const int P = min(a.npre, nt);          // preloaded tokens of this CTA's own tile (the last may be short)
  const int tail0 = static_cast<int>(t0);  // the preloaded rows are tokens [t0, t0 + P)
  const bool own_tile = a.own_tile != 0;  // the CTA scatters its own tile (and never waits at the second barrier)
  const int64_t row_bytes = 2 * static_cast<int64_t>(a.H);
  FusedSmem s = carve_fused(smem_raw, a.E, a.TW, P, a.H);

  // tokens of the scatter's own part (TokenPlan): the whole tile in own-tile mode
  int own = a.tile;
  if (!own_tile) {
    if constexpr (FMT == kFmtBf16)
      own = min(a.tile, kOwnPerWarp * (kFusedBlock / 32));
    else
      own = min(a.tile, kOwnPerGroup * coded_groups(a.H));
  }

  if (tid == 0) mbar_init(&xbar, 1);
  for (int i = tid; i < a.E * a.TW; i += kFusedBlock) s.mask[i] = 0u;
  pdl_wait();  // logits and x may come from the kernel before this one
  pdl_launch_dependents();
  __syncthreads();
  if (tid == 0 && P > 0) {
    mbar_expect_tx(&xbar, static_cast<uint32_t>(P * row_bytes));
    const char* src = static_cast<const char*>(a.x) + static_cast<int64_t>(tail0) * row_bytes;
    for (int r = 0; r < P; ++r)
      bulk_g2s(s.xpre + r * row_bytes, src + r * row_bytes, static_cast<uint32_t>(row_bytes), &xbar);
  }
  bool pre_ready = P == 0;
  auto wait_pre = [&]() {
    if (!pre_ready) {
      if (!mbar_wait(&xbar, 0, kCopyPolls)) raise_status(a.status, kStatusTimeout);
      pre_ready = true;
    }
  };

  // ---- A: route the tile and count it ---------------------------------------
  route_tile<VPL, VEC4>(a.logits, t0, nt, a.E, a.k, a.lanes_log2, a.renorm, a.TW, s.mask, a.topk_idx, a.topk_w,
                        s.ids);
  __syncthreads();
  tile_word_prefix_row(s.mask, s.pre, a.E, a.TW, a.counts + static_cast<int64_t>(b) * a.E);

  unsigned round = 0u;
  const unsigned expected = static_cast<unsigned>(G + a.extra_arrivals);
  bool ok = count_barrier(a.bar, expected, a.barrier_polls, &round);

  if (ok) {
    // ---- B: this tile's first position within each expert, the offsets ------
    for (int e = tid; e < a.E; e += kFusedBlock) {
      s.base[e] = 0;
      s.kept[e] = 0;
    }
    __syncthreads();
    if (a.small_layout) {
      // every pair of the batch: e's total, and e's pairs in tokens before this tile
      const int np = a.T * a.k;
      const int before = static_cast<int>(t0) * a.k;
      for (int p = tid; p < np; p += kFusedBlock) {
        const int e = __ldcg(a.topk_idx + p);
        atomicAdd(&s.kept[e], 1);
        if (p < before) atomicAdd(&s.base[e], 1);
      }
    } else {
      tile_bases(a.counts, G, a.E, b, s.base, s.kept);
    }
    __syncthreads();
    // capacity clip and the expert offsets: thread e < E of the first 8 warps
    // holds expert e (E <= 256); warp sums meet in shared memory
    {
      const bool on = tid < a.E;
      int raw = 0, kept = 0, incl = 0;
      if (warp < 8) {
        raw = on ? s.kept[tid] : 0;
        kept = min(raw, a.cap);
        incl = warp_inclusive_scan(kept);
        const unsigned drop = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(raw - kept));
        if (lane == 31) {
          scan_s[warp] = incl;
          scan_s[8 + warp] = static_cast<int>(drop);
        }
      }
      __syncthreads();
      if (on) {  // tid < E <= 256: warps 0..7
        int before = 0, total = 0, drop_tot = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const int v = scan_s[w];
          total += v;
          if (w < warp) before += v;
          drop_tot += scan_s[8 + w];
        }
        const int off = before + incl - kept;
        s.kept[tid] = off;  // from here on: the expert's offset
        if (b == 0) {
          const int Gr = a.E / a.R;  // rank r starts at its first expert r*Gr
          a.expert_counts[tid] = kept;
          if (a.expert_raw) a.expert_raw[tid] = raw;
          a.expert_off[tid] = off;
          if (tid % Gr == 0) a.rank_off[tid / Gr] = off;
          if (tid == a.E - 1) {
            a.expert_off[a.E] = total;
            a.rank_off[a.R] = total;
            *a.n_dropped = drop_tot;
          }
        }
      }
    }
    __syncthreads();
    // the rows of this tile's pairs: slot_row / row_slot
    for (int p = tid; p < nt * a.k; p += kFusedBlock) {
      const int tl = p / a.k;
      fused_row(a, s, t0 + tl, tl, p - tl * a.k);
    }
    // this tile's rows are written: arrive at the second grid barrier (its
    // wait comes when the own part is done)
    __syncthreads();
    if (tid == 0) split_arrive(a.bar, expected, a.work);  // in own-tile mode too: the last arrival resets the words
  }
  if (!ok) {
    if (tid == 0) {
      raise_status(a.status, kStatusTimeout);
      if (P > 0) mbar_wait(&xbar, 0, kCopyPolls);  // no bulk copy may still target this CTA at exit
    }
    return;
  }

  // ---- C: scatter -------------------------------------------------------------------
  // The groups (or warps) of the CTA take tokens t0 + g, t0 + g + n, ... of
  // its own tile's first part, then the rest of every tile from the shared
  // counter once the second barrier has completed (TokenPlan). Own-tile mode:
  // the whole tile is the first part (x preloaded in shared memory) and
  // nothing is shared.
  const uint64_t pol = l2_evict_first_policy();  // x and payload lines: first out of L2
  auto x_src = [&](int t) -> const char* {  // a token's x row: shared memory for the preloaded tail
    if (t >= tail0 && t < tail0 + P) return reinterpret_cast<const char*>(s.xpre) + (t - tail0) * row_bytes;
    return nullptr;
  };

  if constexpr (FMT == kFmtBf16) {
    // a warp per token: lanes j < k hold slot j's row, a ballot keeps the
    // slots not dropped, each 16-byte chunk of x is read once (none when every
    // slot was dropped) and stored to every kept row, in groups of 8 rows
    constexpr int U = 8;
    char* const pbase = static_cast<char*>(a.payload);
    const int nchunk = a.H >> 3;
    const int end = a.T;
    // the token sequence of this warp (lane 0): its share of the own part,
    // then the shared part (own-tile mode: the whole tile is the own part)
    const TokenPlan tp{a.work, a.bar.round, a.status, round, a.T, a.tile, own, static_cast<int>(t0),
                       static_cast<int>(t0) + min(nt, own)};
    int own_next = static_cast<int>(t0) + warp;
    bool shared_ok = false;
    auto issue = [&]() -> int { return lane == 0 ? plan_issue(tp, own_next, kFusedBlock / 32, shared_ok) : 0; };
    auto resolve = [&](int ticket) -> int { return lane == 0 ? plan_resolve(tp, ticket) : 0; };
    auto slot_rows = [&](int tok) {
      return tok < end && lane < a.k ? __ldcg(a.slot_row + static_cast<int64_t>(tok) * a.k + lane) : -1;
    };
    int t = __shfl_sync(0xffffffffu, resolve(issue()), 0);
    int tn = __shfl_sync(0xffffffffu, resolve(issue()), 0);
    int pend = issue();  // the ticket of the token after next: read one token later
    int row = slot_rows(t), row_n = slot_rows(tn);  // this token's and the next token's rows
    while (t < end) {
      const int tnn = __shfl_sync(0xffffffffu, tn < end ? resolve(pend) : end, 0);
      pend = tnn < end ? issue() : 0;
      const int row_nn = slot_rows(tnn);  // in flight for two tokens
      const unsigned kept = __ballot_sync(0xffffffffu, row >= 0);
      if (kept != 0u) {
        const char* sx = x_src(t);
        if (sx) wait_pre();
        const char* xr = sx ? sx : static_cast<const char*>(a.x) + static_cast<int64_t>(t) * row_bytes;
        unsigned msk = kept;
        while (msk) {
          char* p[8];
          int n = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int srcl = msk ? __ffs(msk) - 1 : 0;  // uniform across the warp
            const int r = __shfl_sync(0xffffffffu, row, srcl);
            p[i] = pbase + static_cast<int64_t>(r < 0 ? 0 : r) * row_bytes;
            if (msk) ++n;
            msk &= msk - 1u;
          }
          for (int c0 = lane; c0 < nchunk; c0 += 32 * U) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int c = c0 + 32 * u;
              if (c >= nchunk)
                v[u] = make_uint4(0, 0, 0, 0);
              else if (sx)
                v[u] = *reinterpret_cast<const uint4*>(xr + 16 * c);
              else
                v[u] = ld_stream_v4_hint(xr + 16 * static_cast<int64_t>(c), pol);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int c = c0 + 32 * u;
              if (c >= nchunk) break;
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (i < n) st_v4_hint(p[i] + 16 * static_cast<int64_t>(c), v[u], pol);
            }
          }
        }
      }
      t = tn;
      tn = tnn;
      row = row_n;
      row_n = row_nn;
    }
  } else {
    // a group of gw warps per token (two 16-element groups per thread); the
    // group's named barrier (a warp sync for one-warp groups) orders one
    // exchange per token: the warps' amax of this token and the rows of the
    // next. The next token's row is loaded while this one is coded, and the
    // rows two tokens ahead, so that no exchange waits for a load.
    const int ngrp16 = a.H >> 4;
    const int gw = coded_group_warps(a.H);  // warps per token
    const int ngroups = coded_groups(a.H);
    const int g = warp / gw;
    if (g < ngroups) {
      const int gsz = gw * 32;
      const int c = tid - g * gsz;  // thread within the group
      const int wg = c >> 5;        // warp within the group
      auto gsync = [&]() {
        if (gw == 1)
          __syncwarp();
        else
          group_sync(1 + g, gsz);
      };
      const int end = a.T;
      // the group's token sequence (thread 0): its share of the own part,
      // then the shared part (own-tile mode: the whole tile is the own part)
      const TokenPlan tp{a.work, a.bar.round, a.status, round, a.T, a.tile, own, static_cast<int>(t0),
                         static_cast<int>(t0) + min(nt, own)};
      int own_next = static_cast<int>(t0) + g;
      bool shared_ok = false;
      auto issue = [&]() -> int { return plan_issue(tp, own_next, ngroups, shared_ok); };
      auto resolve = [&](int ticket) -> int { return plan_resolve(tp, ticket); };
      auto load_x = [&](int t, uint4 (&v)[4]) {  // this thread's 32 elements of token t's row
        const char* sx = x_src(t);
        if (sx) wait_pre();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int grp = c + q * gsz;
          if (grp < ngrp16) {
            if (sx) {
              const uint4* pp = reinterpret_cast<const uint4*>(sx + 32 * grp);
              v[2 * q] = pp[0];
              v[2 * q + 1] = pp[1];
            } else {
              ld_x32_global(static_cast<const char*>(a.x) + static_cast<int64_t>(t) * row_bytes + 32 * grp,
                            v[2 * q], v[2 * q + 1]);
            }
          } else {
            v[2 * q] = v[2 * q + 1] = make_uint4(0, 0, 0, 0);
          }
        }
      };
      auto slot_rows = [&](int tok) {
        return tok < end && c < a.k ? __ldcg(a.slot_row + static_cast<int64_t>(tok) * a.k + c) : -1;
      };
      int pend = 0;
      if (c == 0) {
        ids_s[g][0] = resolve(issue());
        ids_s[g][1] = ids_s[g][0] < end ? resolve(issue()) : end;
        pend = ids_s[g][1] < end ? issue() : 0;  // the ticket after next: read at the next exchange
      }
      gsync();
      int t = ids_s[g][0], tn = ids_s[g][1];
      uint4 cur[4];
      if (t < end) load_x(t, cur);
      if (c < a.k) rows_s[g][0][c] = slot_rows(t);
      int r_n = slot_rows(tn);  // the next token's rows, in a register until its turn
      gsync();
      int rb = 0, ab = 0;  // rows buffer of token t (three deep), amax / id buffer (two deep)
      while (t < end) {
        const int rbn = rb == 2 ? 0 : rb + 1;
        uint4 nxt[4];
        if (tn < end) load_x(tn, nxt);  // in flight while this token is coded
        if (c < a.k) rows_s[g][rbn][c] = r_n;
        if (c == 0) {
          const int tnn = tn < end ? resolve(pend) : end;
          ids_s[g][ab] = tnn;
          pend = tnn < end ? issue() : 0;  // read at the next exchange
        }
        float m = fmaxf(absmax_bf16x16(cur[0], cur[1]), absmax_bf16x16(cur[2], cur[3]));
        m = warp_max(m);
        if (lane == 0) amax_s[g][ab][wg] = m;
        gsync();
        const int tnn = ids_s[g][ab];
        const int r_nn = slot_rows(tnn);  // in flight until the next exchange
        float am = amax_s[g][ab][0];
        for (int i = 1; i < gw; ++i) am = fmaxf(am, amax_s[g][ab][i]);
        const float scale = __fdiv_rn(am, CodeMax<FMT>::kValue);
        const float inv = __frcp_rn(scale);
        const int32_t* rows = rows_s[g][rb];
        // both of this thread's groups coded first, then one pass over the
        // kept rows, each row's address formed once
        const int grp0 = c, grp1 = c + gsz;
        const bool has1 = grp1 < ngrp16;
        if (grp0 < ngrp16) {
          if constexpr (FMT == kFmtInt4) {
            const uint2 q0 = quant16_int4_coded(cur[0], cur[1], scale, inv);
            const uint2 q1 = has1 ? quant16_int4_coded(cur[2], cur[3], scale, inv) : make_uint2(0, 0);
            char* const pb = static_cast<char*>(a.payload);
            for (int j = 0; j < a.k; ++j) {
              const int row = rows[j];
              if (row < 0) continue;
              char* dst = pb + static_cast<int64_t>(row) * (a.H / 2);
              st_v2_hint(dst + 8 * grp0, q0, pol);
              if (has1) st_v2_hint(dst + 8 * grp1, q1, pol);
            }
          } else {
            const uint4 q0 = quant16_fmt<FMT>(cur[0], cur[1], scale, inv);
            const uint4 q1 = has1 ? quant16_fmt<FMT>(cur[2], cur[3], scale, inv) : make_uint4(0, 0, 0, 0);
            char* const pb = static_cast<char*>(a.payload);
            for (int j = 0; j < a.k; ++j) {
              const int row = rows[j];
              if (row < 0) continue;
              char* dst = pb + static_cast<int64_t>(row) * a.H;
              st_v4_hint(dst + 16 * grp0, q0, pol);
              if (has1) st_v4_hint(dst + 16 * grp1, q1, pol);
            }
          }
        }
        if (c < a.k && rows[c] >= 0) a.scales[rows[c]] = scale;
#pragma unroll
        for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
        t = tn;
        tn = tnn;
        r_n = r_nn;
        rb = rbn;
        ab ^= 1;
      }
    }
  }
  // a CTA whose preloaded rows were never read (every slot of those tokens
  // dropped) still waits for their copies before it exits
  if (tid == 0 && !pre_ready) mbar_wait(&xbar, 0, kCopyPolls);
}

}  // namespace

namespace {

// Per device and kernel instance: the dynamic shared memory a CTA may use
// (the opt-in maximum less the kernel's static shared memory), or -1 when the
// kernel cannot run there (no cooperative launch, or not one CTA per SM).
// Asks for the smallest shared-memory share of the SM's L1 / shared storage
// that holds `bytes` (the rest stays L1); remembered per device in `last`.
// The split outlives the kernel: the combine that follows (no shared memory,
// many loads in flight, whose data all passes through L1) runs in it, and
// with the largest shared share it ran 15-20 % slower.
template <class K>
void fused_carveout(K kernel, size_t bytes, int* last) {
  int dev = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return;
  if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess || per_sm <= 0)
    return;
  int pct = static_cast<int>((bytes * 100 + per_sm - 1) / static_cast<size_t>(per_sm));
  pct = pct < 1 ? 1 : (pct > 100 ? 100 : pct);
  if (cache_load(&last[dev]) == pct) return;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, pct) == cudaSuccess)
    cache_store(&last[dev], pct);
  else
    (void)cudaGetLastError();  // a preference only
}

template <class K>
int fused_prepare(K kernel, int* cache) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  if (dev < 64) {
    const int c = cache_load(&cache[dev]);
    if (c != 0) return c;
  }
  int v = -1;
  int coop = 0, optin = 0;
  cudaFuncAttributes fa;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
      cudaFuncGetAttributes(&fa, kernel) == cudaSuccess) {
    const int dyn = optin - static_cast<int>(fa.sharedSizeBytes);
    int nb = 0;
    if (dyn > 0 && cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, kFusedBlock, dyn) == cudaSuccess && nb >= 1)
      v = dyn;
  }
  if (v < 0) (void)cudaGetLastError();  // a refused query is not an error of this call
  if (dev < 64) cache_store(&cache[dev], v);
  return v;
}

template <int VPL, bool VEC4, int FMT>
cudaError_t launch_fused_t(FusedArgs fa, int G, cudaStream_t s, bool dry) {
  auto kernel = route_dispatch_fused_kernel<VPL, VEC4, FMT>;
  static int prep[64], carve[64], static_smem[64];
  const int dyn = fused_prepare(kernel, prep);
  const size_t fixed = fused_smem_fixed(fa.E, fa.TW, fa.k);
  if (dyn < 0 || static_cast<size_t>(dyn) < fixed) return cudaErrorNotSupported;
  if (dry) return cudaSuccess;
  // the static tail: as many x rows per CTA as shared memory holds, at most
  // floor(T / G) so that every CTA has as many; when the tail is each CTA's
  // own tile, no CTA waits at the second grid barrier
  const int64_t row_bytes = 2 * static_cast<int64_t>(fa.H);
  const int64_t room = static_cast<int64_t>(dyn) - static_cast<int64_t>(fixed);
  const bool small = static_cast<int64_t>(fa.tile) * row_bytes <= (room < kPreloadBytes ? room : kPreloadBytes);
  const int64_t even = fa.T / G;
  fa.npre = small ? static_cast<int>(fa.tile < even ? fa.tile : even) : 0;
  fa.own_tile = (fa.npre == fa.tile && static_cast<int64_t>(G) * fa.npre == fa.T) ? 1 : 0;
  // few pairs: every CTA counts the routed ids themselves rather than every tile's counts
  fa.small_layout = static_cast<int64_t>(fa.T) * fa.k <= kSmallLayoutPairs ? 1 : 0;
  const size_t smem = static_cast<size_t>(fa.npre) * row_bytes + fixed;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
      int st = cache_load(&static_smem[dev]);
      if (st == 0) {
        cudaFuncAttributes attr;
        st = cudaFuncGetAttributes(&attr, kernel) == cudaSuccess ? static_cast<int>(attr.sharedSizeBytes) + 1 : -1;
        cache_store(&static_smem[dev], st);
      }
      if (st > 0) fused_carveout(kernel, smem + static_cast<size_t>(st - 1) + 1024, carve);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(G));
  cfg.blockDim = dim3(kFusedBlock);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident at once: the grid barrier cannot wait on a CTA
  attr[0].val.cooperative = 1;                  // that has not started
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, fa);
}

template <int VPL, bool VEC4>
cudaError_t launch_fused_fmt(const FusedArgs& fa, int fmt, int G, cudaStream_t s, bool dry) {
  switch (fmt) {
    case kFmtBf16: return launch_fused_t<VPL, VEC4, kFmtBf16>(fa, G, s, dry);
    case kFmtInt8: return launch_fused_t<VPL, VEC4, kFmtInt8>(fa, G, s, dry);
    case kFmtFp8: return launch_fused_t<VPL, VEC4, kFmtFp8>(fa, G, s, dry);
    case kFmtInt4: return launch_fused_t<VPL, VEC4, kFmtInt4>(fa, G, s, dry);
    default: return cudaErrorNotSupported;
  }
}

int g_force_wait_timeout = 0;  // set by ep_debug_force_wait_timeout (tests only)

}  // namespace

void set_force_wait_timeout(int enable) { cache_store(&g_force_wait_timeout, enable ? 1 : 0); }

cudaError_t launch_route_dispatch_fused(const RouteCountArgs& r, const DispatchArgs& a, int sms, cudaStream_t s,
                                        bool dry) {
  if (r.T <= 0 || r.E > kFusedMaxExperts || sms < 1) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(a.x) & 31u) != 0) return cudaErrorNotSupported;  // 32-byte row loads
  const int G0 = sms < kFusedMaxCTAs ? sms : kFusedMaxCTAs;
  const int tile = (r.T + G0 - 1) / G0;
  if (tile > 1024) return cudaErrorNotSupported;  // at most 32 mask words per expert
  const int G = (r.T + tile - 1) / tile;          // no empty CTA
  int TW = 1;
  while (TW * 32 < tile) TW <<= 1;
  int lanes_log2 = 0;
  while ((1 << lanes_log2) < r.E && lanes_log2 < 5) ++lanes_log2;
  const int L = 1 << lanes_log2;
  const int vpl = (r.E + L - 1) / L;  // <= 8 for E <= 256
  const bool vec4 = (L == 32) && (r.E % 128 == 0);

  FusedArgs fa;
  fa.logits = r.logits;
  fa.x = a.x;
  fa.T = r.T;
  fa.H = a.H;
  fa.E = r.E;
  fa.k = r.k;
  fa.R = a.R;
  fa.cap = a.cap;
  fa.renorm = r.renorm;
  fa.lanes_log2 = lanes_log2;
  fa.tile = tile;
  fa.TW = TW;
  fa.npre = 0;
  fa.own_tile = 0;
  fa.small_layout = 0;
  fa.topk_idx = r.topk_idx;
  fa.topk_w = r.topk_w;
  fa.payload = a.payload;
  fa.scales = a.scales;
  fa.row_slot = a.row_slot;
  fa.slot_row = a.slot_row;
  fa.expert_counts = a.expert_counts;
  fa.expert_raw = a.expert_raw;
  fa.expert_off = a.expert_off;
  fa.rank_off = a.rank_off;
  fa.n_dropped = a.n_dropped;
  fa.counts = a.tile_counts;
  fa.status = a.status;
  fa.bar.count = a.bar_count;
  fa.bar.round = a.bar_round;
  fa.work = a.work;
  const bool force = cache_load(&g_force_wait_timeout) != 0;
  fa.extra_arrivals = force ? 1 : 0;
  fa.barrier_polls = force ? (1ll << 14) : kBarrierPolls;

  if (vec4)
    return vpl == 4 ? launch_fused_fmt<4, true>(fa, a.fmt, G, s, dry) : launch_fused_fmt<8, true>(fa, a.fmt, G, s, dry);
  if (vpl <= 1) return launch_fused_fmt<1, false>(fa, a.fmt, G, s, dry);
  if (vpl <= 2) return launch_fused_fmt<2, false>(fa, a.fmt, G, s, dry);
  if (vpl <= 4) return launch_fused_fmt<4, false>(fa, a.fmt, G, s, dry);
  return launch_fused_fmt<8, false>(fa, a.fmt, G, s, dry);
}

}  // namespace ep
