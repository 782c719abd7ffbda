// dispatch.cu — rank-major send layout: histogram, device-wide scan, row
// assignment, and a stable scatter fused with the per-token int8 code.
//
// The layout is the one the pages describe: every copy headed for one
// destination sits in one contiguous block ("aggregate by target card",
// ThunderEP on consumer GPUs, bjdmk.com.cn, §2.1), blocks in rank order at
// running sums of the counts (NCCL EP article, hotelren.com, §3.3), and the
// payload may be the token's per-token int8 code (ThunderEP §2.3).
//
// Three launches, so that every destination row is decided before any
// payload byte moves and the scatter is a pure read-once / write-k stream:
//   count    one CTA per tile of `tile` tokens: per-expert bit masks of the
//            tile's tokens in shared memory (atomicOr, order-free); their
//            popcounts give the tile's per-expert count and each pair's rank
//            within the tile in token order;
//   scan     one warp per expert: the exclusive running sum over tiles (each
//            tile's first position within the expert) and the capacity clip;
//            the last CTA to finish (atomic ticket after a fence — no CTA
//            ever waits for another) sums the kept counts over experts into
//            expert_off / rank_off;
//   scatter  a grid-stride loop over tokens. Threads j < k turn the token's
//            pairs into rows (row = expert_off[e] + tile base + rank in
//            tile, or -1 past the cap) and write slot_row / row_slot, two
//            tokens ahead. int8: one CTA per token, 32 elements per thread,
//            the next token's row loaded while this one is coded (exact amax,
//            IEEE scale, exact int8 code), one 16-byte store per kept row and
//            group. bf16: one warp per token, each 16-byte chunk of x loaded
//            once and stored to every kept row.
#include "ep_internal.h"
#include "pairs.cuh"

namespace ep {
namespace {

template <class Pairs>
__global__ void __launch_bounds__(512) count_kernel(const Pairs src, int T, int E, int k, int tile, int ntiles,
                                                    int32_t* __restrict__ tile_counts,
                                                    int32_t* __restrict__ lrank, uint32_t* status,
                                                    uint32_t* ticket) {
  extern __shared__ uint32_t smem[];
  pdl_wait();  // the expert ids come from the kernel before this one
  pdl_launch_dependents();
  if (blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0u;  // the scan that follows counts its CTAs from 0
  const int TW = tile >> 5;
  uint32_t* mask = smem;         // [E][TW] bit b of word w: token 32*w+b of the tile chose e
  uint32_t* pre = smem + E * TW;  // [E][TW] set bits of e in the words before w
  const int b = blockIdx.x;
  const int64_t t0 = static_cast<int64_t>(b) * tile;
  const int nt = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(tile), T - t0)));
  for (int i = threadIdx.x; i < E * TW; i += blockDim.x) mask[i] = 0u;
  __syncthreads();

  const int64_t base = t0 * k;
  const int npairs = nt * k;
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    const int tl = p / k;
    const int e = src.expert(t0 + tl, p - tl * k);
    if (p - tl * k == 0 && !src.count_ok(t0 + tl)) raise_status(status, kStatusBadIndex);
    if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
      raise_status(status, kStatusBadIndex);
      continue;
    }
    const uint32_t bit = 1u << (tl & 31);
    const uint32_t old = atomicOr(&mask[e * TW + (tl >> 5)], bit);
    if (old & bit) raise_status(status, kStatusBadIndex);  // expert repeated within one token
  }
  __syncthreads();
  if (nt == 0) return;

  tile_word_prefix(mask, pre, E, TW, tile_counts, ntiles, b);
  __syncthreads();

  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    const int tl0 = p / k;
    const int e = src.expert(t0 + tl0, p - tl0 * k);
    int r = -1;
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
      const int tl = tl0;
      const int w = tl >> 5;
      r = static_cast<int>(pre[e * TW + w]) + __popc(mask[e * TW + w] & ((1u << (tl & 31)) - 1u));
    }
    lrank[base + p] = r;
  }
}

// One warp per expert (eight per CTA): the exclusive running sum of the
// expert's tile counts (each tile's first position within the expert, eight
// tiles per lane per pass) and the capacity clip; the last CTA to finish
// (atomic ticket after a fence — no CTA ever waits for another) sums the kept
// counts over experts into expert_off / rank_off.
constexpr int kScanWarps = 8;

__global__ void __launch_bounds__(32 * kScanWarps) scan_kernel(
    const int32_t* __restrict__ tile_counts, int E, int R, int ntiles, int cap, int32_t* __restrict__ tile_base,
    int32_t* __restrict__ expert_counts, int32_t* __restrict__ expert_raw, int32_t* __restrict__ expert_off,
    int32_t* __restrict__ rank_off, int32_t* __restrict__ n_dropped, int32_t* kept_g, int32_t* drop_g,
    uint32_t* ticket) {
  constexpr int V = 8;
  __shared__ int warp_s[8];
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kScanWarps + warp;
  pdl_wait();  // tile counts come from the counting kernel
  pdl_launch_dependents();
  if (e < E) {
    const int32_t* tc = tile_counts + static_cast<int64_t>(e) * ntiles;
    int32_t* tb = tile_base + static_cast<int64_t>(e) * ntiles;
    int carry = 0;
    for (int c0 = 0; c0 < ntiles; c0 += 32 * V) {
      int v[V];
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const int i = c0 + lane * V + j;
        v[j] = i < ntiles ? tc[i] : 0;
      }
      int run = 0;
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const int x = v[j];
        v[j] = run;
        run += x;
      }
      const int incl = warp_inclusive_scan(run);
      const int base = carry + incl - run;
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const int i = c0 + lane * V + j;
        if (i < ntiles) tb[i] = base + v[j];
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      const int kept = min(carry, cap);
      expert_counts[e] = kept;
      if (expert_raw) expert_raw[e] = carry;
      kept_g[e] = kept;
      drop_g[e] = carry - kept;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(ticket, 1u);
    is_last = (prev == static_cast<unsigned>(gridDim.x) - 1u);
  }
  __syncthreads();
  if (!is_last) return;

  // last CTA: every other CTA's kept/drop values are visible (fence + ticket)
  __threadfence();
  int carry_off = 0, drops = 0;
  const int G = E / R;  // rank r starts at its first expert r*G
  for (int c0 = 0; c0 < E; c0 += blockDim.x) {
    const int i = c0 + threadIdx.x;
    const int v = i < E ? __ldcg(kept_g + i) : 0;
    const int d = i < E ? __ldcg(drop_g + i) : 0;
    int tot, dtot;
    const int ex = block_exclusive_scan(v, tot, warp_s);
    block_exclusive_scan(d, dtot, warp_s);
    if (i < E) expert_off[i] = carry_off + ex;
    if (i < E && i % G == 0) rank_off[i / G] = carry_off + ex;
    carry_off += tot;
    drops += dtot;
  }
  if (threadIdx.x == 0) {
    expert_off[E] = carry_off;
    rank_off[R] = carry_off;
    *n_dropped = drops;
  }
}

// Destination row of pair p = t*k + j, formed in three steps that the
// scatter spreads over three tokens so that no step waits on the load issued
// by the step before it within one token's time:
//   A  load the pair's expert e and rank within its tile (from count);
//   B  load the tile's first position within e and e's offset (from scan);
//   C  row = offset + position if position < cap, else -1 (dropped); write
//      slot_row and row_slot.
// A bad expert id (already reported by count) gives row -1.
struct PairA {
  int e, lr;
};
struct PairB {
  int pos, off;  // pos < 0: no row
};

__device__ __forceinline__ PairA pair_load_a(const DispatchArgs& a, int64_t t, int j) {
  PairA r{-1, -1};
  if (t < a.T) {
    const int64_t p = t * a.k + j;
    r.e = a.topk_idx[p];
    r.lr = a.lrank[p];
  }
  return r;
}

__device__ __forceinline__ PairB pair_load_b(const DispatchArgs& a, int64_t t, PairA x, int tile_log2) {
  PairB r{-1, 0};
  if (t < a.T && static_cast<unsigned>(x.e) < static_cast<unsigned>(a.E) && x.lr >= 0) {
    r.pos = a.tile_base[static_cast<int64_t>(x.e) * a.ntiles + (t >> tile_log2)] + x.lr;
    r.off = a.expert_off[x.e];
  }
  return r;
}

__device__ __forceinline__ int pair_finish(const DispatchArgs& a, int64_t t, int j, PairB x) {
  if (t >= a.T) return -1;
  const int64_t p = t * a.k + j;
  const int row = (x.pos >= 0 && x.pos < a.cap) ? x.off + x.pos : -1;
  a.slot_row[p] = row;
  if (row >= 0) a.row_slot[row] = static_cast<int32_t>(p);
  return row;
}

constexpr unsigned kFull = 0xffffffffu;

// Gathers the next (up to) 8 kept slots of `mask` (lowest slot first) from
// the lanes that hold them: their payload row addresses, in every lane.
__device__ __forceinline__ int gather_rows(unsigned& mask, int row, char* base, int64_t row_bytes, char* (&p)[8]) {
  int n = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int src = mask ? __ffs(mask) - 1 : 0;  // uniform across the warp
    const int r = __shfl_sync(kFull, row, src);
    p[i] = base + static_cast<int64_t>(r < 0 ? 0 : r) * row_bytes;
    if (mask) ++n;
    mask &= mask - 1u;
  }
  return n;
}

// 32 bytes (16 bf16) of x per thread: one 32-byte load when the row base is
// 32-byte aligned (V8), else two 16-byte loads; either way the lines read
// become the first to leave L2 (pol: an evict-first policy).
template <bool V8>
__device__ __forceinline__ void ld_x32(const char* p, uint4& lo, uint4& hi, uint64_t pol) {
  if constexpr (V8) {
    asm volatile("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
                 : "l"(p));
  } else {
    lo = ld_stream_v4_hint(p, pol);
    hi = ld_stream_v4_hint(p + 16, pol);
  }
}

// int8, FP8 or int4 payload: one CTA per token in flight (grid-stride). Thread c codes the
// 16-element groups c and c + blockDim.x of the row, so that every warp-wide
// store covers whole 32-byte sectors. The next token's row is loaded while
// this one is coded; threads j < k carry slot j's row (rows pipeline above,
// two tokens ahead). amax: exact per-thread halfword maxima, a warp max and one
// shared-memory step; scale = amax/127 (int8), amax/448 (FP8) or amax/7
// (int4) with IEEE division; the code is the branch-free corrected-quotient
// path; an int4 group is 8 bytes of packed nibbles.
template <bool V8, int FMT>
__global__ void __launch_bounds__(512) scatter_code_kernel(const DispatchArgs a, int tile_log2) {
  constexpr int G = 2;  // 16-element groups per thread
  __shared__ int32_t rows_s[2][32];
  __shared__ float amax_s[2][16];
  const int c = threadIdx.x;
  const int B = blockDim.x;
  const int ngroup = a.H >> 4;
  const bool slot = c < a.k;
  const int warp = c >> 5, lane = c & 31, nw = B >> 5;
  const char* xb = static_cast<const char*>(a.x);
  const int64_t GS = gridDim.x;
  const uint64_t pol = l2_evict_first_policy();  // x and payload lines: first out of L2
  auto ld_tok = [&](int64_t t, uint4 (&v)[2 * G]) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int grp = c + g * B;
      if (t < a.T && grp < ngroup)
        ld_x32<V8>(xb + (t * a.H + 16 * grp) * 2, v[2 * g], v[2 * g + 1], pol);
      else
        v[2 * g] = v[2 * g + 1] = make_uint4(0, 0, 0, 0);
    }
  };
  int64_t t = blockIdx.x;
  // Before the wait: x and the pair data of the count kernel (two launches
  // back, unless pairs_early is 0) only; tile bases and offsets come from the
  // scan just before.
  uint4 cur[2 * G];
  ld_tok(t, cur);
  PairA a0{-1, -1}, a1{-1, -1}, a_next2{-1, -1};
  if (!a.pairs_early) pdl_wait();
  if (slot) {
    a0 = pair_load_a(a, t, c);
    a1 = pair_load_a(a, t + GS, c);
    a_next2 = pair_load_a(a, t + 2 * GS, c);
  }
  pdl_wait();
  pdl_launch_dependents();
  int my_row = -1;
  PairB b_next{-1, 0};
  if (slot) {
    my_row = pair_finish(a, t, c, pair_load_b(a, t, a0, tile_log2));
    b_next = pair_load_b(a, t + GS, a1, tile_log2);
  }
  int buf = 0;
  for (; t < a.T; t += GS) {
    const int64_t tn = t + GS;
    uint4 nxt[2 * G];
    ld_tok(tn, nxt);
    int next_row = -1;
    if (slot) {
      rows_s[buf][c] = my_row;
      next_row = pair_finish(a, tn, c, b_next);
      b_next = pair_load_b(a, tn + GS, a_next2, tile_log2);
      a_next2 = pair_load_a(a, tn + 2 * GS, c);
    }
    float m = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) m = fmaxf(m, absmax_bf16x16(cur[2 * g], cur[2 * g + 1]));
    m = warp_max(m);
    if (lane == 0) amax_s[buf][warp] = m;
    __syncthreads();
    float am = amax_s[buf][0];
    for (int i = 1; i < nw; ++i) am = fmaxf(am, amax_s[buf][i]);
    const float scale = __fdiv_rn(am, CodeMax<FMT>::kValue);
    const float inv = __frcp_rn(scale);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int grp = c + g * B;
      if (grp >= ngroup) break;
      if constexpr (FMT == kFmtInt4) {  // 8 bytes of packed nibbles per group, rows of H/2 bytes
        const uint2 q = quant16_int4_coded(cur[2 * g], cur[2 * g + 1], scale, inv);
        for (int j = 0; j < a.k; ++j) {
          const int row = rows_s[buf][j];
          if (row >= 0) st_v2_hint(static_cast<char*>(a.payload) + static_cast<int64_t>(row) * (a.H / 2) + 8 * grp, q, pol);
        }
      } else {
        const uint4 q = quant16_fmt<FMT>(cur[2 * g], cur[2 * g + 1], scale, inv);
        for (int j = 0; j < a.k; ++j) {
          const int row = rows_s[buf][j];
          if (row >= 0) st_v4_hint(static_cast<int8_t*>(a.payload) + static_cast<int64_t>(row) * a.H + 16 * grp, q, pol);
        }
      }
    }
    if (slot && my_row >= 0) a.scales[my_row] = scale;
#pragma unroll
    for (int i = 0; i < 2 * G; ++i) cur[i] = nxt[i];
    my_row = next_row;
    buf ^= 1;
  }
}

// bf16 payload: one warp per token in flight; no block-level synchronisation.
// Lanes j < k carry slot j's row (rows pipeline over this warp's tokens t,
// t+W, t+2W); a ballot keeps the slots that were not dropped and their row
// addresses are gathered into every lane, so a token with no kept slot costs
// nothing; each 16-byte chunk of x is loaded once (8 chunks per lane in
// flight) and stored to every kept row.
__global__ void __launch_bounds__(256) scatter_bf16_kernel(const DispatchArgs a, int tile_log2) {
  constexpr int U = 8;  // 16-byte chunks per lane per pass
  const int lane = threadIdx.x & 31;
  const int64_t W = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const bool slot = lane < a.k;
  const int64_t row_bytes = 2 * static_cast<int64_t>(a.H);
  const int nchunk = a.H >> 3;  // 16-byte chunks (8 elements)
  char* const pbase = static_cast<char*>(a.payload);
  const uint64_t pol = l2_evict_first_policy();  // x and payload lines: first out of L2

  PairA a0{-1, -1}, a1{-1, -1}, a_next2{-1, -1};
  if (!a.pairs_early) pdl_wait();
  if (slot) {  // before the wait: pair data of the count kernel, two launches back
    a0 = pair_load_a(a, w0, lane);
    a1 = pair_load_a(a, w0 + W, lane);
    a_next2 = pair_load_a(a, w0 + 2 * W, lane);
  }
  pdl_wait();  // tile bases and offsets come from the scan just before
  pdl_launch_dependents();
  int my_row = -1;
  PairB b_next{-1, 0};
  if (slot) {
    my_row = pair_finish(a, w0, lane, pair_load_b(a, w0, a0, tile_log2));
    b_next = pair_load_b(a, w0 + W, a1, tile_log2);
  }
  for (int64_t t = w0; t < a.T; t += W) {
    const int row = my_row;
    if (slot) {
      my_row = pair_finish(a, t + W, lane, b_next);
      b_next = pair_load_b(a, t + 2 * W, a_next2, tile_log2);
      a_next2 = pair_load_a(a, t + 3 * W, lane);
    }
    const unsigned kept = __ballot_sync(kFull, row >= 0);
    if (kept == 0u) continue;  // every copy of this token was dropped
    const int nk = __popc(kept);
    const char* xr = static_cast<const char*>(a.x) + t * row_bytes;
    char* p[8];
    if (nk <= 8) {
      unsigned msk = kept;
      gather_rows(msk, row, pbase, row_bytes, p);
      for (int c0 = lane; c0 < nchunk; c0 += 32 * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = c0 + 32 * u;
          v[u] = c < nchunk ? ld_stream_v4_hint(xr + 16 * static_cast<int64_t>(c), pol) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = c0 + 32 * u;
          if (c >= nchunk) break;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i < nk) st_v4_hint(p[i] + 16 * static_cast<int64_t>(c), v[u], pol);
        }
      }
    } else {
      // more than 8 kept slots (k > 8): groups of 8 per chunk; the loop bound
      // is warp-uniform because the gathers shuffle across all lanes
      for (int c0 = 0; c0 < nchunk; c0 += 32) {
        const int c = c0 + lane;
        const uint4 v = c < nchunk ? ld_stream_v4_hint(xr + 16 * static_cast<int64_t>(c), pol) : make_uint4(0, 0, 0, 0);
        unsigned msk = kept;
        while (msk) {
          const int n = gather_rows(msk, row, pbase, row_bytes, p);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i < n && c < nchunk) st_v4_hint(p[i] + 16 * static_cast<int64_t>(c), v, pol);
        }
      }
    }
  }
}

int count_smem_bytes(int E, int tile) { return 2 * E * (tile / 32) * static_cast<int>(sizeof(uint32_t)); }

}  // namespace

// The counting kernel for one pair source; it also clears the scan's ticket,
// so it runs (one CTA) even for an empty batch.
template <class Pairs>
cudaError_t launch_count(const DispatchArgs& a, const Pairs& src, cudaStream_t s) {
  static int smem_set[64];  // per device: largest dynamic shared size already allowed
  const int smem = count_smem_bytes(a.E, a.tile);
  if (smem > 48 * 1024) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 64 || cache_load(&smem_set[dev]) < smem) {
      err = cudaFuncSetAttribute(count_kernel<Pairs>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (err != cudaSuccess) return err;
      if (dev < 64) cache_store(&smem_set[dev], smem);
    }
  }
  int cblock = ((a.tile * a.k + 31) / 32) * 32;
  cblock = cblock < 64 ? 64 : (cblock > 512 ? 512 : cblock);
  return launch_pdl(count_kernel<Pairs>, a.ntiles > 0 ? a.ntiles : 1, cblock, static_cast<size_t>(smem), s, src, a.T,
                    a.E, a.k, a.tile, a.ntiles, a.tile_counts, a.lrank, a.status, a.ticket);
}

cudaError_t launch_scan(const DispatchArgs& a, cudaStream_t s) {
  return launch_pdl(scan_kernel, (a.E + kScanWarps - 1) / kScanWarps, 32 * kScanWarps, 0, s, a.tile_counts, a.E,
                    a.R, a.ntiles, a.cap, a.tile_base, a.expert_counts, a.expert_raw, a.expert_off, a.rank_off,
                    a.n_dropped, a.kept, a.dropped, a.ticket);
}

cudaError_t launch_dispatch(const DispatchArgs& a, int sms, cudaStream_t s) {
  const cudaError_t err = launch_count(a, IdxPairs{a.topk_idx, a.k}, s);
  if (err != cudaSuccess) return err;
  return launch_scan_scatter(a, sms, s);
}

cudaError_t launch_layout_from_bitmap(const DispatchArgs& a, const uint32_t* bitmap, int words, cudaStream_t s) {
  const cudaError_t err = launch_count(a, BitmapPairs{bitmap, words, a.k}, s);
  if (err != cudaSuccess) return err;
  return launch_scan(a, s);
}

cudaError_t launch_scan_scatter(const DispatchArgs& a, int sms, cudaStream_t s) {
  const cudaError_t err = launch_scan(a, s);
  if (err != cudaSuccess) return err;
  return launch_scatter(a, sms, s);
}

cudaError_t launch_scatter(const DispatchArgs& a, int sms, cudaStream_t s) {
  cudaError_t err = cudaSuccess;
  if (a.T == 0) return cudaSuccess;

  const int tile_log2 = __builtin_ctz(static_cast<unsigned>(a.tile));
  if (a.fmt != kFmtBf16) {
    // two 16-element groups per thread: ceil(H/32) threads per token, rounded
    // up to whole warps (>= 32 >= k)
    const int block = (((a.H / 16 + 1) / 2 + 31) / 32) * 32;
    const bool v8 = (reinterpret_cast<uintptr_t>(a.x) & 31u) == 0;  // rows are then 32-byte aligned too
    static int occ[6][16][64];  // per load width x format, block size / 32, device
    auto go = [&](auto kernel, int which) {
      const int per_sm = resident_ctas(kernel, block, 0, occ[which][block / 32 - 1]);
      const int64_t want = static_cast<int64_t>(sms) * per_sm;
      const int grid = static_cast<int>(a.T < want ? a.T : want);
      return launch_pdl(kernel, grid, block, 0, s, a, tile_log2);
    };
    if (a.fmt == kFmtInt4)
      err = v8 ? go(scatter_code_kernel<true, kFmtInt4>, 5) : go(scatter_code_kernel<false, kFmtInt4>, 4);
    else if (a.fmt == kFmtFp8)
      err = v8 ? go(scatter_code_kernel<true, kFmtFp8>, 3) : go(scatter_code_kernel<false, kFmtFp8>, 2);
    else
      err = v8 ? go(scatter_code_kernel<true, kFmtInt8>, 1) : go(scatter_code_kernel<false, kFmtInt8>, 0);
  } else {
    constexpr int kBlock = 256;
    static int occ[64];
    const int per_sm = resident_ctas(scatter_bf16_kernel, kBlock, 0, occ);
    const int64_t want = static_cast<int64_t>(sms) * per_sm;
    const int64_t need = (static_cast<int64_t>(a.T) + kBlock / 32 - 1) / (kBlock / 32);
    const int grid = static_cast<int>(need < want ? need : want);
    err = launch_pdl(scatter_bf16_kernel, grid, kBlock, 0, s, a, tile_log2);
  }
  return err;
}

}  // namespace ep
