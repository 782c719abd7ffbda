// dispatch.cu — rank-major send layout: histogram, device-wide scan, row
// assignment, and a stable scatter fused with the per-token int8 code.
//
// The layout is the one the pages describe: every copy headed for one
// destination sits in one contiguous block ("aggregate by target card",
// ThunderEP on consumer GPUs, bjdmk.com.cn, §2.1), blocks in rank order at
// running sums of the counts (NCCL EP article, hotelren.com, §3.3), and the
// payload may be the token's per-token int8 code (ThunderEP §2.3).
//
// Four launches, so that every destination row is decided before any
// payload byte moves and the scatter is a pure read-once / write-k stream:
//   count    one CTA per tile of `tile` tokens: per-expert bit masks of the
//            tile's tokens in shared memory (atomicOr, order-free); their
//            popcounts give the tile's per-expert count and each pair's rank
//            within the tile in token order;
//   scan     one CTA per expert: the exclusive running sum over tiles (each
//            tile's first position within the expert) and the capacity clip;
//            the last CTA to finish (atomic ticket after a fence — no CTA
//            ever waits for another) sums the kept counts over experts into
//            expert_off / rank_off;
//   rows     one thread per (token, slot): row = expert_off[e] + position,
//            or -1 past the cap; writes slot_row and row_slot;
//   scatter  a grid-stride loop over tokens, one CTA per token row in
//            flight: 16 elements per thread, 16-byte loads of x and of the
//            next token's slot_row prefetched during this token, amax by warp
//            shuffles and one shared step, IEEE scale/code, k 16-byte stores.
#include "ep_internal.h"

namespace ep {
namespace {

__global__ void __launch_bounds__(512) count_kernel(const int32_t* __restrict__ idx, int T, int E, int k, int tile,
                                                    int ntiles, int32_t* __restrict__ tile_counts,
                                                    int32_t* __restrict__ lrank, uint32_t* status,
                                                    uint32_t* ticket) {
  extern __shared__ uint32_t smem[];
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
    const int e = idx[base + p];
    if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
      raise_status(status, kStatusBadIndex);
      continue;
    }
    const int tl = p / k;
    const uint32_t bit = 1u << (tl & 31);
    const uint32_t old = atomicOr(&mask[e * TW + (tl >> 5)], bit);
    if (old & bit) raise_status(status, kStatusBadIndex);  // expert repeated within one token
  }
  __syncthreads();
  if (nt == 0) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int e = warp; e < E; e += nw) {
    const int c = lane < TW ? __popc(mask[e * TW + lane]) : 0;
    const int incl = warp_inclusive_scan(c);
    if (lane < TW) pre[e * TW + lane] = static_cast<uint32_t>(incl - c);
    if (lane == 31) tile_counts[static_cast<int64_t>(e) * ntiles + b] = incl;
  }
  __syncthreads();

  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    const int e = idx[base + p];
    int r = -1;
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
      const int tl = p / k;
      const int w = tl >> 5;
      r = static_cast<int>(pre[e * TW + w]) + __popc(mask[e * TW + w] & ((1u << (tl & 31)) - 1u));
    }
    lrank[base + p] = r;
  }
}

// Exclusive scan of one value per thread over a 256-thread block; returns the
// exclusive prefix and sets `total` (same in every thread).
__device__ __forceinline__ int block_exclusive_scan_256(int v, int& total, int* warp_s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int incl = warp_inclusive_scan(v);
  __syncthreads();  // warp_s may still be read by a previous call
  if (lane == 31) warp_s[warp] = incl;
  __syncthreads();
  int wpre = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int x = warp_s[i];
    wpre += i < warp ? x : 0;
    tot += x;
  }
  total = tot;
  return wpre + incl - v;
}

__global__ void __launch_bounds__(256) scan_kernel(const int32_t* __restrict__ tile_counts, int E, int R, int ntiles,
                                                    int cap, int32_t* __restrict__ tile_base,
                                                    int32_t* __restrict__ expert_counts,
                                                    int32_t* __restrict__ expert_raw,
                                                    int32_t* __restrict__ expert_off, int32_t* __restrict__ rank_off,
                                                    int32_t* __restrict__ n_dropped, int32_t* kept_g,
                                                    int32_t* drop_g, uint32_t* ticket) {
  __shared__ int warp_s[8];
  __shared__ int is_last;
  const int e = blockIdx.x;
  // this expert's running sum over tiles
  int carry = 0;
  for (int c0 = 0; c0 < ntiles; c0 += blockDim.x) {
    const int i = c0 + threadIdx.x;
    const int v = i < ntiles ? tile_counts[static_cast<int64_t>(e) * ntiles + i] : 0;
    int tot;
    const int ex = block_exclusive_scan_256(v, tot, warp_s);
    if (i < ntiles) tile_base[static_cast<int64_t>(e) * ntiles + i] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) {
    const int kept = min(carry, cap);
    expert_counts[e] = kept;
    if (expert_raw) expert_raw[e] = carry;
    kept_g[e] = kept;
    drop_g[e] = carry - kept;
    __threadfence();
    const unsigned prev = atomicAdd(ticket, 1u);
    is_last = (prev == static_cast<unsigned>(gridDim.x) - 1u);
  }
  __syncthreads();
  if (!is_last) return;

  // last CTA: every other CTA's kept/drop values are visible (fence + ticket)
  __threadfence();
  int carry_off = 0, drops = 0;
  for (int c0 = 0; c0 < E; c0 += blockDim.x) {
    const int i = c0 + threadIdx.x;
    const int v = i < E ? __ldcg(kept_g + i) : 0;
    const int d = i < E ? __ldcg(drop_g + i) : 0;
    int tot, dtot;
    const int ex = block_exclusive_scan_256(v, tot, warp_s);
    block_exclusive_scan_256(d, dtot, warp_s);
    if (i < E) expert_off[i] = carry_off + ex;
    // rank r starts at its first expert r*G
    const int G = E / R;
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

__global__ void __launch_bounds__(256) rows_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ lrank,
                                                    const int32_t* __restrict__ tile_base,
                                                    const int32_t* __restrict__ expert_off, int64_t npairs, int E,
                                                    int k, int tile_log2, int ntiles, int cap,
                                                    int32_t* __restrict__ slot_row, int32_t* __restrict__ row_slot) {
  for (int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p < npairs;
       p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int e = idx[p];
    const int lr = lrank[p];
    int row = -1;
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E) && lr >= 0) {
      const int64_t t = p / k;
      const int pos = tile_base[static_cast<int64_t>(e) * ntiles + (t >> tile_log2)] + lr;
      if (pos < cap) row = expert_off[e] + pos;
    }
    slot_row[p] = row;
    if (row >= 0) row_slot[row] = static_cast<int32_t>(p);
  }
}

template <bool INT8>
__global__ void __launch_bounds__(1024) scatter_kernel(const DispatchArgs a) {
  __shared__ int32_t rows_s[2][32];
  __shared__ float amax_s[2][32];
  const int c = threadIdx.x;
  const int nchunk = a.H >> 4;  // 16 elements per thread
  const bool on = c < nchunk;
  const int warp = c >> 5, lane = c & 31, nw = blockDim.x >> 5;
  const char* xb = static_cast<const char*>(a.x);

  int64_t t = blockIdx.x;
  uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0;
  int my_row = -1;  // threads c < k: destination row of slot c of token t
  if (t < a.T) {
    if (on) {
      const char* p = xb + (t * a.H + 16 * c) * 2;
      a0 = ld_stream_v4(p);
      a1 = ld_stream_v4(p + 16);
    }
    if (c < a.k) my_row = a.slot_row[t * a.k + c];
  }
  int buf = 0;
  for (; t < a.T; t += gridDim.x) {
    // prefetch the next token's x chunk and slot rows while this one is coded
    const int64_t tn = t + gridDim.x;
    uint4 n0 = make_uint4(0, 0, 0, 0), n1 = n0;
    int next_row = -1;
    if (tn < a.T) {
      if (on) {
        const char* p = xb + (tn * a.H + 16 * c) * 2;
        n0 = ld_stream_v4(p);
        n1 = ld_stream_v4(p + 16);
      }
      if (c < a.k) next_row = a.slot_row[tn * a.k + c];
    }
    if (c < a.k) rows_s[buf][c] = my_row;
    float scale = 0.f;
    if constexpr (INT8) {
      float m = on ? fmaxf(absmax_bf16x8(a0), absmax_bf16x8(a1)) : 0.f;
      m = warp_max(m);
      if (lane == 0) amax_s[buf][warp] = m;
      __syncthreads();
      float am = amax_s[buf][0];
      for (int i = 1; i < nw; ++i) am = fmaxf(am, amax_s[buf][i]);
      scale = __fdiv_rn(am, 127.0f);
    } else {
      __syncthreads();
    }
    if (on) {
      if constexpr (INT8) {
        const uint4 q = quant16(a0, a1, scale);
        for (int j = 0; j < a.k; ++j) {
          const int row = rows_s[buf][j];
          if (row >= 0) st_v4(static_cast<int8_t*>(a.payload) + static_cast<int64_t>(row) * a.H + 16 * c, q);
        }
      } else {
        for (int j = 0; j < a.k; ++j) {
          const int row = rows_s[buf][j];
          if (row >= 0) {
            char* p = static_cast<char*>(a.payload) + (static_cast<int64_t>(row) * a.H + 16 * c) * 2;
            st_v4(p, a0);
            st_v4(p + 16, a1);
          }
        }
      }
    }
    if constexpr (INT8) {
      if (c < a.k && my_row >= 0) a.scales[my_row] = scale;
    }
    a0 = n0;
    a1 = n1;
    my_row = next_row;
    buf ^= 1;
  }
}

int count_smem_bytes(int E, int tile) { return 2 * E * (tile / 32) * static_cast<int>(sizeof(uint32_t)); }

int g_count_smem_set[64];  // per device: largest dynamic shared size already allowed

}  // namespace

cudaError_t launch_dispatch(const DispatchArgs& a, int sms, cudaStream_t s) {
  cudaError_t err;
  // count: also clears the scan's ticket, so it runs even for an empty batch
  const int smem = count_smem_bytes(a.E, a.tile);
  if (smem > 48 * 1024) {
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if (dev >= 64 || g_count_smem_set[dev] < smem) {
      err = cudaFuncSetAttribute(count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (err != cudaSuccess) return err;
      if (dev < 64) g_count_smem_set[dev] = smem;
    }
  }
  int cblock = ((a.tile * a.k + 31) / 32) * 32;
  cblock = cblock < 64 ? 64 : (cblock > 512 ? 512 : cblock);
  count_kernel<<<a.ntiles > 0 ? a.ntiles : 1, cblock, smem, s>>>(a.topk_idx, a.T, a.E, a.k, a.tile, a.ntiles,
                                                                 a.tile_counts, a.lrank, a.status, a.ticket);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  scan_kernel<<<a.E, 256, 0, s>>>(a.tile_counts, a.E, a.R, a.ntiles, a.cap, a.tile_base, a.expert_counts,
                                  a.expert_raw, a.expert_off, a.rank_off, a.n_dropped, a.kept, a.dropped, a.ticket);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if (a.T == 0) return cudaSuccess;

  const int64_t npairs = static_cast<int64_t>(a.T) * a.k;
  const int64_t rblocks_need = (npairs + 255) / 256;
  const int64_t rblocks_cap = static_cast<int64_t>(sms) * 8;
  const int tile_log2 = __builtin_ctz(static_cast<unsigned>(a.tile));
  rows_kernel<<<static_cast<int>(rblocks_need < rblocks_cap ? rblocks_need : rblocks_cap), 256, 0, s>>>(
      a.topk_idx, a.lrank, a.tile_base, a.expert_off, npairs, a.E, a.k, tile_log2, a.ntiles, a.cap, a.slot_row,
      a.row_slot);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;

  const int nchunk = a.H / 16;
  const int block = ((nchunk + 31) / 32) * 32;
  const int per_sm = block >= 2048 ? 1 : 2048 / block;
  const int64_t want = static_cast<int64_t>(sms) * per_sm;
  const int grid = static_cast<int>(a.T < want ? a.T : want);
  if (a.int8)
    scatter_kernel<true><<<grid, block, 0, s>>>(a);
  else
    scatter_kernel<false><<<grid, block, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ep
