// dispatch.cu — rank-major send layout: histogram, device-wide scan, and a
// stable scatter fused with the per-token int8 code.
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
//            tile's tokens in shared memory (atomicOr, order-free), their
//            popcounts give each tile's per-expert count and each pair's
//            rank within the tile in token order;
//   scan     one CTA: per expert, the exclusive running sum over tiles (the
//            pair's position within its expert), the capacity clip, then the
//            exclusive running sum over experts (expert_off, rank_off);
//   scatter  a grid-stride loop over tokens, one CTA per token row in
//            flight: 16 elements per thread, 16-byte loads of x (the next
//            token's row prefetched), amax by warp shuffles and one shared
//            step, IEEE scale/code, and k 16-byte stores per thread.
#include "ep_internal.h"

namespace ep {
namespace {

__global__ void __launch_bounds__(512) count_kernel(const int32_t* __restrict__ idx, int T, int E, int k, int tile,
                                                    int ntiles, int32_t* __restrict__ tile_counts,
                                                    int32_t* __restrict__ lrank, uint32_t* status) {
  extern __shared__ uint32_t smem[];
  const int TW = tile >> 5;
  uint32_t* mask = smem;         // [E][TW] bit t of word w: token w*32+t of the tile chose e
  uint32_t* pre = smem + E * TW;  // [E][TW] set bits of e in the words before w
  const int b = blockIdx.x;
  const int64_t t0 = static_cast<int64_t>(b) * tile;
  const int nt = static_cast<int>(min(static_cast<int64_t>(tile), static_cast<int64_t>(T) - t0));
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

__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ tile_counts, int E, int R,
                                                     int ntiles, int cap, int32_t* __restrict__ tile_base,
                                                     int32_t* __restrict__ expert_counts,
                                                     int32_t* __restrict__ expert_raw,
                                                     int32_t* __restrict__ expert_off,
                                                     int32_t* __restrict__ rank_off,
                                                     int32_t* __restrict__ n_dropped) {
  __shared__ int32_t kept_s[1025];
  __shared__ int32_t drop_s[1024];
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t warp_drop[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;

  // per expert: running sum over tiles -> each tile's first position
  for (int e = warp; e < E; e += nw) {
    int carry = 0;
    for (int c0 = 0; c0 < ntiles; c0 += 32) {
      const int i = c0 + lane;
      const int v = i < ntiles ? tile_counts[static_cast<int64_t>(e) * ntiles + i] : 0;
      const int incl = warp_inclusive_scan(v);
      if (i < ntiles) tile_base[static_cast<int64_t>(e) * ntiles + i] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      const int kept = min(carry, cap);
      kept_s[e] = kept;
      drop_s[e] = carry - kept;
      if (expert_raw) expert_raw[e] = carry;
    }
  }
  __syncthreads();

  // exclusive running sum of the kept counts over experts (E <= 1024)
  const int e = threadIdx.x;
  const int v = e < E ? kept_s[e] : 0;
  int d = e < E ? drop_s[e] : 0;
  const int incl = warp_inclusive_scan(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
  if (lane == 31) warp_tot[warp] = incl;
  if (lane == 0) warp_drop[warp] = d;
  __syncthreads();
  if (warp == 0) {
    const int wt = lane < nw ? warp_tot[lane] : 0;
    const int wincl = warp_inclusive_scan(wt);
    warp_tot[lane] = wincl - wt;
    int dd = lane < nw ? warp_drop[lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, o);
    if (lane == 0) *n_dropped = dd;
  }
  __syncthreads();
  const int excl = warp_tot[warp] + incl - v;
  __syncthreads();  // every thread has read kept_s before it is overwritten
  if (e < E) {
    expert_counts[e] = v;
    expert_off[e] = excl;
    kept_s[e] = excl;
    if (e == E - 1) {
      expert_off[E] = excl + v;
      kept_s[E] = excl + v;
    }
  }
  if (E == 0 && e == 0) {
    expert_off[0] = 0;
    kept_s[0] = 0;
  }
  __syncthreads();
  const int G = R > 0 ? E / R : 1;
  for (int r = threadIdx.x; r <= R; r += blockDim.x) rank_off[r] = kept_s[r * G];
}

template <bool INT8>
__global__ void __launch_bounds__(1024) scatter_kernel(const DispatchArgs a) {
  __shared__ int32_t rows_s[2][32];
  __shared__ float amax_s[2][32];
  const int c = threadIdx.x;
  const int nchunk = a.H >> 4;  // 16 elements per thread
  const bool on = c < nchunk;
  const int warp = c >> 5, lane = c & 31, nw = blockDim.x >> 5;
  const int tile_log2 = __ffs(a.tile) - 1;
  const char* xb = static_cast<const char*>(a.x);

  int64_t t = blockIdx.x;
  uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0;
  if (t < a.T && on) {
    const char* p = xb + (t * a.H + 16 * c) * 2;
    a0 = ld_stream_v4(p);
    a1 = ld_stream_v4(p + 16);
  }
  int buf = 0;
  for (; t < a.T; t += gridDim.x) {
    // prefetch the next token's chunk while this one is coded and stored
    const int64_t tn = t + gridDim.x;
    uint4 n0 = make_uint4(0, 0, 0, 0), n1 = n0;
    if (tn < a.T && on) {
      const char* p = xb + (tn * a.H + 16 * c) * 2;
      n0 = ld_stream_v4(p);
      n1 = ld_stream_v4(p + 16);
    }
    // destination row of each slot: expert_off[e] + first position of the
    // tile within e + rank within the tile; past the cap -> dropped
    if (c < a.k) {
      const int64_t s = t * a.k + c;
      const int e = a.topk_idx[s];
      const int lr = a.lrank[s];
      int row = -1;
      if (static_cast<unsigned>(e) < static_cast<unsigned>(a.E) && lr >= 0) {
        const int pos = a.tile_base[static_cast<int64_t>(e) * a.ntiles + (t >> tile_log2)] + lr;
        if (pos < a.cap) row = a.expert_off[e] + pos;
      }
      rows_s[buf][c] = row;
      a.slot_row[s] = row;
      if (row >= 0) a.row_slot[row] = static_cast<int32_t>(s);
    }
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
      if (c < a.k) {
        const int row = rows_s[buf][c];
        if (row >= 0) a.scales[row] = scale;
      }
    }
    a0 = n0;
    a1 = n1;
    buf ^= 1;
  }
}

int count_smem_bytes(int E, int tile) { return 2 * E * (tile / 32) * static_cast<int>(sizeof(uint32_t)); }

}  // namespace

cudaError_t launch_dispatch(const DispatchArgs& a, int sms, cudaStream_t s) {
  cudaError_t err;
  if (a.T > 0) {
    const int smem = count_smem_bytes(a.E, a.tile);
    if (smem > 48 * 1024) {
      err = cudaFuncSetAttribute(count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (err != cudaSuccess) return err;
    }
    count_kernel<<<a.ntiles, 512, smem, s>>>(a.topk_idx, a.T, a.E, a.k, a.tile, a.ntiles, a.tile_counts, a.lrank,
                                             a.status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  scan_kernel<<<1, 1024, 0, s>>>(a.tile_counts, a.E, a.R, a.ntiles, a.cap, a.tile_base, a.expert_counts,
                                 a.expert_raw, a.expert_off, a.rank_off, a.n_dropped);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if (a.T == 0) return cudaSuccess;
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
