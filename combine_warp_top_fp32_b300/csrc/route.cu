// route.cu — warp-level top-k gating with softmax weights over fp32 logits.
//
// Computes, per token, the k experts with the largest router logit (ties to
// the lower expert id) and their softmax weights: the Router of the MoE
// sparse-communication article (intelliparadigm.com, §2.1), which applies
// softmax over all E logits and then topk. Selecting on the logits is the
// same selection (softmax is monotone) without ties invented by rounding.
//
// Design (one token per group of L lanes, L = min(32, pow2ceil(E))):
//   - the row is read once with coalesced loads (16-byte float4 loads when
//     L == 32 and E % 128 == 0), each lane holding VPL = ceil(E/L) values;
//   - each value becomes a 64-bit key (order-preserving float bits << 32 |
//     ~expert id), so one unsigned max picks (logit desc, id asc) exactly;
//   - k rounds of: lane-local max, group max, the owner clears the winning
//     key; lane j keeps slot j. With one token per warp (E >= 32) the group
//     max is two redux.sync reductions (value max, then lowest id holding
//     it), and for E <= 256 each lane sorts its keys once so that its local
//     max is always its first key; with several tokens per warp the group max
//     is a __shfl_xor_sync butterfly;
//   - softmax denominator: exp(l - l_max) with the subtraction's rounding
//     error carried into the exponential (exp_shifted_term), summed with
//     compensated (TwoSum) arithmetic; each chosen expert's numerator uses
//     expf, so the weight stays within 1e-6 of the exact value.
//
// Kernels: route_topk_kernel (ep_route: routing alone, a grid-stride loop
// over tokens); route_count_kernel (ep_route_dispatch: one CTA per tile of
// tokens routes the tile and writes its per-expert counts and in-tile ranks,
// the dispatch's count step); route_layout_cluster_kernel (ep_route_dispatch
// on batches of at most eight 32-token tiles: one thread-block cluster routes
// the batch and forms the whole layout, the count and scan steps together).
#include "ep_internal.h"
#include "layout.cuh"

namespace ep {
namespace {

// Float -> unsigned key whose unsigned order is the float order; -0 and +0
// map to the same key (they compare equal as floats): adding +0 turns -0 into
// +0 and leaves every other value unchanged; then negative values have all
// bits flipped and non-negative ones only the sign bit.
__device__ __forceinline__ uint32_t ordered_bits(float v) {
  const uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));
  return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint64_t key) {
  uint32_t o = static_cast<uint32_t>(key >> 32);
  uint32_t u = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
  return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t make_key(float v, int e) {
  return (static_cast<uint64_t>(ordered_bits(v)) << 32) | static_cast<uint32_t>(0xffffffffu - static_cast<uint32_t>(e));
}

__device__ __forceinline__ int key_expert(uint64_t key) {
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(key));
}

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }

// Compare-exchange so that key[i] >= key[j].
template <int N>
__device__ __forceinline__ void cx(uint64_t (&key)[N], int i, int j) {
  const uint64_t a = key[i], b = key[j];
  key[i] = a > b ? a : b;
  key[j] = a > b ? b : a;
}

// Sorts a lane's keys in descending order (fixed networks: Batcher's
// odd-even merge sort for 8, its 5-exchange form for 4).
template <int N>
__device__ __forceinline__ void sort_desc(uint64_t (&key)[N]) {
  if constexpr (N == 2) {
    cx(key, 0, 1);
  } else if constexpr (N == 4) {
    cx(key, 0, 1); cx(key, 2, 3); cx(key, 0, 2); cx(key, 1, 3); cx(key, 1, 2);
  } else if constexpr (N == 8) {
    cx(key, 0, 1); cx(key, 2, 3); cx(key, 4, 5); cx(key, 6, 7);
    cx(key, 0, 2); cx(key, 1, 3); cx(key, 4, 6); cx(key, 5, 7);
    cx(key, 1, 2); cx(key, 5, 6);
    cx(key, 0, 4); cx(key, 1, 5); cx(key, 2, 6); cx(key, 3, 7);
    cx(key, 2, 4); cx(key, 3, 5);
    cx(key, 1, 2); cx(key, 3, 4); cx(key, 5, 6);
  }
}

// exp(v - m) with the rounding error of the subtraction folded back in:
// v - m = d + err exactly (TwoSum), exp(d + err) ~= exp(d) * (1 + err).
__device__ __forceinline__ float exp_shifted(float v, float m) {
  const float nm = -m;
  const float d = __fadd_rn(v, nm);
  const float bb = __fsub_rn(d, v);
  const float err = __fadd_rn(__fsub_rn(v, __fsub_rn(d, bb)), __fsub_rn(nm, bb));
  const float e = expf(d);
  return __fmaf_rn(e, err, e);
}

// exp(v - m) for a softmax denominator term, built on the hardware base-2
// exponential: v - m = d + err exactly (TwoSum); (d + err) * log2(e) is
// carried as p + c with p = fl(d * L1), L1 = log2(e) rounded to fp32, and c
// collecting the product's exact rounding error (fma), d * (log2(e) - L1) and
// err * L1; then 2^(p + c) ~= 2^p * (1 + c * ln 2). Relative error about 3.4
// fp32 ulp (measured over d in [-87, 0] against a double-precision exp),
// against 2.6 for expf. Results below 2^-126 flush to zero, which changes a
// sum that is at least 1 by less than 2^-126 per term.
__device__ __forceinline__ float exp_shifted_term(float v, float m) {
  constexpr float kLog2eHi = 1.44269502162933349609375f;  // fp32 nearest to log2(e)
  constexpr float kLog2eLo = 1.925963033500011e-08f;      // log2(e) - kLog2eHi
  constexpr float kLn2 = 0.693147180559945309f;
  const float nm = -m;
  const float d = __fadd_rn(v, nm);
  const float bb = __fsub_rn(d, v);
  const float err = __fadd_rn(__fsub_rn(v, __fsub_rn(d, bb)), __fsub_rn(nm, bb));
  const float p = __fmul_rn(d, kLog2eHi);
  const float c = __fmaf_rn(err, kLog2eHi, __fmaf_rn(d, kLog2eLo, __fmaf_rn(d, kLog2eHi, -p)));
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(p));
  return __fmaf_rn(r, __fmul_rn(c, kLn2), r);
}

// Compensated accumulation of x into (s, c): TwoSum gives the exact rounding
// error of s + x, which is added to the running correction c.
__device__ __forceinline__ void comp_add(float& s, float& c, float x) {
  const float t = __fadd_rn(s, x);
  const float bb = __fsub_rn(t, s);
  c = __fadd_rn(c, __fadd_rn(__fsub_rn(s, __fsub_rn(t, bb)), __fsub_rn(x, bb)));
  s = t;
}

// Butterfly sum of compensated pairs over the L-lane group; every lane of the
// group ends with the same (s, c) because each step is symmetric.
__device__ __forceinline__ float group_comp_sum(float s, float c, int L) {
  for (int o = L >> 1; o > 0; o >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float c2 = __shfl_xor_sync(0xffffffffu, c, o);
    const float t = __fadd_rn(s, s2);
    const float bb = __fsub_rn(t, s);
    const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bb)), __fsub_rn(s2, bb));
    c = __fadd_rn(__fadd_rn(c, c2), err);
    s = t;
  }
  return __fadd_rn(s, c);
}

// Routes one token per L-lane group: on return lanes sub < k of the group
// hold slot sub's expert id (*e_out) and weight (*w_out). All 32 lanes of the
// warp must call it together (warp-wide reductions).
template <int VPL, bool VEC4>
__device__ __forceinline__ void route_token(const float* __restrict__ logits, int64_t t, bool active, int E, int k,
                                            int L, int sub, int renorm, int* e_out, float* w_out) {
  const float* row = logits + (active ? t : 0) * static_cast<int64_t>(E);

  float val[VPL];
  uint64_t key[VPL];
  if constexpr (VEC4) {
    // lane `sub` holds experts 4*sub + 128*i + c, i < VPL/4, c < 4
#pragma unroll
    for (int i = 0; i < VPL / 4; ++i) {
      const int e0 = 4 * sub + 128 * i;
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (active) f = __ldg(reinterpret_cast<const float4*>(row + e0));
      val[4 * i + 0] = f.x;
      val[4 * i + 1] = f.y;
      val[4 * i + 2] = f.z;
      val[4 * i + 3] = f.w;
#pragma unroll
      for (int c = 0; c < 4; ++c) key[4 * i + c] = active ? make_key(val[4 * i + c], e0 + c) : 0ull;
    }
  } else {
    // lane `sub` holds experts sub + L*i
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = sub + L * i;
      const bool ok = active && e < E;
      val[i] = ok ? __ldg(row + e) : 0.f;
      key[i] = ok ? make_key(val[i], e) : 0ull;  // 0 is below every real key
    }
  }

  // k rounds of group argmax; lane j of the group keeps slot j.
  int my_e = 0;
  float my_v = 0.f;
  float l_max = 0.f;
  if (L == 32 && VPL <= 8) {
    // One token per warp, each lane's keys sorted once (largest first):
    // every round the lanes offer their head key; redux.sync max over the
    // value bits finds the largest logit, redux.sync min over the ids of
    // the lanes offering it breaks the tie toward the lower expert id, and
    // the winning lane drops its head (a shift of its sorted list).
    sort_desc<VPL>(key);
    uint32_t my_bits = 0, max_bits = 0;
    for (int r = 0; r < k; ++r) {
      const uint32_t hv = static_cast<uint32_t>(key[0] >> 32);
      const uint32_t gmax = __reduce_max_sync(0xffffffffu, hv);
      const uint32_t cand = (hv == gmax) ? 0xffffffffu - static_cast<uint32_t>(key[0]) : 0xffffffffu;
      const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
      if (r == 0) max_bits = gmax;
      if (sub == r) {
        my_e = static_cast<int>(win);
        my_bits = gmax;
      }
      if (cand == win) {
#pragma unroll
        for (int i = 0; i + 1 < VPL; ++i) key[i] = key[i + 1];
        key[VPL - 1] = 0ull;  // 0 is below every real key
      }
    }
    l_max = key_value(static_cast<uint64_t>(max_bits) << 32);
    my_v = key_value(static_cast<uint64_t>(my_bits) << 32);
  } else if (L == 32) {
    // One token per warp: two single-instruction warp reductions per round.
    // redux.sync max over the order-preserving value bits finds the largest
    // logit, redux.sync min over the ids of the lanes holding it breaks the
    // tie toward the lower expert id. Within a lane the ids grow with i, so
    // a strict '>' keeps the lowest id among the lane's equal values.
    uint32_t ob[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) ob[i] = static_cast<uint32_t>(key[i] >> 32);
    for (int r = 0; r < k; ++r) {
      uint32_t bv = ob[0];
      int bi = 0;
#pragma unroll
      for (int i = 1; i < VPL; ++i)
        if (ob[i] > bv) {
          bv = ob[i];
          bi = i;
        }
      const uint32_t gmax = __reduce_max_sync(0xffffffffu, bv);
      uint32_t my_id = 0xffffffffu;
#pragma unroll
      for (int i = 0; i < VPL; ++i)
        if (i == bi) my_id = 0xffffffffu - static_cast<uint32_t>(key[i]);
      const uint32_t cand = (bv == gmax) ? my_id : 0xffffffffu;
      const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
      const float v = key_value(static_cast<uint64_t>(gmax) << 32);
      if (r == 0) l_max = v;
      if (sub == r) {
        my_e = static_cast<int>(win);
        my_v = v;
      }
      if (cand == win) {
#pragma unroll
        for (int i = 0; i < VPL; ++i)
          if (i == bi) ob[i] = 0u;  // 0 is below every real value
      }
    }
  } else {
    for (int r = 0; r < k; ++r) {
      uint64_t best = key[0];
#pragma unroll
      for (int i = 1; i < VPL; ++i) best = umax64(best, key[i]);
      for (int o = L >> 1; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
      const float v = key_value(best);
      if (r == 0) l_max = v;
      if (sub == r) {
        my_e = key_expert(best);
        my_v = v;
      }
#pragma unroll
      for (int i = 0; i < VPL; ++i)
        if (key[i] == best) key[i] = 0ull;
    }
  }

  // softmax denominator: all E experts, or the k chosen when renormalising
  float s = 0.f, c = 0.f;
  if (renorm) {
    if (sub < k) s = exp_shifted_term(my_v, l_max);
  } else {
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      bool ok;
      if constexpr (VEC4)
        ok = active;
      else
        ok = active && (sub + L * i) < E;
      if (ok) comp_add(s, c, exp_shifted_term(val[i], l_max));
    }
  }
  const float denom = group_comp_sum(s, c, L);

  *e_out = my_e;
  *w_out = __fdiv_rn(exp_shifted(my_v, l_max), denom);
}

// NQ tokens per warp at once (one token per 32 lanes, E >= 32, at most 8
// values per lane; the kernels use NQ = 2 up to 4 values per lane, where the
// doubled registers still leave room for many warps): the same steps as route_token on the sorted-key path, with
// every per-token value held for all NQ tokens so that the NQ independent
// chains of reductions and exponentials interleave in one warp. On return lane
// j < k holds slot j of token q in e_out[q] / w_out[q].
template <int NQ, int VPL, bool VEC4>
__device__ __forceinline__ void route_tokens_sorted(const float* __restrict__ logits, const int64_t (&t)[NQ],
                                                    const bool (&active)[NQ], int E, int k, int lane, int renorm,
                                                    int (&e_out)[NQ], float (&w_out)[NQ]) {
  float val[NQ][VPL];
  uint64_t key[NQ][VPL];
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const float* row = logits + (active[q] ? t[q] : 0) * static_cast<int64_t>(E);
    if constexpr (VEC4) {
#pragma unroll
      for (int i = 0; i < VPL / 4; ++i) {
        const int e0 = 4 * lane + 128 * i;
        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
        if (active[q]) f = __ldg(reinterpret_cast<const float4*>(row + e0));
        val[q][4 * i + 0] = f.x;
        val[q][4 * i + 1] = f.y;
        val[q][4 * i + 2] = f.z;
        val[q][4 * i + 3] = f.w;
#pragma unroll
        for (int c = 0; c < 4; ++c) key[q][4 * i + c] = active[q] ? make_key(val[q][4 * i + c], e0 + c) : 0ull;
      }
    } else {
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        const bool ok = active[q] && e < E;
        val[q][i] = ok ? __ldg(row + e) : 0.f;
        key[q][i] = ok ? make_key(val[q][i], e) : 0ull;
      }
    }
  }
#pragma unroll
  for (int q = 0; q < NQ; ++q) sort_desc<VPL>(key[q]);

  uint32_t my_bits[NQ], max_bits[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    my_bits[q] = 0u;
    max_bits[q] = 0u;
    e_out[q] = 0;
  }
  for (int r = 0; r < k; ++r) {
    uint32_t gmax[NQ], cand[NQ], win[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) gmax[q] = __reduce_max_sync(0xffffffffu, static_cast<uint32_t>(key[q][0] >> 32));
#pragma unroll
    for (int q = 0; q < NQ; ++q)
      cand[q] = (static_cast<uint32_t>(key[q][0] >> 32) == gmax[q]) ? 0xffffffffu - static_cast<uint32_t>(key[q][0])
                                                                      : 0xffffffffu;
#pragma unroll
    for (int q = 0; q < NQ; ++q) win[q] = __reduce_min_sync(0xffffffffu, cand[q]);
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (r == 0) max_bits[q] = gmax[q];
      if (lane == r) {
        e_out[q] = static_cast<int>(win[q]);
        my_bits[q] = gmax[q];
      }
      if (cand[q] == win[q]) {
#pragma unroll
        for (int i = 0; i + 1 < VPL; ++i) key[q][i] = key[q][i + 1];
        key[q][VPL - 1] = 0ull;  // 0 is below every real key
      }
    }
  }

  float l_max[NQ], my_v[NQ], s[NQ], c[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    l_max[q] = key_value(static_cast<uint64_t>(max_bits[q]) << 32);
    my_v[q] = key_value(static_cast<uint64_t>(my_bits[q]) << 32);
    s[q] = 0.f;
    c[q] = 0.f;
  }
  if (renorm) {
#pragma unroll
    for (int q = 0; q < NQ; ++q)
      if (lane < k) s[q] = exp_shifted_term(my_v[q], l_max[q]);
  } else {
#pragma unroll
    for (int i = 0; i < VPL; ++i)
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const bool ok = VEC4 ? active[q] : (active[q] && (lane + 32 * i) < E);
        if (ok) comp_add(s[q], c[q], exp_shifted_term(val[q][i], l_max[q]));
      }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const float s2 = __shfl_xor_sync(0xffffffffu, s[q], o);
      const float c2 = __shfl_xor_sync(0xffffffffu, c[q], o);
      const float tt = __fadd_rn(s[q], s2);
      const float bb = __fsub_rn(tt, s[q]);
      const float err = __fadd_rn(__fsub_rn(s[q], __fsub_rn(tt, bb)), __fsub_rn(s2, bb));
      c[q] = __fadd_rn(__fadd_rn(c[q], c2), err);
      s[q] = tt;
    }
  }
#pragma unroll
  for (int q = 0; q < NQ; ++q) w_out[q] = __fdiv_rn(exp_shifted(my_v[q], l_max[q]), __fadd_rn(s[q], c[q]));
}

template <int VPL, bool VEC4>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int lanes_log2, int renorm, int32_t* __restrict__ topk_idx,
                                                         float* __restrict__ topk_w) {
  const int L = 1 << lanes_log2;
  const int lane = threadIdx.x & 31;
  const int sub = lane & (L - 1);
  const int groups_per_warp = 32 >> lanes_log2;
  const int grp = lane >> lanes_log2;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  pdl_wait();  // the logits may come from the kernel before this one
  pdl_launch_dependents();

  if constexpr (VPL <= 4) {
    if (L == 32) {  // two tokens per warp in flight: tokens w and w + n_warps
      for (int64_t tb = warp_id; tb < T; tb += 2 * n_warps) {
        const int64_t tq[2] = {tb, tb + n_warps};
        const bool act[2] = {true, tb + n_warps < T};
        int e[2];
        float w[2];
        route_tokens_sorted<2, VPL, VEC4>(logits, tq, act, E, k, lane, renorm, e, w);
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (act[q] && lane < k) {
            topk_idx[tq[q] * k + lane] = e[q];
            topk_w[tq[q] * k + lane] = w[q];
          }
      }
      return;
    }
  }
  for (int64_t tb = warp_id * groups_per_warp; tb < T; tb += n_warps * groups_per_warp) {
    const int64_t t = tb + grp;
    const bool active = t < T;
    int e;
    float w;
    route_token<VPL, VEC4>(logits, t, active, E, k, L, sub, renorm, &e, &w);
    if (active && sub < k) {
      topk_idx[t * k + sub] = e;
      topk_w[t * k + sub] = w;
    }
  }
}

// Routes the nt tokens of the tile starting at token t0 (one L-lane group
// per token; two tokens per warp in flight when L = 32 and VPL <= 4), writes
// their slots and sets their bits in the tile's per-expert masks in shared
// memory: mask[e][w] bit b = token 32w+b of the tile chose e. The masks must
// be zero on entry; the caller synchronises the CTA afterwards.
template <int VPL, bool VEC4>
__device__ __forceinline__ void route_tile(const float* __restrict__ logits, int64_t t0, int nt, int E, int k,
                                           int lanes_log2, int renorm, int TW, uint32_t* mask,
                                           int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  const int L = 1 << lanes_log2;
  const int lane = threadIdx.x & 31;
  const int sub = lane & (L - 1);
  const int groups_per_warp = 32 >> lanes_log2;
  const int grp = lane >> lanes_log2;
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  bool routed = false;
  if constexpr (VPL <= 4) {
    if (L == 32) {  // two tokens per warp in flight: tile tokens w and w + nw
      for (int tl0 = warp; tl0 < nt; tl0 += 2 * nw) {
        const int tlq[2] = {tl0, tl0 + nw};
        const int64_t tq[2] = {t0 + tl0, t0 + tl0 + nw};
        const bool act[2] = {true, tl0 + nw < nt};
        int e[2];
        float w[2];
        route_tokens_sorted<2, VPL, VEC4>(logits, tq, act, E, k, lane, renorm, e, w);
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (act[q] && lane < k) {
            topk_idx[tq[q] * k + lane] = e[q];
            topk_w[tq[q] * k + lane] = w[q];
            atomicOr(&mask[e[q] * TW + (tlq[q] >> 5)], 1u << (tlq[q] & 31));
          }
      }
      routed = true;
    }
  }
  if (!routed) {
    for (int tl0 = warp * groups_per_warp; tl0 < nt; tl0 += nw * groups_per_warp) {
      const int tl = tl0 + grp;
      const bool active = tl < nt;
      const int64_t t = t0 + tl;
      int e;
      float w;
      route_token<VPL, VEC4>(logits, t, active, E, k, L, sub, renorm, &e, &w);
      if (active && sub < k) {
        topk_idx[t * k + sub] = e;
        topk_w[t * k + sub] = w;
        atomicOr(&mask[e * TW + (tl >> 5)], 1u << (tl & 31));
      }
    }
  }
}

// Routing fused with the per-tile count of the dispatch (the ThunderEP
// article's §5.2 suggestion to bucket by destination while routing): CTA b
// routes the tokens of tile b = [b*tile, (b+1)*tile), writes their slots,
// and builds the tile's per-expert bit masks in shared memory, from which it
// writes the tile's count per expert and each pair's rank within the tile in
// token order (the same tile_counts / lrank as the dispatch's count kernel).
template <int VPL, bool VEC4>
__global__ void __launch_bounds__(VPL >= 16 ? 256 : 512) route_count_kernel(
    const float* __restrict__ logits, int T, int E, int k, int lanes_log2, int renorm, int tile, int ntiles,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ tile_counts,
    int32_t* __restrict__ lrank, uint32_t* ticket) {
  extern __shared__ uint32_t smem[];
  const int TW = tile >> 5;
  uint32_t* mask = smem;          // [E][TW] bit b of word w: token 32*w+b of the tile chose e
  uint32_t* pre = smem + E * TW;  // [E][TW] set bits of e in the words before w
  const int b = blockIdx.x;
  const int64_t t0 = static_cast<int64_t>(b) * tile;
  const int nt = static_cast<int>(min(static_cast<int64_t>(tile), T - t0));
  for (int i = threadIdx.x; i < E * TW; i += blockDim.x) mask[i] = 0u;
  pdl_wait();  // the logits may come from the kernel before this one
  pdl_launch_dependents();
  if (b == 0 && threadIdx.x == 0) *ticket = 0u;  // the scan that follows counts its CTAs from 0
  __syncthreads();
  if (nt <= 0) return;  // an empty batch: only the ticket
  route_tile<VPL, VEC4>(logits, t0, nt, E, k, lanes_log2, renorm, TW, mask, topk_idx, topk_w);
  __syncthreads();

  tile_word_prefix(mask, pre, E, TW, tile_counts, ntiles, b);
  __syncthreads();

  const int64_t base = t0 * k;
  for (int p = threadIdx.x; p < nt * k; p += blockDim.x) {
    const int e = topk_idx[base + p];  // written above by this CTA
    const int tl = p / k;
    const int w = tl >> 5;
    lrank[base + p] = static_cast<int>(pre[e * TW + w]) + __popc(mask[e * TW + w] & ((1u << (tl & 31)) - 1u));
  }
}

// Small batches (at most kClusterTiles tiles of 32 tokens): one cluster of
// one CTA per tile, a warp per token. Each CTA routes its tile and ranks its
// pairs as route_count_kernel does, but pushes its per-expert tile counts
// into CTA 0's shared memory instead of global memory; after a cluster
// barrier CTA 0 alone forms what the scan kernel would from them (tile bases,
// raw and kept counts, expert and rank offsets, the number dropped), so the
// whole layout costs one launch. The outputs are those of route_count_kernel
// + scan_kernel, bit for bit.
template <int VPL, bool VEC4>
__global__ void __launch_bounds__(1024, 1) route_layout_cluster_kernel(
    const float* __restrict__ logits, int T, int E, int k, int lanes_log2, int renorm, int R, int cap,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ lrank,
    int32_t* __restrict__ tile_base, int32_t* __restrict__ expert_counts, int32_t* __restrict__ expert_raw,
    int32_t* __restrict__ expert_off, int32_t* __restrict__ rank_off, int32_t* __restrict__ n_dropped) {
  extern __shared__ uint32_t smem[];
  const int C = gridDim.x;  // tiles = CTAs = the cluster
  uint32_t* mask = smem;                                // [E] this tile's word per expert
  int* counts_s = reinterpret_cast<int*>(smem + E);    // [E][C] (CTA 0) every tile's count per expert
  int* kept_s = counts_s + E * C;                      // [E] (CTA 0)
  int* drop_s = kept_s + E;                            // [E] (CTA 0)
  const int warp = threadIdx.x >> 5;
  const int b = blockIdx.x;
  const int64_t t0 = static_cast<int64_t>(b) * 32;
  const int nt = min(32, T - static_cast<int>(t0));  // >= 1: the grid has ceil(T/32) CTAs
  for (int i = threadIdx.x; i < E; i += blockDim.x) mask[i] = 0u;
  cluster_arrive_relaxed();  // CTA 0 must be running before anyone writes into it
  pdl_wait();                // the logits may come from the kernel before this one
  pdl_launch_dependents();
  __syncthreads();
  route_tile<VPL, VEC4>(logits, t0, nt, E, k, lanes_log2, renorm, 1, mask, topk_idx, topk_w);
  __syncthreads();

  cluster_wait();
  const uint32_t counts0 = cluster_map(counts_s, 0);
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    st_cluster_u32(counts0 + 4u * static_cast<uint32_t>(e * C + b), static_cast<uint32_t>(__popc(mask[e])));
  const int64_t base = t0 * k;
  for (int p = threadIdx.x; p < nt * k; p += blockDim.x) {
    const int e = topk_idx[base + p];  // written above by this CTA
    const int tl = p / k;
    lrank[base + p] = __popc(mask[e] & ((1u << tl) - 1u));
  }
  cluster_sync();  // every tile's counts are in CTA 0
  if (b != 0) return;

  // one thread per (expert, tile), segments of Cp lanes (C rounded up to a
  // power of two, the padding lanes adding 0): a segmented scan gives the
  // tile bases, and the segment's last lane the expert's raw total
  int Cp = 1;
  while (Cp < C) Cp <<= 1;
  for (int i0 = 0; i0 < E * Cp; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    const int e = i / Cp, w = i & (Cp - 1);  // w == lane & (Cp - 1): i0 is a multiple of 32
    const bool ok = i < E * Cp && w < C;
    const int c = ok ? counts_s[e * C + w] : 0;
    int v = c;
    for (int o = 1; o < Cp; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (w >= o) v += u;
    }
    if (ok) tile_base[e * C + w] = v - c;
    if (i < E * Cp && w == Cp - 1) {
      const int kept = min(v, cap);
      expert_counts[e] = kept;
      if (expert_raw) expert_raw[e] = v;
      kept_s[e] = kept;
      drop_s[e] = v - kept;
    }
  }
  __syncthreads();
  if (warp != 0) return;

  expert_offsets_warp(kept_s, drop_s, E, R, expert_off, rank_off, n_dropped);
}

template <int VPL, bool VEC4>
cudaError_t launch_route_layout_cluster_t(const RouteCountArgs& r, const DispatchArgs& a, int lanes_log2,
                                          cudaStream_t s) {
  constexpr int kBlock = 1024;  // a warp per token of the tile
  const int C = (r.T + 31) / 32;
  const int smem = (r.E + r.E * C + 2 * r.E) * static_cast<int>(sizeof(uint32_t));  // <= 11 KB
  static ClusterFits fits;
  return launch_cluster_pdl(route_layout_cluster_kernel<VPL, VEC4>, C, kBlock, static_cast<size_t>(smem), s, fits,
                            r.logits, r.T, r.E, r.k, lanes_log2, r.renorm, a.R, a.cap, r.topk_idx, r.topk_w, a.lrank,
                            a.tile_base, a.expert_counts, a.expert_raw, a.expert_off, a.rank_off, a.n_dropped);
}

template <int VPL, bool VEC4>
cudaError_t launch_route_t(const float* logits, int T, int E, int k, int lanes_log2, int renorm, int32_t* idx,
                           float* w, int sms, cudaStream_t s) {
  const int groups_per_warp = 32 >> lanes_log2;
  const int64_t warps = (static_cast<int64_t>(T) + groups_per_warp - 1) / groups_per_warp;
  const int64_t blocks_needed = (warps + 7) / 8;
  static int occ[64];  // one cache per template instance
  const int64_t cap_blocks = static_cast<int64_t>(sms) * resident_ctas(route_topk_kernel<VPL, VEC4>, 256, 0, occ);
  const int grid = static_cast<int>(blocks_needed < cap_blocks ? blocks_needed : cap_blocks);
  return launch_pdl(route_topk_kernel<VPL, VEC4>, grid, 256, 0, s, logits, T, E, k, lanes_log2, renorm, idx, w);
}

template <int VPL, bool VEC4>
cudaError_t launch_route_count_t(const RouteCountArgs& r, int lanes_log2, cudaStream_t s) {
  constexpr int kBlock = VPL >= 16 ? 256 : 512;
  static int smem_set[64];  // per device: largest dynamic shared size already allowed
  const int smem = 2 * r.E * (r.tile / 32) * static_cast<int>(sizeof(uint32_t));
  if (smem > 48 * 1024) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 64 || cache_load(&smem_set[dev]) < smem) {
      err = cudaFuncSetAttribute(route_count_kernel<VPL, VEC4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (err != cudaSuccess) return err;
      if (dev < 64) cache_store(&smem_set[dev], smem);
    }
  }
  return launch_pdl(route_count_kernel<VPL, VEC4>, r.ntiles > 0 ? r.ntiles : 1, kBlock, static_cast<size_t>(smem),
                    s, r.logits, r.T, r.E, r.k, lanes_log2, r.renorm, r.tile, r.ntiles, r.topk_idx, r.topk_w,
                    r.tile_counts, r.lrank, r.ticket);
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int renorm, int32_t* idx, float* w, int sms,
                         cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  int lanes_log2 = 0;
  while ((1 << lanes_log2) < E && lanes_log2 < 5) ++lanes_log2;
  const int L = 1 << lanes_log2;
  const int vpl = (E + L - 1) / L;
  const bool vec4 = (L == 32) && (E % 128 == 0);
  if (vec4) {
    switch (vpl) {
      case 4: return launch_route_t<4, true>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
      case 8: return launch_route_t<8, true>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
      case 16: return launch_route_t<16, true>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
      case 32: return launch_route_t<32, true>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
      default: break;
    }
  }
  if (vpl <= 1) return launch_route_t<1, false>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
  if (vpl <= 2) return launch_route_t<2, false>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
  if (vpl <= 4) return launch_route_t<4, false>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
  if (vpl <= 8) return launch_route_t<8, false>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
  if (vpl <= 16) return launch_route_t<16, false>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
  return launch_route_t<32, false>(logits, T, E, k, lanes_log2, renorm, idx, w, sms, s);
}

}  // namespace ep

namespace ep {

cudaError_t launch_route_count(const RouteCountArgs& r, cudaStream_t s) {
  int lanes_log2 = 0;
  while ((1 << lanes_log2) < r.E && lanes_log2 < 5) ++lanes_log2;
  const int L = 1 << lanes_log2;
  const int vpl = (r.E + L - 1) / L;
  const bool vec4 = (L == 32) && (r.E % 128 == 0);
  if (vec4) {
    switch (vpl) {
      case 4: return launch_route_count_t<4, true>(r, lanes_log2, s);
      case 8: return launch_route_count_t<8, true>(r, lanes_log2, s);
      case 16: return launch_route_count_t<16, true>(r, lanes_log2, s);
      case 32: return launch_route_count_t<32, true>(r, lanes_log2, s);
      default: break;
    }
  }
  if (vpl <= 1) return launch_route_count_t<1, false>(r, lanes_log2, s);
  if (vpl <= 2) return launch_route_count_t<2, false>(r, lanes_log2, s);
  if (vpl <= 4) return launch_route_count_t<4, false>(r, lanes_log2, s);
  if (vpl <= 8) return launch_route_count_t<8, false>(r, lanes_log2, s);
  if (vpl <= 16) return launch_route_count_t<16, false>(r, lanes_log2, s);
  return launch_route_count_t<32, false>(r, lanes_log2, s);
}

}  // namespace ep

namespace ep {

bool small_batch(int T, int E, int tile) {
  return T > 0 && T <= 32 * kClusterTiles && E <= kClusterExperts && tile == 32;
}

cudaError_t launch_route_layout_small(const RouteCountArgs& r, const DispatchArgs& a, cudaStream_t s) {
  if (!small_batch(r.T, r.E, r.tile)) return cudaErrorNotSupported;
  int lanes_log2 = 0;
  while ((1 << lanes_log2) < r.E && lanes_log2 < 5) ++lanes_log2;
  const int L = 1 << lanes_log2;
  const int vpl = (r.E + L - 1) / L;  // <= 8 for E <= 256
  const bool vec4 = (L == 32) && (r.E % 128 == 0);
  if (vec4) return vpl == 4 ? launch_route_layout_cluster_t<4, true>(r, a, lanes_log2, s)
                            : launch_route_layout_cluster_t<8, true>(r, a, lanes_log2, s);
  if (vpl <= 1) return launch_route_layout_cluster_t<1, false>(r, a, lanes_log2, s);
  if (vpl <= 2) return launch_route_layout_cluster_t<2, false>(r, a, lanes_log2, s);
  if (vpl <= 4) return launch_route_layout_cluster_t<4, false>(r, a, lanes_log2, s);
  return launch_route_layout_cluster_t<8, false>(r, a, lanes_log2, s);
}

}  // namespace ep
