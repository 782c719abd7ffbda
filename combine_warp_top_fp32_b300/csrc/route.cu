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
//     error carried into the exponential, summed with compensated (Neumaier /
//     TwoSum) arithmetic, so the weight stays within 1e-6 of the exact value.
#include "ep_internal.h"

namespace ep {
namespace {

// Float -> unsigned key whose unsigned order is the float order; -0 and +0
// map to the same key (they compare equal as floats).
__device__ __forceinline__ uint32_t ordered_bits(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u & 0x7fffffffu) == 0u) u = 0u;  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
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

// Neumaier compensated accumulation of x into (s, c).
__device__ __forceinline__ void comp_add(float& s, float& c, float x) {
  const float t = __fadd_rn(s, x);
  if (fabsf(s) >= fabsf(x))
    c = __fadd_rn(c, __fadd_rn(__fsub_rn(s, t), x));
  else
    c = __fadd_rn(c, __fadd_rn(__fsub_rn(x, t), s));
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

  for (int64_t tb = warp_id * groups_per_warp; tb < T; tb += n_warps * groups_per_warp) {
    const int64_t t = tb + grp;
    const bool active = t < T;
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
      for (int r = 0; r < k; ++r) {
        const uint32_t hv = static_cast<uint32_t>(key[0] >> 32);
        const uint32_t gmax = __reduce_max_sync(0xffffffffu, hv);
        const uint32_t cand = (hv == gmax) ? 0xffffffffu - static_cast<uint32_t>(key[0]) : 0xffffffffu;
        const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
        const float v = key_value(static_cast<uint64_t>(gmax) << 32);
        if (r == 0) l_max = v;
        if (sub == r) {
          my_e = static_cast<int>(win);
          my_v = v;
        }
        if (cand == win) {
#pragma unroll
          for (int i = 0; i + 1 < VPL; ++i) key[i] = key[i + 1];
          key[VPL - 1] = 0ull;  // 0 is below every real key
        }
      }
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
      if (sub < k) s = exp_shifted(my_v, l_max);
    } else {
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        bool ok;
        if constexpr (VEC4)
          ok = active;
        else
          ok = active && (sub + L * i) < E;
        if (ok) comp_add(s, c, exp_shifted(val[i], l_max));
      }
    }
    const float denom = group_comp_sum(s, c, L);

    if (active && sub < k) {
      const float num = exp_shifted(my_v, l_max);
      topk_idx[t * k + sub] = my_e;
      topk_w[t * k + sub] = __fdiv_rn(num, denom);
    }
  }
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
