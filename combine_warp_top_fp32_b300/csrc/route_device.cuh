// route_device.cuh — warp-level top-k gating with softmax weights over fp32
// logits: the per-token routing shared by the routing kernels (route.cu) and
// the fused route+layout+scatter kernel (fused.cu).
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
#pragma once

#include "ep_device.cuh"

namespace ep {
namespace routing {

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

// exp_shifted_term of both halves of v2 at once (nm2 = -m in both halves),
// with packed f32x2 operations: each is the IEEE operation of the scalar form
// on each half (p is formed negated, pn = fl(d * -log2e_hi) = -fl(d * log2e_hi)
// exactly), so the two results equal exp_shifted_term's bit for bit.
__device__ __forceinline__ uint64_t exp_shifted_term2(uint64_t v2, uint64_t nm2) {
  constexpr float kLog2eHi = 1.44269502162933349609375f;
  constexpr float kLog2eLo = 1.925963033500011e-08f;
  constexpr float kLn2 = 0.693147180559945309f;
  const uint64_t d = f32x2_add(v2, nm2);
  const uint64_t bb = f32x2_sub(d, v2);
  const uint64_t err = f32x2_add(f32x2_sub(v2, f32x2_sub(d, bb)), f32x2_sub(nm2, bb));
  const uint64_t pn = f32x2_mul(d, f32x2_splat(-kLog2eHi));
  const uint64_t c = f32x2_fma(err, f32x2_splat(kLog2eHi),
                               f32x2_fma(d, f32x2_splat(kLog2eLo), f32x2_fma(d, f32x2_splat(kLog2eHi), pn)));
  float r0, r1;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(-f32x2_lo(pn)));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(-f32x2_hi(pn)));
  const uint64_t r = f32x2_pack(__float_as_uint(r0), __float_as_uint(r1));
  return f32x2_fma(r, f32x2_mul(c, f32x2_splat(kLn2)), r);
}

// comp_add on both halves of (s, c) at once.
__device__ __forceinline__ void comp_add2(uint64_t& s, uint64_t& c, uint64_t x) {
  const uint64_t t = f32x2_add(s, x);
  const uint64_t bb = f32x2_sub(t, s);
  c = f32x2_add(c, f32x2_add(f32x2_sub(s, f32x2_sub(t, bb)), f32x2_sub(x, bb)));
  s = t;
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
// warp must call it together (warp-wide reductions). The kernels use it for
// E < 32 (several tokens per warp) and for more than 8 values per lane
// (E > 256); route_tokens_sorted covers the rest.
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
  if (L == 32) {
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

// The logits of NQ tokens (one per 32 lanes, E >= 32): lane `lane` gets
// experts 4*lane + 128*i + c (VEC4: float4 loads) or lane + 32*i. Values of
// inactive tokens and of ids >= E are 0 (their keys are cleared later).
template <int NQ, int VPL, bool VEC4>
__device__ __forceinline__ void load_logits(const float* __restrict__ logits, const int64_t (&t)[NQ],
                                            const bool (&active)[NQ], int E, int lane, float (&val)[NQ][VPL]) {
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const float* row = logits + (active[q] ? t[q] : 0) * static_cast<int64_t>(E);
    if constexpr (VEC4) {
#pragma unroll
      for (int i = 0; i < VPL / 4; ++i) {
        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
        if (active[q]) f = __ldg(reinterpret_cast<const float4*>(row + 4 * lane + 128 * i));
        val[q][4 * i + 0] = f.x;
        val[q][4 * i + 1] = f.y;
        val[q][4 * i + 2] = f.z;
        val[q][4 * i + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        val[q][i] = (active[q] && e < E) ? __ldg(row + e) : 0.f;
      }
    }
  }
}

// NQ tokens per warp at once (one token per 32 lanes, E >= 32, at most 8
// values per lane, logits already in registers; the kernels use NQ = 2 up to
// 4 values per lane, where the doubled registers still leave room for many
// warps, and NQ = 1 above): the same steps as route_token on the sorted-key
// path, with every per-token value held for all NQ tokens so that the NQ
// independent chains of reductions and exponentials interleave in one warp.
// KMAX > 0: the top-k rounds are unrolled for k <= KMAX (the round index is
// then a constant in each copy); 0: a loop. With an even number of values per
// lane the softmax denominator takes its terms two at a time in packed f32x2
// arithmetic (two interleaved compensated sums per lane, merged before the
// butterfly). On return lane j < k holds slot j of token q in e_out[q] /
// w_out[q].
template <int NQ, int VPL, bool VEC4, int KMAX>
__device__ __forceinline__ void route_tokens_sorted(const float (&val)[NQ][VPL], const bool (&active)[NQ], int E,
                                                    int k, int lane, int renorm, int (&e_out)[NQ],
                                                    float (&w_out)[NQ]) {
  uint64_t key[NQ][VPL];
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = VEC4 ? 4 * lane + 128 * (i / 4) + (i % 4) : lane + 32 * i;
      key[q][i] = (active[q] && (VEC4 || e < E)) ? make_key(val[q][i], e) : 0ull;  // 0 is below every real key
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
  auto round = [&](int r) {
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
  };
  if constexpr (KMAX > 0) {
#pragma unroll
    for (int r = 0; r < KMAX; ++r) {
      if (r >= k) break;
      round(r);
    }
  } else {
    for (int r = 0; r < k; ++r) round(r);
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
  } else if constexpr (VPL % 2 == 0) {
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const uint64_t nm2 = f32x2_splat(-l_max[q]);
      uint64_t s2 = 0ull, c2 = 0ull;
#pragma unroll
      for (int i = 0; i < VPL; i += 2) {
        uint64_t term = exp_shifted_term2(f32x2_pack(__float_as_uint(val[q][i]), __float_as_uint(val[q][i + 1])), nm2);
        // a value that is not an expert's adds +0, which leaves (s, c) as they were
        const bool ok0 = VEC4 ? active[q] : (active[q] && (lane + 32 * i) < E);
        const bool ok1 = VEC4 ? active[q] : (active[q] && (lane + 32 * (i + 1)) < E);
        term &= (ok0 ? 0x00000000ffffffffull : 0ull) | (ok1 ? 0xffffffff00000000ull : 0ull);
        comp_add2(s2, c2, term);
      }
      // the lane's two compensated sums, merged as the butterfly merges lanes
      const float sa = f32x2_lo(s2), sb = f32x2_hi(s2);
      const float tt = __fadd_rn(sa, sb);
      const float bb = __fsub_rn(tt, sa);
      const float err = __fadd_rn(__fsub_rn(sa, __fsub_rn(tt, bb)), __fsub_rn(sb, bb));
      c[q] = __fadd_rn(__fadd_rn(f32x2_lo(c2), f32x2_hi(c2)), err);
      s[q] = tt;
    }
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

// One warp routes tokens base + j for j = first + i*step + q*qstride (q < NQ,
// i = 0, 1, ...) while j < end, NQ at a time, the next NQ tokens' logits
// loaded while this NQ are routed (a warp otherwise waits a memory latency
// per step). emit(j, t, e, w) is called by lanes < k of each routed token.
template <int NQ, int VPL, bool VEC4, typename Emit>
__device__ __forceinline__ void route_warp(const float* __restrict__ logits, int64_t base, int64_t first, int64_t step,
                                           int64_t qstride, int64_t end, int E, int k, int lane, int renorm,
                                           Emit&& emit) {
  if (first >= end) return;
  int64_t j[NQ], t[NQ];
  bool act[NQ];
  float cur[NQ][VPL];
  auto locate = [&](int64_t j0, int64_t (&jj)[NQ], int64_t (&tt)[NQ], bool (&aa)[NQ]) {
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      jj[q] = j0 + q * qstride;
      aa[q] = jj[q] < end;
      tt[q] = base + jj[q];
    }
  };
  locate(first, j, t, act);
  load_logits<NQ, VPL, VEC4>(logits, t, act, E, lane, cur);
  for (int64_t j0 = first; j0 < end; j0 += step) {
    int64_t jn[NQ], tn[NQ];
    bool an[NQ];
    float nxt[NQ][VPL];
    locate(j0 + step, jn, tn, an);
    load_logits<NQ, VPL, VEC4>(logits, tn, an, E, lane, nxt);  // in flight during this step
    int e[NQ];
    float w[NQ];
    if (k <= 8)
      route_tokens_sorted<NQ, VPL, VEC4, 8>(cur, act, E, k, lane, renorm, e, w);
    else
      route_tokens_sorted<NQ, VPL, VEC4, 0>(cur, act, E, k, lane, renorm, e, w);
#pragma unroll
    for (int q = 0; q < NQ; ++q)
      if (act[q] && lane < k) emit(j[q], t[q], e[q], w[q]);
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      j[q] = jn[q];
      t[q] = tn[q];
      act[q] = an[q];
#pragma unroll
      for (int i = 0; i < VPL; ++i) cur[q][i] = nxt[q][i];
    }
  }
}

// Routes the nt tokens of the tile starting at token t0 (one L-lane group
// per token; with L = 32, two tokens per warp in flight up to 4 values per
// lane and one above, the next ones' logits loaded meanwhile), writes their
// slots and sets their bits in the tile's per-expert masks in shared memory:
// mask[e][w] bit b = token 32w+b of the tile chose e, and, when `ids` is
// given (E <= 256), ids[tl * k + j] = the expert of the tile's token tl in
// slot j. The masks must be zero on entry; the caller synchronises the CTA
// afterwards.
template <int VPL, bool VEC4>
__device__ __forceinline__ void route_tile(const float* __restrict__ logits, int64_t t0, int nt, int E, int k,
                                           int lanes_log2, int renorm, int TW, uint32_t* mask,
                                           int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                           uint8_t* ids = nullptr) {
  const int L = 1 << lanes_log2;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  auto emit = [&](int64_t tl, int64_t t, int e, float w) {
    topk_idx[t * k + lane] = e;
    topk_w[t * k + lane] = w;
    atomicOr(&mask[e * TW + static_cast<int>(tl >> 5)], 1u << (tl & 31));
    if (ids) ids[tl * k + lane] = static_cast<uint8_t>(e);
  };
  if constexpr (VPL <= 8) {
    if (L == 32) {
      constexpr int NQ = VPL <= 4 ? 2 : 1;
      route_warp<NQ, VPL, VEC4>(logits, t0, warp, NQ * nw, nw, nt, E, k, lane, renorm, emit);
      return;
    }
  }
  const int sub = lane & (L - 1);
  const int groups_per_warp = 32 >> lanes_log2;
  const int grp = lane >> lanes_log2;
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
      if (ids) ids[tl * k + sub] = static_cast<uint8_t>(e);
    }
  }
}

}  // namespace routing
}  // namespace ep
