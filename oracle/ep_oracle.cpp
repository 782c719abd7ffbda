// ep_oracle.cpp — the CPU oracle for MoE expert-parallel dispatch and combine.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link or
// call this file; only the tests, the package's smoke check and the bench's
// CPU-baseline leg use it. It shares no code, header, table or helper with the
// CUDA library: every conversion and every loop below is written out here.
//
// It is plain, single-threaded C++ that follows the method's steps in the
// order the pages give them:
//   1. route      softmax over the router logits, then top-k
//                 (MoE sparse-communication article, intelliparadigm.com,
//                  §2.1 "dynamic routing", the Router listing; NCCL EP article,
//                  hotelren.com, §3.4 MoELayer.forward step 1)
//   2. placement  expert e lives on rank e / (E/R)
//                 (MoE communication-wall explainer, juhe.plus, the
//                  "64 experts on 8 GPUs" EP example and the t1..t4 routing)
//   3. counts     per-expert counts, the capacity cap, then offsets as running
//                 sums of the counts (NCCL EP article §3.3, the flat sendbuff
//                 and its sendcounts; intelliparadigm §2.1 capacity factor)
//   4. layout     one contiguous block per destination, segments in rank order
//                 (ThunderEP on consumer GPUs, bjdmk.com.cn, §2.1 "aggregate
//                  by target card"; NCCL EP article §3.3)
//   5. payload    per-token dynamic int8 quantisation, one scale per token
//                 (ThunderEP §2.3 "per-token dynamic quantisation"); or the
//                 same per-token scheme with an FP8 E4M3 or a 4-bit code
//                 (ThunderEP §5.2 "lower-precision payloads"; NCCL EP article
//                 §6.3 FP8)
//   6. dequant    v = q * scale at the receiver (ThunderEP §2.3)
//   7. combine    gate-weighted sum of the k expert outputs back at the source
//                 (ThunderEP §1.3, steps 3 and 4 of the EP flow; §3.3 combine)
//
// Where the pages are silent, the plainest reading is taken and stated at the
// step. Precision: softmax weights in double, rounded once to fp32. The int8
// code and the combine are fixed in fp32 by their definition (scale =
// amax/127 in fp32, q = rint(x/scale) ties-to-even, fp32 accumulate with one
// fused multiply-add per slot), so the oracle computes them in fp32 and must
// be compiled without -ffast-math and with -ffp-contract=off.
//
// Every function returns 0 on success and a negative number on bad arguments.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

// ---- bf16 <-> fp32, written out from the bf16 format (top 16 bits of fp32) --

float bf16_bits_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

// Round-to-nearest-even from fp32 to bf16 (finite inputs; NaN kept quiet).
uint16_t float_to_bf16_bits_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x0040u);
  uint32_t lower = u & 0xffffu;
  uint32_t upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return static_cast<uint16_t>(upper);
}

// ---- FP8 E4M3, written out from the format: sign bit, 4 exponent bits with
// bias 7, 3 mantissa bits; exponent field 0 holds subnormals m * 2^-9; no
// infinities; the all-ones pattern S.1111.111 is NaN, so the largest finite
// magnitude is 1.75 * 2^8 = 448 (code 0x7e). -----------------------------------

double e4m3_magnitude(int code7) {  // code without its sign bit, not NaN
  const int ex = (code7 >> 3) & 15, m = code7 & 7;
  if (ex == 0) return std::ldexp(static_cast<double>(m), -9);
  return std::ldexp(1.0 + m / 8.0, ex - 7);
}

float e4m3_code_to_float(uint8_t c) {
  const double v = e4m3_magnitude(c & 0x7f);
  return static_cast<float>((c & 0x80) ? -v : v);
}

// Nearest E4M3 value of a finite float, ties to the even code (the one whose
// last mantissa bit is 0), magnitudes above 448 saturated to 448; the sign of
// zero is kept. In each binade [2^e, 2^(e+1)) the representable values are
// spaced 2^(e-3) (2^-9 below 2^-6), so |v| / spacing is exact in double and
// rounding it to the nearest integer, ties to even, is the nearest value.
uint8_t float_to_e4m3_rne_sat(float v) {
  const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  double a = std::fabs(static_cast<double>(v));
  if (a > 448.0) a = 448.0;
  if (a == 0.0) return sign;
  int e2;
  std::frexp(a, &e2);        // a = f * 2^e2 with f in [0.5, 1)
  int ex = e2 - 1;           // a in [2^ex, 2^(ex+1))
  if (ex < -6) ex = -6;      // the subnormal spacing
  const double spacing = std::ldexp(1.0, ex - 3);
  const double r = std::nearbyint(a / spacing);  // default rounding: nearest, ties to even
  const double val = r * spacing;                // exactly representable (maybe the next binade)
  if (val < std::ldexp(1.0, -6)) return static_cast<uint8_t>(sign | static_cast<int>(r));  // subnormal m
  std::frexp(val, &e2);
  const int vex = e2 - 1;
  const int m = static_cast<int>((std::ldexp(val, -vex) - 1.0) * 8.0);
  return static_cast<uint8_t>(sign | ((vex + 7) << 3) | m);
}

// "a ranks before b" for expert selection: larger logit first, and on equal
// logits the lower expert id first. Comparison is as floats, so -0 == +0.
bool ranks_before(const float* l, int a, int b) {
  if (l[a] > l[b]) return true;
  if (l[a] < l[b]) return false;
  return a < b;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// Step 1 — route (intelliparadigm §2.1 Router: probs = softmax(logits), then
// topk(probs, k); NCCL EP article §3.4: torch.topk(scores, k)).
//
// For each token t the E experts are ranked by (logit desc, expert id asc) and
// the first k are taken; slot j holds the j-th in that order, as a sorted topk
// returns them. Selection uses the logits themselves: softmax is monotone, so
// this is the same set, and it avoids ties invented by rounding probabilities.
// Reading (pages silent): ties go to the lower expert id.
//
// Weights: p_e = exp(l_e - l_max) / sum_{e'} exp(l_e' - l_max) in double,
// rounded once to fp32, and w[t,j] = p_{idx[t,j]} (softmax over all E before
// topk, as the Router listing does it). With renormalize != 0 the denominator
// runs over the k selected experts only, so the k weights sum to one.
// ---------------------------------------------------------------------------
int oracle_route(int T, int E, int k, int renormalize, const float* logits,
                 int32_t* topk_idx, float* topk_w) {
  if (T < 0 || E < 1 || k < 1 || k > E) return -1;
  std::vector<int> order(static_cast<size_t>(E));
  for (int t = 0; t < T; ++t) {
    const float* l = logits + static_cast<size_t>(t) * E;
    for (int e = 0; e < E; ++e) order[e] = e;
    std::sort(order.begin(), order.end(), [l](int a, int b) { return ranks_before(l, a, b); });
    const double l_max = static_cast<double>(l[order[0]]);
    double denom = 0.0;
    if (renormalize) {
      for (int j = 0; j < k; ++j) denom += std::exp(static_cast<double>(l[order[j]]) - l_max);
    } else {
      for (int e = 0; e < E; ++e) denom += std::exp(static_cast<double>(l[e]) - l_max);
    }
    for (int j = 0; j < k; ++j) {
      const int e = order[j];
      topk_idx[static_cast<size_t>(t) * k + j] = e;
      topk_w[static_cast<size_t>(t) * k + j] =
          static_cast<float>(std::exp(static_cast<double>(l[e]) - l_max) / denom);
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Step 2 — placement (juhe.plus EP example: 64 experts on 8 GPUs, GPU0 holds
// experts 0..7, GPU1 8..15, ..., GPU7 56..63; t2 -> expert 18 -> GPU2).
// Experts are split into R contiguous groups of G = E/R.
// ---------------------------------------------------------------------------
int oracle_expert_rank(int E, int R, int e) {
  if (R < 1 || E % R != 0 || e < 0 || e >= E) return -1;
  return e / (E / R);
}

// Per-expert capacity: ceil(cf * T * k / E), evaluated in double in that
// order; cf <= 0 means dropless (no cap). Returns the cap, or T when dropless
// (a token sends at most one copy to an expert, so no expert gets more than T).
int64_t oracle_capacity(int T, int E, int k, float capacity_factor) {
  if (!(capacity_factor > 0.0f)) return T;
  double c = std::ceil(static_cast<double>(capacity_factor) * T * k / E);
  return static_cast<int64_t>(c);
}

// ---------------------------------------------------------------------------
// Steps 3 and 4 — counts, capacity and the rank-major layout.
//
// (t, j) pairs are visited in (token, slot) order; the n-th pair that chose
// expert e gets position n within e. A pair is dropped iff its position is
// >= cap (intelliparadigm §2.1 capacity factor; the drop order and "dropped
// weight excluded" are the reading used throughout). kept_e = min(count_e,
// cap). expert_off is the exclusive running sum of kept_e over e = 0..E-1 and
// rank_off[r] = expert_off[r * G]: segment r begins where the counts of all
// earlier ranks end and an empty segment takes no room (NCCL EP article §3.3,
// the flat [rank0_data, rank1_data, ...] sendbuff). Because the experts of a
// rank are contiguous, expert-major order is rank-major order.
//
// Row expert_off[e] + pos holds the copy of (t, j): row_slot[row] = t*k + j
// and slot_row[t*k + j] = row, or -1 if dropped.
//
// Outputs: expert_counts[E] (kept), expert_raw[E] (before the cap),
// expert_off[E+1], rank_off[R+1], slot_row[T*k], row_slot[N], n_dropped[1].
// row_slot must hold at least N = T*k - drops entries.
// ---------------------------------------------------------------------------
int oracle_layout(int T, int E, int k, int R, float capacity_factor, const int32_t* topk_idx,
                  int32_t* expert_counts, int32_t* expert_raw, int32_t* expert_off,
                  int32_t* rank_off, int32_t* slot_row, int32_t* row_slot, int32_t* n_dropped) {
  if (T < 0 || E < 1 || k < 1 || k > E || R < 1 || E % R != 0) return -1;
  const int64_t cap = oracle_capacity(T, E, k, capacity_factor);
  std::vector<int64_t> seen(static_cast<size_t>(E), 0);
  std::vector<int64_t> pos(static_cast<size_t>(T) * k, -1);
  for (int t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j) {
      const int e = topk_idx[static_cast<size_t>(t) * k + j];
      if (e < 0 || e >= E) return -2;
      pos[static_cast<size_t>(t) * k + j] = seen[e]++;
    }
  }
  int64_t drops = 0;
  for (int e = 0; e < E; ++e) {
    const int64_t kept = std::min(seen[e], cap);
    expert_raw[e] = static_cast<int32_t>(seen[e]);
    expert_counts[e] = static_cast<int32_t>(kept);
    drops += seen[e] - kept;
  }
  expert_off[0] = 0;
  for (int e = 0; e < E; ++e) expert_off[e + 1] = expert_off[e] + expert_counts[e];
  const int G = E / R;
  for (int r = 0; r <= R; ++r) rank_off[r] = expert_off[r * G];
  for (int t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j) {
      const size_t s = static_cast<size_t>(t) * k + j;
      const int e = topk_idx[s];
      if (pos[s] < cap) {
        const int32_t row = expert_off[e] + static_cast<int32_t>(pos[s]);
        slot_row[s] = row;
        row_slot[row] = static_cast<int32_t>(s);
      } else {
        slot_row[s] = -1;
      }
    }
  }
  *n_dropped = static_cast<int32_t>(drops);
  return 0;
}

// ---------------------------------------------------------------------------
// Step 5 — per-token dynamic int8 code of one row (ThunderEP §2.3: every token
// gets its own scale; per-tensor scaling loses much more accuracy).
//   a     = max_h |x_h|               (exact: a max of floats)
//   scale = a / 127.0f                (fp32 IEEE division, nearest-even)
//   q_h   = clamp(rint(x_h / scale), -127, 127), fp32 division, ties-to-even
// Reading (pages silent): a == 0 gives scale 0 and q 0, avoiding 0/0;
// subnormals are kept; the clamp means -128 never appears.
// ---------------------------------------------------------------------------
int oracle_quantize_row(int H, const uint16_t* x_row, int8_t* q_row, float* scale_out) {
  if (H < 0) return -1;
  float a = 0.0f;
  for (int h = 0; h < H; ++h) {
    const float v = std::fabs(bf16_bits_to_float(x_row[h]));
    if (v > a) a = v;
  }
  const float scale = a / 127.0f;
  for (int h = 0; h < H; ++h) {
    if (scale == 0.0f) {
      q_row[h] = 0;
      continue;
    }
    float r = std::rint(bf16_bits_to_float(x_row[h]) / scale);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    q_row[h] = static_cast<int8_t>(r);
  }
  *scale_out = scale;
  return 0;
}

// Expert-side int8 return path: the same per-row code for n rows of width H.
int oracle_quantize_rows(int n, int H, const uint16_t* in, int8_t* q, float* scales) {
  if (n < 0 || H < 0) return -1;
  for (int i = 0; i < n; ++i)
    oracle_quantize_row(H, in + static_cast<size_t>(i) * H, q + static_cast<size_t>(i) * H, &scales[i]);
  return 0;
}

// ---------------------------------------------------------------------------
// Step 5, FP8 variant — the same per-token scheme with an E4M3 code (ThunderEP
// §5.2 lists FP8 among the lower-precision payloads; the NCCL EP article, §6.3,
// uses FP8 for the exchanged data while routing scores stay in high precision).
//   a     = max_h |x_h|
//   scale = a / 448.0f                (448 = largest E4M3 magnitude; fp32 IEEE)
//   q_h   = E4M3 nearest-even of fl(x_h / scale), saturated to +-448
// Reading (pages silent): the scale maps the row's largest magnitude to the
// largest finite code, as the int8 code maps it to 127; a == 0 codes every
// element as +0 with scale 0.
// ---------------------------------------------------------------------------
int oracle_quantize_row_fp8(int H, const uint16_t* x_row, uint8_t* q_row, float* scale_out) {
  if (H < 0) return -1;
  float a = 0.0f;
  for (int h = 0; h < H; ++h) {
    const float v = std::fabs(bf16_bits_to_float(x_row[h]));
    if (v > a) a = v;
  }
  const float scale = a / 448.0f;
  for (int h = 0; h < H; ++h)
    q_row[h] = scale == 0.0f ? 0 : float_to_e4m3_rne_sat(bf16_bits_to_float(x_row[h]) / scale);
  *scale_out = scale;
  return 0;
}

int oracle_quantize_rows_fp8(int n, int H, const uint16_t* in, uint8_t* q, float* scales) {
  if (n < 0 || H < 0) return -1;
  for (int i = 0; i < n; ++i)
    oracle_quantize_row_fp8(H, in + static_cast<size_t>(i) * H, q + static_cast<size_t>(i) * H, &scales[i]);
  return 0;
}

// ---------------------------------------------------------------------------
// Step 5, int4 variant — the per-token scheme with 4-bit codes (ThunderEP
// §5.2 names 4-bit payloads as the next, more aggressive compression).
//   a     = max_h |x_h|
//   scale = a / 7.0f                  (fp32 IEEE division)
//   q_h   = clamp(rint(x_h / scale), -7, 7), fp32 division, ties to even
//   byte i of the row = (q_{2i} & 0xF) | ((q_{2i+1} & 0xF) << 4)
// Reading (pages silent): the int8 scheme with 7 in place of 127, so that -8
// is never used and the code is symmetric; two's-complement nibbles, the
// lower-indexed element in the low nibble; a == 0 gives scale 0 and 0 bytes.
// ---------------------------------------------------------------------------
int oracle_quantize_row_int4(int H, const uint16_t* x_row, uint8_t* q_row, float* scale_out) {
  if (H < 0 || H % 2 != 0) return -1;
  float a = 0.0f;
  for (int h = 0; h < H; ++h) {
    const float v = std::fabs(bf16_bits_to_float(x_row[h]));
    if (v > a) a = v;
  }
  const float scale = a / 7.0f;
  for (int i = 0; i < H / 2; ++i) {
    int q[2] = {0, 0};
    for (int j = 0; j < 2 && scale != 0.0f; ++j) {
      float r = std::rint(bf16_bits_to_float(x_row[2 * i + j]) / scale);
      if (r > 7.0f) r = 7.0f;
      if (r < -7.0f) r = -7.0f;
      q[j] = static_cast<int>(r);
    }
    q_row[i] = static_cast<uint8_t>((q[0] & 0xF) | ((q[1] & 0xF) << 4));
  }
  *scale_out = scale;
  return 0;
}

int oracle_quantize_rows_int4(int n, int H, const uint16_t* in, uint8_t* q, float* scales) {
  if (n < 0 || H < 0 || H % 2 != 0) return -1;
  for (int i = 0; i < n; ++i)
    oracle_quantize_row_int4(H, in + static_cast<size_t>(i) * H, q + static_cast<size_t>(i) * (H / 2), &scales[i]);
  return 0;
}

// Element h of an int4 row: its nibble, sign-extended, times the scale.
float oracle_dequant_int4(const uint8_t* q_row, int h, float scale) {
  const int nib = (q_row[h / 2] >> (4 * (h % 2))) & 0xF;
  return static_cast<float>(nib >= 8 ? nib - 16 : nib) * scale;
}

// E4M3 helpers exported for the tests' pins of the oracle's conversions.
uint8_t oracle_float_to_e4m3(float v) { return float_to_e4m3_rne_sat(v); }
float oracle_e4m3_to_float(uint8_t c) { return e4m3_code_to_float(c); }

// ---------------------------------------------------------------------------
// Step 4+5 — the dispatch payload (ThunderEP §2.1 "aggregate by target card"
// then §2.3 compression): every kept row is a copy of its token's x row,
// bf16 bytes unchanged (mode 0), that token's int8 code and scale (mode 1),
// its FP8 E4M3 code and scale (mode 2), or its packed int4 code and scale
// (mode 3). Rows are written from row_slot, N rows. payload is [N, H] uint16
// (bf16), int8 or uint8 (E4M3 codes), or [N, H/2] uint8 (int4 pairs); scales
// is [N] (modes 1 to 3).
// ---------------------------------------------------------------------------
int oracle_payload(int T, int H, int k, int N, int mode, const uint16_t* x,
                   const int32_t* row_slot, void* payload, float* scales) {
  if (T < 0 || H < 0 || k < 1 || N < 0 || mode < 0 || mode > 3) return -1;
  std::vector<int8_t> q(static_cast<size_t>(H));
  for (int row = 0; row < N; ++row) {
    const int32_t s = row_slot[row];
    if (s < 0 || s >= T * k) return -2;
    const int t = s / k;
    const uint16_t* xr = x + static_cast<size_t>(t) * H;
    if (mode == 3) {
      float scale;
      oracle_quantize_row_int4(H, xr, static_cast<uint8_t*>(payload) + static_cast<size_t>(row) * (H / 2), &scale);
      scales[row] = scale;
    } else if (mode == 2) {
      float scale;
      oracle_quantize_row_fp8(H, xr, static_cast<uint8_t*>(payload) + static_cast<size_t>(row) * H, &scale);
      scales[row] = scale;
    } else if (mode == 1) {
      float scale;
      oracle_quantize_row(H, xr, q.data(), &scale);
      std::memcpy(static_cast<int8_t*>(payload) + static_cast<size_t>(row) * H, q.data(),
                  static_cast<size_t>(H));
      scales[row] = scale;
    } else {
      std::memcpy(static_cast<uint16_t*>(payload) + static_cast<size_t>(row) * H, xr,
                  static_cast<size_t>(H) * sizeof(uint16_t));
    }
  }
  return 0;
}

// Step 6 — dequantised value of one element: one fp32 multiply (ThunderEP §2.3,
// "decompress back at the target card").
float oracle_dequant(int8_t q, float scale) { return static_cast<float>(q) * scale; }
float oracle_dequant_fp8(uint8_t q, float scale) { return e4m3_code_to_float(q) * scale; }

// ---------------------------------------------------------------------------
// Step 7 — combine (ThunderEP §1.3: the expert's card sends results back and
// the source card takes the weighted sum; §3.3 combine(outputs)).
//   acc = 0; for j = 0..k-1 in slot order: skip if slot_row == -1 (dropped:
//   its weight is excluded, not redistributed); v = value of row
//   slot_row[t,j] (bf16 widened, or q * scale); acc = fmaf(w[t,j], v, acc).
//   y[t,h] = bf16 round-to-nearest-even of acc.
// Reading: fused multiply-add per slot (the pages fix no order or rounding;
// fixed slot order is what makes the result reproducible).
// out_mode 0: expert_out is [*, H] bf16 bits; 1: int8 codes with
// out_scales[*]; 2: E4M3 codes with out_scales[*]; 3: [*, H/2] packed int4
// codes with out_scales[*].
// ---------------------------------------------------------------------------
int oracle_combine(int T, int H, int k, int out_mode, const void* expert_out,
                   const float* out_scales, const int32_t* slot_row, const float* topk_w,
                   uint16_t* y) {
  if (T < 0 || H < 0 || k < 1 || out_mode < 0 || out_mode > 3) return -1;
  for (int t = 0; t < T; ++t) {
    for (int h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (int j = 0; j < k; ++j) {
        const int32_t row = slot_row[static_cast<size_t>(t) * k + j];
        if (row < 0) continue;
        const size_t at = static_cast<size_t>(row) * H + h;
        float v;
        if (out_mode == 3)
          v = oracle_dequant_int4(static_cast<const uint8_t*>(expert_out) + static_cast<size_t>(row) * (H / 2), h,
                                  out_scales[row]);
        else if (out_mode == 2)
          v = oracle_dequant_fp8(static_cast<const uint8_t*>(expert_out)[at], out_scales[row]);
        else if (out_mode == 1)
          v = oracle_dequant(static_cast<const int8_t*>(expert_out)[at], out_scales[row]);
        else
          v = bf16_bits_to_float(static_cast<const uint16_t*>(expert_out)[at]);
        acc = std::fmaf(topk_w[static_cast<size_t>(t) * k + j], v, acc);
      }
      y[static_cast<size_t>(t) * H + h] = float_to_bf16_bits_rne(acc);
    }
  }
  return 0;
}

// Combine for a subset of tokens only (sampled parity at full size): y rows
// are written in the order of `tokens`.
int oracle_combine_tokens(int n_tokens, const int32_t* tokens, int H, int k, int out_mode,
                          const void* expert_out, const float* out_scales,
                          const int32_t* slot_row, const float* topk_w, uint16_t* y) {
  for (int i = 0; i < n_tokens; ++i) {
    const int t = tokens[i];
    if (t < 0) return -1;
    for (int h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (int j = 0; j < k; ++j) {
        const int32_t row = slot_row[static_cast<size_t>(t) * k + j];
        if (row < 0) continue;
        const size_t at = static_cast<size_t>(row) * H + h;
        float v;
        if (out_mode == 3)
          v = oracle_dequant_int4(static_cast<const uint8_t*>(expert_out) + static_cast<size_t>(row) * (H / 2), h,
                                  out_scales[row]);
        else if (out_mode == 2)
          v = oracle_dequant_fp8(static_cast<const uint8_t*>(expert_out)[at], out_scales[row]);
        else if (out_mode == 1)
          v = oracle_dequant(static_cast<const int8_t*>(expert_out)[at], out_scales[row]);
        else
          v = bf16_bits_to_float(static_cast<const uint16_t*>(expert_out)[at]);
        acc = std::fmaf(topk_w[static_cast<size_t>(t) * k + j], v, acc);
      }
      y[static_cast<size_t>(i) * H + h] = float_to_bf16_bits_rne(acc);
    }
  }
  return 0;
}

// Load statistic (intelliparadigm §2.1: watch how unevenly experts are called;
// the coefficient of variation should stay below 0.3): population standard
// deviation of the per-expert counts over their mean, in double.
double oracle_count_cv(int E, const int32_t* counts) {
  if (E < 1) return 0.0;
  double mean = 0.0;
  for (int e = 0; e < E; ++e) mean += counts[e];
  mean /= E;
  if (mean == 0.0) return 0.0;
  double var = 0.0;
  for (int e = 0; e < E; ++e) var += (counts[e] - mean) * (counts[e] - mean);
  var /= E;
  return std::sqrt(var) / mean;
}

// bf16 helpers exported for the tests' own pins of the oracle's conversions.
float oracle_bf16_to_float(uint16_t b) { return bf16_bits_to_float(b); }
uint16_t oracle_float_to_bf16(float f) { return float_to_bf16_bits_rne(f); }

}  // extern "C"
