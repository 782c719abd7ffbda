"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test ties one oracle step to a worked example printed on the pages, a
closed form, an invariant, brute force on tiny inputs, or an independent
library routine (numpy's stable argsort, scipy's softmax, Python's
ties-to-even ``round``, torch's bf16 conversion). None of them needs a GPU.
"""
import itertools
import json
import math
from pathlib import Path

import numpy as np
import pytest
import scipy.special
import torch

GOLDEN = Path(__file__).resolve().parent / "golden"


def _load(name):
    return json.loads((GOLDEN / name).read_text())


def _f32_bits_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Exact bf16 bits of fp32 values that are representable in bf16."""
    a = np.asarray(a, np.float32)
    bits = a.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value is not exact in bf16"
    return (bits >> 16).astype(np.uint16)


def _bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# step 2: placement — the juhe.plus worked example
# --------------------------------------------------------------------------
def test_expert_rank_worked_example(orc):
    g = _load("ep_example_64x8.json")
    E, R = g["E"], g["R"]
    for gpu, (lo, hi) in g["gpu_expert_ranges"].items():
        for e in range(lo, hi + 1):
            assert orc.expert_rank(E, R, e) == int(gpu)
    for tok in g["tokens"]:
        assert orc.expert_rank(E, R, tok["expert"]) == tok["gpu"], tok["name"]


def test_layout_places_worked_example_tokens_in_their_rank_block(orc):
    g = _load("ep_example_64x8.json")
    E, R = g["E"], g["R"]
    idx = np.array([[t["expert"]] for t in g["tokens"]], np.int32)  # k = 1
    lay = orc.layout(idx, E, R)
    roff = lay["rank_off"]
    for t, tok in enumerate(g["tokens"]):
        row = lay["slot_row"][t]
        gpu = tok["gpu"]
        assert roff[gpu] <= row < roff[gpu + 1], tok["name"]


def test_expert_rank_rejects_non_divisible(orc):
    with pytest.raises(ValueError):
        orc.expert_rank(10, 4, 1)


# --------------------------------------------------------------------------
# steps 3-4: flat send buffer — the NCCL EP article's sendcounts example
# --------------------------------------------------------------------------
def test_flat_sendbuff_offsets_follow_sendcounts(orc):
    g = _load("ncclep_sendcounts.json")
    counts_bytes = g["sendcounts_bytes"]
    R = len(counts_bytes)
    H = 512
    row_bytes = H * 2  # one bf16 row
    counts_rows = [c // row_bytes for c in counts_bytes]
    assert all(c % row_bytes == 0 for c in counts_bytes)
    # one expert per rank, k = 1; tokens interleaved so no rank's tokens are adjacent
    dest = []
    remaining = list(counts_rows)
    while any(remaining):
        for r in range(R):
            if remaining[r]:
                dest.append(r)
                remaining[r] -= 1
    idx = np.array(dest, np.int32).reshape(-1, 1)
    lay = orc.layout(idx, E=R, R=R)
    roff = lay["rank_off"]
    assert roff[0] == 0
    assert [int(roff[r + 1] - roff[r]) for r in range(R)] == counts_rows
    # the buffer holds exactly the sum of the counts; empty segments take no room
    assert int(roff[R]) * row_bytes == sum(counts_bytes)
    for r in range(R):
        if counts_rows[r] == 0:
            assert roff[r] == roff[r + 1]


# --------------------------------------------------------------------------
# all-to-all volume — the juhe.plus formula and its worked example
# --------------------------------------------------------------------------
def test_a2a_volume_worked_example(orc):
    g = _load("a2a_volume.json")
    from combine_warp_top_fp32_b300 import workloads

    w = workloads.WORKLOADS["large"]
    assert (w.T, w.H, w.k) == (g["T"], g["H"], g["k"])
    # dropless: every (token, slot) pair becomes one row — checked through the
    # oracle's layout on a slice of routed tokens, then scaled by T
    rng = np.random.default_rng(0)
    T_small = 64
    idx = np.stack([rng.permutation(w.E)[: w.k] for _ in range(T_small)]).astype(np.int32)
    lay = orc.layout(idx, w.E, w.R, 0.0)
    assert lay["N"] == T_small * w.k and lay["n_dropped"] == 0
    rows = lay["N"] // T_small * w.T
    one_way = rows * w.H * g["b"]
    assert one_way == 17_179_869_184
    assert round(one_way / 1e9, 1) == g["one_direction_gb"]
    assert round(2 * one_way / 1e9, 1) == g["both_directions_gb"]
    assert 100.0 * g["active_experts"] / g["total_experts"] == g["active_percent"]
    assert w.max_rows() == rows


# --------------------------------------------------------------------------
# step 1: route — brute force, ties, independent library routines
# --------------------------------------------------------------------------
def _beats(l, a, b):
    return l[a] > l[b] or (l[a] == l[b] and a < b)


@pytest.mark.parametrize("E,k", [(3, 1), (5, 2), (6, 3), (8, 2), (8, 8), (7, 4)])
@pytest.mark.parametrize("ties", [False, True])
def test_route_selection_brute_force(orc, E, k, ties):
    rng = np.random.default_rng(E * 100 + k + (7 if ties else 0))
    T = 40
    if ties:
        logits = rng.integers(0, 3, size=(T, E)).astype(np.float32)
        logits[rng.random((T, E)) < 0.2] = -0.0  # -0 and +0 must tie
    else:
        logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, _ = orc.route(logits, k)
    for t in range(T):
        l = logits[t]
        winners = [S for S in itertools.combinations(range(E), k)
                   if all(_beats(l, a, b) for a in S for b in range(E) if b not in S)]
        assert len(winners) == 1
        S = winners[0]
        assert sorted(idx[t].tolist()) == sorted(S)
        # slots in rank order
        for j in range(k - 1):
            assert _beats(l, idx[t, j], idx[t, j + 1])


def test_route_matches_stable_argsort(orc):
    rng = np.random.default_rng(3)
    for E, k in [(64, 6), (128, 8), (256, 8), (8, 2)]:
        logits = rng.standard_normal((200, E)).astype(np.float32)
        logits[:20] = np.round(logits[:20])  # plenty of exact ties
        idx, _ = orc.route(logits, k)
        ref = np.argsort(-logits, axis=1, kind="stable")[:, :k]
        np.testing.assert_array_equal(idx, ref)


def test_route_weights_against_scipy_softmax(orc):
    rng = np.random.default_rng(4)
    for E, k in [(8, 2), (64, 6), (128, 8), (256, 8)]:
        logits = (rng.standard_normal((100, E)) + rng.standard_normal(E)).astype(np.float32)
        idx, w = orc.route(logits, k, renormalize=False)
        p = scipy.special.softmax(logits.astype(np.float64), axis=1)
        ref = np.take_along_axis(p, idx.astype(np.int64), axis=1)
        np.testing.assert_allclose(w, ref.astype(np.float32), rtol=2 ** -23, atol=0)
        idx2, w2 = orc.route(logits, k, renormalize=True)
        np.testing.assert_array_equal(idx, idx2)
        ref2 = ref / ref.sum(axis=1, keepdims=True)
        np.testing.assert_allclose(w2, ref2.astype(np.float32), rtol=2 ** -23, atol=0)
        assert np.all(np.abs(w2.astype(np.float64).sum(axis=1) - 1.0) <= k * 2 ** -24)


def test_route_full_softmax_sums_to_one_when_k_equals_E(orc):
    rng = np.random.default_rng(5)
    logits = (3 * rng.standard_normal((50, 16))).astype(np.float32)
    _, w = orc.route(logits, 16, renormalize=False)
    assert np.all(np.abs(w.astype(np.float64).sum(axis=1) - 1.0) <= 16 * 2 ** -24)


def test_route_two_experts_is_a_logistic(orc):
    a = np.linspace(-6, 6, 25, dtype=np.float32)
    b = np.float32(0.75)
    logits = np.stack([a, np.full_like(a, b)], axis=1)
    idx, w = orc.route(logits, 1, renormalize=False)
    for t in range(len(a)):
        top = 0 if (a[t] > b or a[t] == b) else 1
        other = 1 - top
        d = float(logits[t, other]) - float(logits[t, top])
        assert idx[t, 0] == top
        assert w[t, 0] == np.float32(1.0 / (1.0 + math.exp(d)))


def test_route_renormalized_k1_weight_is_one(orc):
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((30, 9)).astype(np.float32)
    _, w = orc.route(logits, 1, renormalize=True)
    assert np.all(w == 1.0)


# --------------------------------------------------------------------------
# steps 3-4: counts, capacity, layout — invariants on tiny and mid inputs
# --------------------------------------------------------------------------
def test_capacity_formula(orc):
    from combine_warp_top_fp32_b300 import workloads

    w = workloads.WORKLOADS["capacity"]
    assert orc.capacity(w.T, w.E, w.k, w.capacity_factor) == 1280 == w.capacity()
    assert orc.capacity(10, 3, 1, 1.0) == 4  # ceil(10/3)
    assert orc.capacity(12, 3, 1, 1.0) == 4  # exact, no rounding up
    assert orc.capacity(100, 4, 2, 0.0) == 100  # dropless


def _random_idx(rng, T, E, k, skew=0.0):
    p = np.exp(skew * rng.standard_normal(E))
    p /= p.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


def _check_layout_invariants(idx, E, R, cf, lay, cap):
    T, k = idx.shape
    counts, raw, eoff, roff = lay["expert_counts"], lay["expert_raw"], lay["expert_off"], lay["rank_off"]
    slot_row, row_slot, N = lay["slot_row"], lay["row_slot"], lay["N"]
    # raw counts are a histogram of idx
    np.testing.assert_array_equal(raw, np.bincount(idx.ravel(), minlength=E))
    # kept = min(raw, cap); sum kept = T*k - drops
    np.testing.assert_array_equal(counts, np.minimum(raw, cap))
    assert int(counts.sum()) == T * k - lay["n_dropped"] == N
    # offsets are running sums starting at 0; rank r starts at its first expert
    assert eoff[0] == 0 and np.all(np.diff(eoff) == counts)
    G = E // R
    np.testing.assert_array_equal(roff, eoff[::G])
    assert roff[R] == N
    # slot_row and row_slot are inverse; kept rows are a permutation of 0..N-1
    kept = np.flatnonzero(slot_row >= 0)
    assert len(kept) == N
    np.testing.assert_array_equal(np.sort(slot_row[kept]), np.arange(N))
    np.testing.assert_array_equal(row_slot[slot_row[kept]], kept)
    # rows ordered by (expert, token); each row lies in its expert's segment
    tok = row_slot // k
    exp = idx.ravel()[row_slot]
    key = exp.astype(np.int64) * (T + 1) + tok
    assert np.all(np.diff(key) > 0)
    for row in range(N):
        e = exp[row]
        assert eoff[e] <= row < eoff[e + 1]
    # drops are exactly the pairs past the first `cap` tokens of their expert
    for e in range(E):
        toks = [t for t in range(T) if e in idx[t]]
        for n, t in enumerate(toks):
            j = int(np.flatnonzero(idx[t] == e)[0])
            assert (slot_row[t * k + j] >= 0) == (n < cap)


@pytest.mark.parametrize("T,E,k,R,cf,skew", [
    (40, 6, 2, 3, 0.0, 0.0),
    (40, 6, 2, 3, 1.0, 1.5),
    (64, 8, 3, 2, 0.75, 1.0),
    (100, 16, 4, 4, 1.25, 2.0),
    (1, 4, 4, 2, 0.0, 0.0),
    (0, 4, 2, 2, 0.0, 0.0),
])
def test_layout_invariants(orc, T, E, k, R, cf, skew):
    rng = np.random.default_rng(T + E + k)
    idx = _random_idx(rng, T, E, k, skew) if T else np.zeros((0, k), np.int32)
    lay = orc.layout(idx, E, R, cf)
    cap = orc.capacity(T, E, k, cf)
    _check_layout_invariants(idx, E, R, cf, lay, cap)
    if cf > 0 and skew > 0 and T >= 40:
        assert lay["n_dropped"] > 0  # the skewed cases do exercise the cap


def test_layout_rejects_bad_expert_id(orc):
    idx = np.array([[0, 9]], np.int32)
    with pytest.raises(ValueError):
        orc.layout(idx, 8, 2)


# --------------------------------------------------------------------------
# step 5-6: int8 code — ties-to-even rows, error bound, special cases
# --------------------------------------------------------------------------
def test_quant_rows_with_exact_scales():
    import oracle

    orc = oracle.Oracle()
    rows = _load("quant_ties.json")["rows"]
    x = np.array(rows, np.float32)
    q, s = orc.quantize_rows(_f32_bits_to_bf16_bits(x))
    for i, row in enumerate(rows):
        amax = max(abs(v) for v in row)
        scale = amax / 127.0  # 1, 2 or 0: exact
        assert s[i] == scale
        for h, v in enumerate(row):
            want = 0 if scale == 0 else max(-127, min(127, round(v / scale)))  # round(): ties to even
            assert q[i, h] == want, (i, h, v)


def test_quant_error_bound_and_extremes(orc):
    rng = np.random.default_rng(8)
    H = 2048
    z = rng.standard_normal((4, 64, H))
    t3 = z[0] / np.sqrt((z[1] ** 2 + z[2] ** 2 + z[3] ** 2) / 3)
    x = np.concatenate([rng.standard_normal((64, H)), 0.5 * t3, 1e-30 * rng.standard_normal((4, H))])
    xb = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # rows of bf16 subnormals (bits 0x0001..0x007f, either sign): the scale is
    # then an fp32 subnormal, the coarsest case for x/scale
    sub = rng.integers(1, 0x80, size=(3, H)).astype(np.uint16) | (rng.integers(0, 2, size=(3, H)) << 15).astype(np.uint16)
    sub[0, 0] = 0x0001  # a row whose largest magnitude is the smallest subnormal
    sub[0, 1:] = 0x8001
    xb = np.concatenate([xb, sub])
    xf = _bf16_bits_to_f32(xb)
    q, s = orc.quantize_rows(xb)
    assert q.min() >= -127
    for i in range(xb.shape[0]):
        amax = np.max(np.abs(xf[i]))
        assert s[i] == np.float32(amax) / np.float32(127.0)
        deq = q[i].astype(np.float32) * s[i]
        err = np.abs(xf[i].astype(np.float64) - deq.astype(np.float64))
        bound = s[i] / 2.0 * (1 + 1e-6) + np.spacing(np.abs(deq)).astype(np.float64)
        assert np.all(err <= bound), i
        # the element of largest magnitude codes to +-127
        at = int(np.argmax(np.abs(xf[i])))
        assert abs(int(q[i, at])) == 127


def test_dequant_is_one_multiply(orc):
    assert orc.dequant(-3, 0.5) == -1.5
    assert orc.dequant(127, 1.0) == 127.0
    s = np.float32(0.0123)
    assert orc.dequant(77, float(s)) == np.float32(77) * s


# --------------------------------------------------------------------------
# bf16 conversion of the oracle against torch's
# --------------------------------------------------------------------------
def test_bf16_round_to_nearest_even_against_torch(orc):
    rng = np.random.default_rng(9)
    vals = np.concatenate([
        rng.standard_normal(2000).astype(np.float32),
        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 2 ** -130, 3e38, 0.0, -0.0], np.float32),
    ])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.float_to_bf16(float(v)) for v in vals], np.uint16)
    np.testing.assert_array_equal(got, ref)
    for b in ref[:50]:
        assert orc.bf16_to_float(int(b)) == _bf16_bits_to_f32(np.array([b]))[0]


# --------------------------------------------------------------------------
# step 7: combine — identity round trip, k=1, all dropped, exact small sums
# --------------------------------------------------------------------------
def _bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v.astype(np.float32))
    e = np.floor(np.log2(np.maximum(a, 2 ** -126)))
    return np.power(2.0, e - 7)


@pytest.mark.parametrize("int8", [False, True])
def test_identity_experts_round_trip(orc, int8):
    rng = np.random.default_rng(10)
    T, H, E, k, R = 96, 256, 16, 4, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    xf = _bf16_bits_to_f32(xb)
    idx, w = orc.route(logits, k, renormalize=True)
    lay = orc.layout(idx, E, R, 0.0)
    pl, sc = orc.payload(xb, lay["row_slot"], k, int8)
    y = orc.combine(pl, sc, lay["slot_row"], w, T, k)
    yf = _bf16_bits_to_f32(y)
    if not int8:
        # sum_j w_j * x = x (1 +- k*2^-24); one bf16 rounding at the end
        assert np.all(np.abs(yf - xf) <= _bf16_ulp(xf))
    else:
        s_tok = np.zeros(T, np.float32)
        s_tok[lay["row_slot"] // k] = sc
        bound = (s_tok / 2.0)[:, None] * 1.0001 + _bf16_ulp(xf) + 1e-30
        assert np.all(np.abs(yf - xf) <= bound)


def test_combine_k1_renormalized_is_exact_copy(orc):
    rng = np.random.default_rng(11)
    T, H, E = 50, 64, 8
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xb = torch.randn(T, H).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    idx, w = orc.route(logits, 1, renormalize=True)
    lay = orc.layout(idx, E, 2, 0.0)
    pl, _ = orc.payload(xb, lay["row_slot"], 1, False)
    y = orc.combine(pl, None, lay["slot_row"], w, T, 1)
    np.testing.assert_array_equal(y, xb)


def test_combine_all_dropped_gives_zero(orc):
    T, H, k = 3, 16, 2
    eo = np.full((4, H), 0x3F80, np.uint16)  # 1.0
    slot_row = np.full(T * k, -1, np.int32)
    w = np.full(T * k, 0.5, np.float32)
    y = orc.combine(eo, None, slot_row, w, T, k)
    assert np.all(y == 0)


def test_combine_exact_small_sums(orc):
    # y = 0.5 * 2 + 0.25 * 4 = 2 exactly; dropped slot ignored; int8 rows dequantised first
    H = 8
    eo = np.zeros((3, H), np.uint16)
    eo[0] = _f32_bits_to_bf16_bits(np.full(H, 2.0, np.float32))
    eo[1] = _f32_bits_to_bf16_bits(np.full(H, 4.0, np.float32))
    eo[2] = _f32_bits_to_bf16_bits(np.full(H, 1000.0, np.float32))
    y = orc.combine(eo, None, np.array([0, 1, -1], np.int32), np.array([0.5, 0.25, 0.25], np.float32), 1, 3)
    assert np.all(_bf16_bits_to_f32(y) == 2.0)
    q = np.array([[10] * H, [-4] * H], np.int8)
    y = orc.combine(q, np.array([0.5, 2.0], np.float32), np.array([1, 0], np.int32),
                    np.array([0.25, 1.0], np.float32), 1, 2)
    assert np.all(_bf16_bits_to_f32(y) == 0.25 * (-8.0) + 1.0 * 5.0)


def test_combine_follows_slot_order(orc):
    # slot order is part of the definition: 2^24 + 1 rounds back to 2^24 in
    # fp32 (ties to even), so 2^24, 1, -2^24 in slot order sum to 0, while any
    # order that adds -2^24 before 1 would give 1
    H = 8
    eo = np.stack([_f32_bits_to_bf16_bits(np.full(H, v, np.float32)) for v in (2.0**24, 1.0, -(2.0**24))])
    y = orc.combine(eo, None, np.array([0, 1, 2], np.int32), np.ones(3, np.float32), 1, 3)
    assert np.all(_bf16_bits_to_f32(y) == 0.0)
    y = orc.combine(eo, None, np.array([2, 1, 0], np.int32), np.ones(3, np.float32), 1, 3)
    assert np.all(_bf16_bits_to_f32(y) == 1.0)


def test_combine_uses_fused_multiply_add(orc):
    # slot 0 puts acc = -P with P = fl(w1 * v1); slot 1 adds w1 * v1. With one
    # rounding per fma the result is the exact residual w1*v1 - P = 2^-27 +
    # 2^-30 (exact in bf16); a separate multiply and add would give 0.
    H = 8
    w1 = np.float32(1.0 + 2.0**-20 + 2.0**-23)
    v1 = np.float32(1.0 + 2.0**-7)
    P = np.float32(w1 * v1)
    residual = float(w1) * float(v1) - float(P)
    assert residual == 2.0**-27 + 2.0**-30
    eo = np.stack([_f32_bits_to_bf16_bits(np.full(H, -1.0, np.float32)),
                   _f32_bits_to_bf16_bits(np.full(H, v1, np.float32))])
    y = orc.combine(eo, None, np.array([0, 1], np.int32), np.array([P, w1], np.float32), 1, 2)
    assert np.all(_bf16_bits_to_f32(y) == np.float32(residual))


def test_combine_tokens_matches_full_combine(orc):
    rng = np.random.default_rng(12)
    T, H, k, N = 20, 32, 3, 50
    eo = torch.randn(N, H).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    slot_row = rng.integers(-1, N, size=T * k).astype(np.int32)
    w = rng.random(T * k).astype(np.float32)
    full = orc.combine(eo, None, slot_row, w, T, k)
    toks = np.array([19, 0, 7, 7], np.int32)
    part = orc.combine_tokens(toks, eo, None, slot_row, w, k)
    np.testing.assert_array_equal(part, full[toks])


def test_count_cv_closed_forms(orc):
    assert orc.count_cv(np.array([5, 5, 5, 5], np.int32)) == 0.0
    assert orc.count_cv(np.array([0, 2], np.int32)) == 1.0
    assert abs(orc.count_cv(np.array([1, 2, 3], np.int32)) - math.sqrt(2 / 3) / 2) < 1e-15


# ----------------------------------------------------------------------------
# FP8 E4M3 per-token payload (ThunderEP §5.2 lower-precision payloads; NCCL EP
# article §6.3 FP8 for the exchanged data): the oracle's E4M3 conversions
# against torch's float8_e4m3fn and against brute force over all 256 codes.
# ----------------------------------------------------------------------------
_E4M3_NAN = (0x7F, 0xFF)


def _e4m3_table():
    codes = np.array([c for c in range(256) if c not in _E4M3_NAN], dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    return codes, vals


def test_e4m3_decode_matches_torch(orc):
    codes, vals = _e4m3_table()
    got = np.array([orc.e4m3_to_float(int(c)) for c in codes], dtype=np.float64)
    np.testing.assert_array_equal(got, vals)
    assert orc.e4m3_to_float(0x7E) == 448.0 and orc.e4m3_to_float(0x01) == 2.0 ** -9


def _brute_force_e4m3(v: float) -> int:
    """Nearest E4M3 code by scanning every code (ties: the code with an even
    last mantissa bit), magnitudes above 448 saturated."""
    codes, vals = _e4m3_table()
    a = min(abs(v), 448.0)
    pos = codes < 0x80
    c, x = codes[pos], vals[pos]
    d = np.abs(x - a)
    best = np.flatnonzero(d == d.min())
    if best.size > 1:
        best = best[(c[best] & 1) == 0]
    code = int(c[best[0]])
    return code | (0x80 if math.copysign(1.0, v) < 0 else 0)


def _e4m3_probe_values():
    _, vals = _e4m3_table()
    mags = np.unique(np.abs(vals))
    mids = (mags[:-1] + mags[1:]) / 2
    probes = [mags, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
              np.nextafter(mids.astype(np.float32), np.float32(1e9))]
    rng = np.random.default_rng(8)
    probes.append(np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 3000)))
    probes.append(np.array([448.0, 449.0, 463.9, 464.0, 470.0, 0.0]))
    p = np.concatenate([np.asarray(x, np.float64) for x in probes]).astype(np.float32)
    return np.concatenate([p, -p])


def test_e4m3_encode_matches_torch_and_brute_force(orc):
    v = _e4m3_probe_values()
    ours = np.array([orc.float_to_e4m3(float(x)) for x in v], dtype=np.uint8)
    in_range = np.abs(v) <= 448.0  # torch turns overflow into NaN; the oracle saturates
    theirs = torch.from_numpy(v[in_range]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours[in_range], theirs)
    for x, c in zip(v[::7], ours[::7]):
        assert c == _brute_force_e4m3(float(x)), x
    # saturation and signed zero
    assert orc.float_to_e4m3(1e30) == 0x7E and orc.float_to_e4m3(-1e30) == 0xFE
    assert orc.float_to_e4m3(-0.0) == 0x80 and orc.float_to_e4m3(0.0) == 0x00


def test_fp8_row_code_properties(orc):
    rng = np.random.default_rng(9)
    x = torch.from_numpy(rng.standard_normal((64, 512)).astype(np.float32) * 3).to(torch.bfloat16)
    x[5] = 0.0
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q, s = orc.quantize_rows(bits, fp8=True)
    xf = x.float().numpy()
    amax = np.abs(xf).max(1)
    np.testing.assert_array_equal(s, (amax / np.float32(448.0)).astype(np.float32))
    assert np.all(q[5] == 0) and s[5] == 0.0
    deq = np.array([[orc.dequant_fp8(int(c), float(sc)) for c in row] for row, sc in zip(q[:8], s[:8])])
    for r in range(8):
        if s[r] == 0:
            continue
        i = int(np.argmax(np.abs(xf[r])))
        assert q[r, i] in (0x7E, 0xFE)  # the largest magnitude takes the largest code
        # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 above 2^-6 * scale,
        # absolute error <= 2^-10 * scale below (the subnormal spacing is 2^-9)
        err = np.abs(deq[r] - xf[r])
        bound = np.maximum(np.abs(xf[r]) * 2.0 ** -4, 2.0 ** -10 * s[r]) * (1 + 1e-6)
        assert np.all(err <= bound)
    # the code of each element is the E4M3 of fl(x / scale)
    r = 3
    want = [orc.float_to_e4m3(float(np.float32(v) / np.float32(s[r]))) for v in xf[r]]
    np.testing.assert_array_equal(q[r], np.array(want, np.uint8))


def test_fp8_payload_and_combine(orc):
    rng = np.random.default_rng(10)
    T, H, E, k, R = 40, 64, 8, 2, 2
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    idx, w = orc.route(logits, k, renormalize=True)
    lay = orc.layout(idx, E, R)
    pl, sc = orc.payload(bits, lay["row_slot"], k, 2)
    q, s = orc.quantize_rows(bits, fp8=True)
    tok = lay["row_slot"] // k
    np.testing.assert_array_equal(pl, q[tok])
    np.testing.assert_array_equal(sc, s[tok])
    # identity experts: the combine of the FP8 payload returns each token within
    # its rows' FP8 error (renormalised weights sum to one)
    y = orc.combine(pl, sc, lay["slot_row"], w, T, k)
    yf = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).float().numpy()
    xf = x.float().numpy()
    bound = np.abs(xf) * 2.0 ** -4 + 2.0 ** -10 * s[:, None] + np.abs(xf) * 2.0 ** -7
    assert np.all(np.abs(yf - xf) <= bound * 1.001)


# ----------------------------------------------------------------------------
# 4-bit per-token payload (ThunderEP §5.2 4-bit compression): two's-complement
# nibbles, the lower-indexed element in the low nibble, scale = amax/7.
# ----------------------------------------------------------------------------
def _unpack_int4(q):
    lo = (q & 0xF).astype(np.int8)
    hi = (q >> 4).astype(np.int8)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    return np.stack([lo, hi], -1).reshape(q.shape[0], -1)


def test_int4_packing_and_ties(orc):
    # amax 7 gives scale 1 exactly, so x / scale = x: the half-integers tie and
    # go to the even neighbour (0.5 -> 0, 1.5 -> 2, 2.5 -> 2, -1.5 -> -2)
    x = torch.tensor([[7.0, -7.0, 0.5, 1.5, 2.5, -0.5, -1.5, 3.25] + [0.0] * 8]).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q, s = orc.quantize_rows(bits, int4=True)
    assert s[0] == 1.0
    # codes 7, -7, 0, 2, 2, 0, -2, 3: bytes (q0 & 15) | (q1 & 15) << 4
    assert q[0].tolist() == [0x97, 0x20, 0x02, 0x3E, 0, 0, 0, 0]
    assert [orc.dequant_int4(q[0], h, s[0]) for h in range(8)] == [7.0, -7.0, 0.0, 2.0, 2.0, 0.0, -2.0, 3.0]


def test_int4_codes_against_numpy_rint(orc):
    rng = np.random.default_rng(12)
    x = torch.from_numpy(rng.standard_normal((48, 256)).astype(np.float32) * 2).to(torch.bfloat16)
    x[7] = 0.0
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q, s = orc.quantize_rows(bits, int4=True)
    xf = x.float().numpy()
    scale = (np.abs(xf).max(1) / np.float32(7.0)).astype(np.float32)
    np.testing.assert_array_equal(s, scale)
    safe = np.where(scale > 0, scale, np.float32(1))
    want = np.where(scale[:, None] > 0, np.clip(np.rint((xf / safe[:, None]).astype(np.float32)), -7, 7), 0)
    np.testing.assert_array_equal(_unpack_int4(q), want.astype(np.int8))
    # error bound and the extremes
    deq = _unpack_int4(q).astype(np.float32) * s[:, None]
    assert np.all(np.abs(deq - xf) <= s[:, None] / 2 * (1 + 1e-6))
    rows = np.flatnonzero(s > 0)
    assert np.all(np.abs(_unpack_int4(q))[rows, np.argmax(np.abs(xf[rows]), 1)] == 7)


def test_int4_payload_and_combine(orc):
    rng = np.random.default_rng(13)
    T, H, E, k, R = 40, 64, 8, 2, 2
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    idx, w = orc.route(logits, k, renormalize=True)
    lay = orc.layout(idx, E, R)
    pl, sc = orc.payload(bits, lay["row_slot"], k, 3)
    q, s = orc.quantize_rows(bits, int4=True)
    tok = lay["row_slot"] // k
    assert pl.shape == (lay["N"], H // 2)
    np.testing.assert_array_equal(pl, q[tok])
    np.testing.assert_array_equal(sc, s[tok])
    y = orc.combine(pl, sc, lay["slot_row"], w, T, k, int4=True)
    yf = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).float().numpy()
    xf = x.float().numpy()
    assert np.all(np.abs(yf - xf) <= (s[:, None] / 2 + np.abs(xf) * 2.0 ** -7) * 1.001)
