"""Comparison helpers for the GPU-vs-oracle parity tests (no GPU needed here).

Tolerances (written where they are used):
  * indices, counts, offsets, permutation, int8 codes, scales, bf16 payload
    bytes: bit-exact;
  * router weights: |w_gpu - w_oracle| <= 1e-6 * |w_oracle|;
  * combine given identical inputs (same w and slot_row): bit-exact;
  * combine through the whole path (the GPU's own weights): within 1 bf16 ulp
    of the oracle, or — where the k terms cancel and the 1e-6 weight error is
    no longer small against the result — within
    ulp_bf16(max|y|) + 2e-6 * sum_j |w_j * v_j| (the weight tolerance carried
    through the sum, plus the final rounding). That fallback may apply to at
    most MAX_FALLBACK_SHARE of the elements (and a handful in tiny outputs):
    it is reached only where the k terms cancel to below about 6e-5 of
    sum_j |w_j v_j|, so a regression that pushes many elements into it fails.
"""
from __future__ import annotations

import numpy as np

W_RTOL = 1e-6
MAX_FALLBACK_SHARE = 1e-4


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.power(2.0, e - 7)


def assert_weights_close(w_gpu: np.ndarray, w_orc: np.ndarray):
    w_gpu = np.asarray(w_gpu, np.float64)
    w_orc = np.asarray(w_orc, np.float64)
    rel = np.abs(w_gpu - w_orc) / np.maximum(np.abs(w_orc), 1e-300)
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= W_RTOL, f"router weight relative error {worst:.3e} > {W_RTOL}"
    return worst


def assert_combine_close(y_gpu_bits, y_orc_bits, w_orc, slot_row, eo_values_fn, k):
    """Whole-path combine check. eo_values_fn(rows) -> float64 [len(rows), H].
    Bit patterns are compared first; the ulp arithmetic runs only where they
    differ, so the check stays cheap on outputs of many millions of elements."""
    yg_bits = np.asarray(y_gpu_bits).astype(np.uint16, copy=False)
    yo_bits = np.asarray(y_orc_bits).astype(np.uint16, copy=False)
    assert yg_bits.shape == yo_bits.shape
    dt, dh = np.nonzero(yg_bits != yo_bits)
    yg = bf16_to_f32(yg_bits[dt, dh]).astype(np.float64)
    yo = bf16_to_f32(yo_bits[dt, dh]).astype(np.float64)
    diff = np.abs(yg - yo)
    ok = diff <= bf16_ulp(yo)
    bad = ~ok
    bad_t, bad_h = dt[bad], dh[bad]
    size = int(yo_bits.size)
    stats = dict(elements=size, exact=size - int(np.count_nonzero(diff != 0)), beyond_1ulp=int(bad_t.size))
    assert bad_t.size <= max(4, MAX_FALLBACK_SHARE * size), f"too many elements beyond 1 bf16 ulp: {stats}"
    if bad_t.size:
        slot_row = np.asarray(slot_row).reshape(-1, k)
        w_orc = np.asarray(w_orc, np.float64).reshape(-1, k)
        ygb, yob, dfb = yg[bad], yo[bad], diff[bad]
        for t in np.unique(bad_t):
            sel = bad_t == t
            hs = bad_h[sel]
            A = np.zeros(hs.size)
            for j in range(k):
                r = slot_row[t, j]
                if r < 0:
                    continue
                A += np.abs(w_orc[t, j] * eo_values_fn(np.array([r]))[0, hs])
            bound = bf16_ulp(np.maximum(np.abs(ygb[sel]), np.abs(yob[sel]))) + 2 * W_RTOL * A
            assert np.all(dfb[sel] <= bound), (t, hs[dfb[sel] > bound][:5])
    return stats
