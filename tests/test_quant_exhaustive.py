"""The per-token int8 code over its whole bf16 domain (ThunderEP on consumer
GPUs, bjdmk.com.cn, §2.3 per-token dynamic int8: one scale per token).

The kernels code x from x * inv corrected by its exact remainder instead of
dividing every element by the scale. These tests show that this is the same
code as the definition, q = clamp(rint(fl(x / scale)), -127, 127) with
scale = fl(amax / 127) for int8, q = E4M3(fl(x / scale)) with
scale = fl(amax / 448) for the FP8 payload, and q = clamp(rint(fl(x / scale)),
-7, 7) with scale = fl(amax / 7) for the int4 payload:

* on the host, exhaustively: tests/quant_exhaustive.c walks every bf16 amax
  (scale >= 2^-100) and every bf16 0 <= x <= amax (523,237,695 pairs for
  int8, 525,448,784 for int4; 1,044,457,888 signed pairs for E4M3, codes
  compared bit for bit);
* on the GPU: ep_quantize_rows(_fp8) and ep_dispatch (E = 1, k = 1, so that
  the payload rows are the tokens in order) code rows that hold every bf16
  amax and every bf16 |x| <= amax with mixed signs, compared bit for bit with
  numpy's IEEE fp32 division and ties-to-even rint (int8) or torch's
  float8_e4m3fn conversion (FP8).
"""
import shutil
import subprocess
from pathlib import Path

import numpy as np
import pytest

HERE = Path(__file__).resolve().parent


def test_division_free_code_matches_ieee_division_exhaustively(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    exe = tmp_path / "quant_exhaustive"
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", str(HERE / "quant_exhaustive.c"), "-o", str(exe),
                    "-lm"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    fields = out.stdout.split()
    got = dict(zip(fields[0::2], map(int, fields[1::2])))
    assert out.returncode == 0, out.stdout
    assert got["pairs"] == 523_237_695
    assert got["corrected_mismatch"] == 0
    assert got["fp8_pairs"] == 1_044_457_888  # both signs of x
    assert got["fp8_corrected_mismatch"] == 0
    assert got["int4_pairs"] == 525_448_784
    assert got["int4_corrected_mismatch"] == 0
    # the correction step is needed: without it some pairs code differently
    assert got["uncorrected_mismatch"] > 0 and got["fp8_uncorrected_mismatch"] > 0
    assert got["int4_uncorrected_mismatch"] > 0


H = 16384  # one column holds the row's amax, the others the swept values


def _rows_for(a_lo, a_hi):
    """bf16 bit rows: for each amax bit pattern a in [a_lo, a_hi), rows whose
    column 0 is +amax and whose other columns sweep x = 0..a (bits), signs
    mixed, zero-padded (0 leaves amax unchanged)."""
    a_vals = np.arange(a_lo, a_hi, dtype=np.int32)
    nrows = (a_vals + 1 + H - 2) // (H - 1)
    a_row = np.repeat(a_vals, nrows)
    first = np.concatenate([[0], np.cumsum(nrows)[:-1]]).astype(np.int32)
    j = np.arange(a_row.size, dtype=np.int32) - np.repeat(first, nrows)
    bits = np.empty((a_row.size, H), dtype=np.uint16)
    bits[:, 0] = a_row
    x = j[:, None] * np.int32(H - 1) + np.arange(H - 1, dtype=np.int32)[None, :]
    x[x > a_row[:, None]] = 0
    x |= ((x ^ (x >> 3) ^ j[:, None]) & 1) << 15  # mixed signs
    bits[:, 1:] = x
    return bits


def _reference(bits):
    f = (bits.astype(np.uint32) << 16).view(np.float32)
    amax = np.abs(f).max(axis=1)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0))
    q = np.rint((f / safe[:, None]).astype(np.float32))
    q = np.where(scale[:, None] > 0, np.clip(q, -127, 127), 0).astype(np.int8)
    return q, scale


def _reference_int4(bits):
    """clamp(rint(fl(x / scale)), -7, 7), scale = fl(amax / 7), packed two per
    byte (element 2i in the low nibble)."""
    f = (bits.astype(np.uint32) << 16).view(np.float32)
    amax = np.abs(f).max(axis=1)
    scale = (amax / np.float32(7.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0))
    q = np.rint((f / safe[:, None]).astype(np.float32))
    q = np.where(scale[:, None] > 0, np.clip(q, -7, 7), 0).astype(np.int8)
    n = (q.astype(np.uint8) & 0xF).reshape(q.shape[0], -1, 2)
    return (n[..., 0] | (n[..., 1] << 4)).astype(np.uint8), scale


def _reference_fp8(bits, device="cpu"):
    """E4M3 codes of fl(x / scale), scale = fl(amax / 448): the quotient by
    numpy's IEEE fp32 division, its nearest-even E4M3 by torch's float8_e4m3fn
    conversion (on `device`); |x / scale| <= 448 (1 + 2^-23) rounds to at most
    448, so nothing overflows."""
    import torch

    f = (bits.astype(np.uint32) << 16).view(np.float32)
    amax = np.abs(f).max(axis=1)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0))
    quot = (f / safe[:, None]).astype(np.float32)
    q = torch.from_numpy(quot).to(device).to(torch.float8_e4m3fn).view(torch.uint8).cpu().numpy()
    q = np.where(scale[:, None] > 0, q, 0).astype(np.uint8)
    return q, scale


def _batches(max_elems=1 << 23):
    a, hi = 0, 0x7F80  # every non-negative finite bf16 amax, 0 included
    while a < hi:
        b, elems = a, 0
        while b < hi and elems < max_elems:
            elems += ((b + 1 + H - 2) // (H - 1)) * H
            b += 1
        yield a, b
        a = b


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["int8", "fp8", "int4"])
def test_gpu_code_over_every_bf16_amax_and_value(fmt):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from combine_warp_top_fp32_b300 import binding as ep

    fp8, int4 = fmt == "fp8", fmt == "int4"
    kind = {"int8": ep.EP_PAYLOAD_INT8, "fp8": ep.EP_PAYLOAD_FP8, "int4": ep.EP_PAYLOAD_INT4}[fmt]
    quant = {"int8": ep.ep_quantize_rows, "fp8": ep.ep_quantize_rows_fp8, "int4": ep.ep_quantize_rows_int4}[fmt]
    n_elems = 0
    for b, (a_lo, a_hi) in enumerate(_batches()):
        bits = _rows_for(a_lo, a_hi)
        n = bits.shape[0]
        if int4:
            q_ref, s_ref = _reference_int4(bits)
        elif fp8:
            # torch's CUDA cast for speed, its CPU cast on every 16th batch
            q_ref, s_ref = _reference_fp8(bits, "cuda")
            if b % 16 == 0:
                np.testing.assert_array_equal(_reference_fp8(bits, "cpu")[0], q_ref)
        else:
            q_ref, s_ref = _reference(bits)
        x = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
        # ep_quantize_rows / _fp8 / _int4
        q = torch.empty(n, H // 2 if int4 else H, dtype=torch.int8 if fmt == "int8" else torch.uint8,
                        device="cuda")
        s = torch.empty(n, dtype=torch.float32, device="cuda")
        quant(x, q, s)
        # ep_dispatch with one expert and k = 1: payload row t is token t's code
        cfg = ep.make_config(n, H, 1, 1, 1, payload=kind)
        buf = ep.EpBuffers.allocate(cfg)
        buf.topk_idx.zero_()
        buf.dispatch(x)
        torch.cuda.synchronize()
        assert ep.ep_get_error(buf.ws) == ep.EP_OK
        np.testing.assert_array_equal(s.cpu().numpy(), s_ref)
        np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
        np.testing.assert_array_equal(buf.scales.cpu().numpy(), s_ref)
        np.testing.assert_array_equal(buf.payload.cpu().numpy(), q_ref)
        n_elems += bits.size
    assert n_elems > 5e8
