"""The per-token int8 code over its whole bf16 domain (ThunderEP on consumer
GPUs, bjdmk.com.cn, §2.3 per-token dynamic int8: one scale per token).

The kernels code x as rint(x * inv) corrected by its exact remainder instead
of dividing every element by the scale. These tests show that this is the
same code as the definition, q = clamp(rint(fl(x / scale)), -127, 127) with
scale = fl(amax / 127):

* on the host, exhaustively: tests/quant_exhaustive.c walks every bf16 amax
  (scale >= 2^-100) and every bf16 0 <= x <= amax (523,237,695 pairs);
* on the GPU: ep_quantize_rows and ep_dispatch (E = 1, k = 1, so that the
  payload rows are the tokens in order) code rows that hold every bf16 amax
  and every bf16 |x| <= amax with mixed signs, compared bit for bit with
  numpy's IEEE fp32 division and ties-to-even rint.
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
    # the correction step is needed: without it some pairs round differently
    assert got["uncorrected_mismatch"] > 0


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
def test_gpu_int8_code_over_every_bf16_amax_and_value():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from combine_warp_top_fp32_b300 import binding as ep

    n_elems = 0
    for a_lo, a_hi in _batches():
        bits = _rows_for(a_lo, a_hi)
        n = bits.shape[0]
        q_ref, s_ref = _reference(bits)
        x = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
        # ep_quantize_rows
        q = torch.empty(n, H, dtype=torch.int8, device="cuda")
        s = torch.empty(n, dtype=torch.float32, device="cuda")
        ep.ep_quantize_rows(x, q, s)
        # ep_dispatch with one expert and k = 1: payload row t is token t's code
        cfg = ep.make_config(n, H, 1, 1, 1, payload=ep.EP_PAYLOAD_INT8)
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
