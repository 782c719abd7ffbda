"""The chunked dispatch -> experts -> combine pipeline (ThunderEP on consumer
GPUs, §2.2 chunked overlap, §3.4 chunk sizes): chunk bounds on the host, and
on the GPU (a) with a row-wise expert and no capacity limit the output does
not depend on the number of chunks, bit for bit; (b) every chunk is its own
batch: its layout and its combine equal the oracle's on that chunk's tokens;
(c) coded payloads and a GEMM stand-in for the experts run through."""
import numpy as np
import pytest
import torch

from combine_warp_top_fp32_b300 import workloads


def _bounds():
    from combine_warp_top_fp32_b300.pipeline import chunk_bounds  # host logic, no GPU needed

    return chunk_bounds


@pytest.mark.parametrize("T,n", [(16384, 4), (16384, 3), (10, 4), (1, 2), (0, 3), (4096, 8), (7, 8), (5, 1)])
def test_chunk_bounds(T, n):
    b = _bounds()(T, n)
    assert b[0] == 0 and b[-1] == T
    assert all(x < y for x, y in zip(b[:-1], b[1:])) or T == 0
    assert len(b) - 1 <= max(n, 1)
    assert all(x % 4 == 0 for x in b[:-1])
    if T >= 4 * n:
        assert len(b) - 1 == n
        sizes = np.diff(b)
        assert sizes.max() - sizes.min() <= 4


def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from combine_warp_top_fp32_b300 import binding, pipeline

    return binding, pipeline


def _identity(buf):
    return buf.payload  # bf16 payload rows are the expert outputs


@pytest.mark.gpu
@pytest.mark.parametrize("n_chunks", [2, 3, 8])
def test_chunked_equals_one_pass_without_capacity(n_chunks):
    ep, pipeline = _gpu()
    w = workloads.WORKLOADS["prefill-mid"]
    cfg = ep.config_from_workload(w, payload=ep.EP_PAYLOAD_BF16)
    d = workloads.generate(w, device="cuda", expert_out=False)
    one = pipeline.ChunkedPipeline(cfg, 1)
    y1 = one.run(d["logits"], d["x"], _identity).clone()
    many = pipeline.ChunkedPipeline(cfg, n_chunks)
    yc = many.run(d["logits"], d["x"], _identity)
    torch.cuda.synchronize()
    for ch in many.chunks:
        assert ep.ep_get_error(ch.buf.ws) == ep.EP_OK
    assert torch.equal(y1, yc)


@pytest.mark.gpu
def test_each_chunk_is_its_own_batch(orc):
    ep, pipeline = _gpu()
    from combine_warp_top_fp32_b300.workloads import bf16_bits

    w = workloads.WORKLOADS["capacity"].replace(T=3000, H=256, seed=11)
    cfg = ep.config_from_workload(w, payload=ep.EP_PAYLOAD_BF16)
    d = workloads.generate(w, device="cuda", expert_out=False)
    pipe = pipeline.ChunkedPipeline(cfg, 3)
    y = pipe.run(d["logits"], d["x"], _identity)
    torch.cuda.synchronize()
    logits = d["logits"].cpu().numpy()
    x_bits = bf16_bits(d["x"])
    y_bits = bf16_bits(y)
    dropped = 0
    for ch in pipe.chunks:
        idx, wts = orc.route(logits[ch.t0:ch.t1], w.k)
        lay = orc.layout(idx, w.E, w.R, w.capacity_factor)  # cap from the chunk's own T
        np.testing.assert_array_equal(ch.buf.slot_row.cpu().numpy(), lay["slot_row"])
        np.testing.assert_array_equal(ch.buf.rank_off.cpu().numpy(), lay["rank_off"])
        pl, _ = orc.payload(x_bits[ch.t0:ch.t1], lay["row_slot"], w.k, 0)
        y_orc = orc.combine(pl, None, lay["slot_row"], ch.buf.topk_w.cpu().numpy(), ch.t1 - ch.t0, w.k)
        np.testing.assert_array_equal(y_bits[ch.t0:ch.t1], y_orc)
        dropped += lay["n_dropped"]
    assert dropped > 0  # the per-chunk caps bind


@pytest.mark.gpu
@pytest.mark.parametrize("payload", [1, 2])
def test_gemm_experts_with_coded_payload(payload):
    ep, pipeline = _gpu()
    w = workloads.WORKLOADS["prefill-mid"].replace(T=1024)
    cfg = ep.config_from_workload(w, payload=payload)
    d = workloads.generate(w, device="cuda", expert_out=False)
    g = torch.Generator(device="cuda").manual_seed(3)
    weight = (torch.randn(w.H, w.H, device="cuda", generator=g) / w.H ** 0.5).to(torch.bfloat16)
    pipe = pipeline.ChunkedPipeline(cfg, 4)
    y = pipe.run(d["logits"], d["x"], pipeline.gemm_experts(weight))
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()
    # the same rows through one pass agree to bf16 GEMM accuracy
    one = pipeline.ChunkedPipeline(cfg, 1)
    y1 = one.run(d["logits"], d["x"], pipeline.gemm_experts(weight))
    torch.cuda.synchronize()
    assert torch.allclose(y.float(), y1.float(), rtol=2e-2, atol=2e-2)
