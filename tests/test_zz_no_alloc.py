"""ep_dispatch_static: the dispatch entry point for callers that cannot
allocate device memory (a plugin host that only hands over input and output
buffers, a runtime with a pre-planned memory arena, a latency-critical path
that cannot take cudaMalloc's synchronisation). It keeps its scratch in a
fixed array inside the library instead of a caller workspace.

The test calls it through the C ABI twice in a row — two different problems,
so the second call runs on scratch the first one left behind — and checks
every output against ep_dispatch with its own workspace, bit for bit (the
dispatch outputs are integer, index and byte data). It also runs an empty
batch, the largest problem whose scratch fits the array (same check) and the
smallest that does not, which is refused before anything runs. The array's
size comes from include/ep.h. This file is collected last and passes alone in
a fresh process as well.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from combine_warp_top_fp32_b300 import binding

    return binding


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _outputs(ep, cfg):
    b = ep.EpBuffers.allocate(cfg)
    for t in (b.payload, b.row_slot, b.slot_row, b.expert_counts, b.expert_raw, b.expert_off, b.rank_off,
              b.n_dropped):
        t.fill_(0x5A if t.dtype != torch.bfloat16 else 0)
    if b.scales is not None:
        b.scales.fill_(-1.0)
    return b


def _static_call(ep, b, x, stream):
    return ep.lib.ep_dispatch_static(ctypes.byref(b.cfg), _p(x), _p(b.topk_idx), _p(b.payload), _p(b.scales),
                                     _p(b.row_slot), _p(b.slot_row), _p(b.expert_counts), _p(b.expert_raw),
                                     _p(b.expert_off), _p(b.rank_off), _p(b.n_dropped),
                                     ctypes.c_void_p(stream.cuda_stream))


def _compare(ref, got):
    N = int(ref.rank_off[-1].item())
    assert int(got.rank_off[-1].item()) == N
    for name in ("topk_idx", "slot_row", "expert_counts", "expert_raw", "expert_off", "rank_off", "n_dropped"):
        assert torch.equal(getattr(ref, name), getattr(got, name)), name
    assert torch.equal(ref.row_slot[:N], got.row_slot[:N])
    assert torch.equal(ref.payload[:N].view(torch.uint8), got.payload[:N].view(torch.uint8))
    if ref.scales is not None:
        assert torch.equal(ref.scales[:N], got.scales[:N])


@pytest.mark.parametrize("problems", [(("capacity", 1), ("prefill-mid", 0))])
def test_static_dispatch_matches_workspace_dispatch_twice(ep, problems):
    from combine_warp_top_fp32_b300 import workloads

    stream = torch.cuda.current_stream()
    for name, payload in problems:  # two calls in a row on the shared scratch
        w = workloads.WORKLOADS[name]
        cfg = ep.config_from_workload(w, payload=payload)
        assert ep.ep_workspace_size(cfg) <= ep.EP_STATIC_SCRATCH_BYTES
        d = workloads.generate(w, device="cuda", expert_out=False)
        ref = _outputs(ep, cfg)
        ref.route(d["logits"])
        ref.dispatch(d["x"])
        got = _outputs(ep, cfg)
        got.topk_idx.copy_(ref.topk_idx)
        assert _static_call(ep, got, d["x"], stream) == ep.EP_OK
        torch.cuda.synchronize()
        assert ep.ep_get_error(ref.ws) == ep.EP_OK
        _compare(ref, got)


def _largest_fitting_T(ep, H, E, k, R):
    """The largest T whose dispatch scratch fits the static array (the
    workspace size grows with T)."""
    lo, hi = 1, 1
    while ep.ep_workspace_size(ep.make_config(hi, H, E, k, R)) <= ep.EP_STATIC_SCRATCH_BYTES:
        lo, hi = hi, hi * 2
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if ep.ep_workspace_size(ep.make_config(mid, H, E, k, R)) <= ep.EP_STATIC_SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid
    return lo


def test_static_dispatch_at_the_limit_and_past_it(ep):
    H, E, k, R = 16, 8, 8, 2
    T = _largest_fitting_T(ep, H, E, k, R)
    assert ep.ep_workspace_size(ep.make_config(T + 1, H, E, k, R)) > ep.EP_STATIC_SCRATCH_BYTES
    stream = torch.cuda.current_stream()
    g = torch.Generator(device="cuda").manual_seed(11)
    x = torch.randn(T + 1, H, device="cuda", generator=g).to(torch.bfloat16)
    logits = torch.randn(T + 1, E, device="cuda", generator=g)
    # at the limit: runs, and writes what ep_dispatch writes
    cfg = ep.make_config(T, H, E, k, R, payload=ep.EP_PAYLOAD_INT8)
    ref = _outputs(ep, cfg)
    ref.route(logits[:T].contiguous())
    ref.dispatch(x[:T].contiguous())
    got = _outputs(ep, cfg)
    got.topk_idx.copy_(ref.topk_idx)
    assert _static_call(ep, got, x, stream) == ep.EP_OK
    torch.cuda.synchronize()
    assert ep.ep_get_error(ref.ws) == ep.EP_OK
    _compare(ref, got)
    # one token more: refused, nothing written
    big = _outputs(ep, ep.make_config(T + 1, H, E, k, R, payload=ep.EP_PAYLOAD_INT8))
    big.slot_row.fill_(7)
    assert _static_call(ep, big, x, stream) == ep.EP_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(big.slot_row == 7)


def test_static_dispatch_of_an_empty_batch(ep):
    cfg = ep.make_config(0, 64, 8, 2, 2, payload=ep.EP_PAYLOAD_INT8)
    b = _outputs(ep, cfg)
    b.expert_off.fill_(7)
    b.rank_off.fill_(7)
    b.n_dropped.fill_(7)
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    assert _static_call(ep, b, x, torch.cuda.current_stream()) == ep.EP_OK
    torch.cuda.synchronize()
    assert b.expert_off.cpu().tolist() == [0] * 9
    assert b.rank_off.cpu().tolist() == [0] * 3
    assert b.n_dropped.item() == 0


def test_static_dispatch_refuses_a_problem_larger_than_its_scratch(ep):
    # T*k*4 bytes of per-pair ranks alone exceed the array
    T, H, E, k = 300_000, 16, 8, 8
    cfg = ep.make_config(T, H, E, k, 2)
    assert ep.ep_workspace_size(cfg) > ep.EP_STATIC_SCRATCH_BYTES
    b = ep.EpBuffers.allocate(cfg)  # real buffers: nothing may run, but nothing could fault either
    x = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    b.slot_row.fill_(7)
    assert _static_call(ep, b, x, torch.cuda.current_stream()) == ep.EP_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(b.slot_row == 7)  # untouched: refused before any launch
