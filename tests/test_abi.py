"""The C-ABI library without a GPU: it loads, exports every symbol that
include/ep.h declares, and its host-side checks reject bad arguments before
any CUDA call. No test here launches a kernel."""
import ctypes
import math
import re
from pathlib import Path

import numpy as np
import pytest

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def ep():
    from combine_warp_top_fp32_b300 import build

    build.build()
    from combine_warp_top_fp32_b300 import binding

    return binding


def _declared_functions():
    text = (ROOT / "include" / "ep.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ep_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(ep):
    declared = _declared_functions()
    assert len(declared) >= 12
    assert sorted(ep.EXPORTS) == declared
    lib = ctypes.CDLL(str(ep.LIB_PATH))
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(ep):
    for s in range(6):
        assert ep.ep_status_string(s) != "unknown status"
    assert ep.ep_status_string(99) == "unknown status"


def test_workload_configs_are_valid(ep):
    from combine_warp_top_fp32_b300 import workloads

    for w in workloads.WORKLOADS.values():
        for p in w.payloads:
            cfg = ep.config_from_workload(w, payload=p)
            assert ep.ep_config_check(cfg) == ep.EP_OK, w.name
            assert ep.ep_capacity(cfg) == min(w.capacity(), w.T)
            assert ep.ep_max_rows(cfg) == w.max_rows()
            assert ep.ep_workspace_size(cfg) >= 256 + 4 * w.T * w.k


def test_capacity_matches_oracle(ep, orc):
    for (T, E, k, cf) in [(16384, 128, 8, 1.25), (100, 7, 3, 1.0), (1000, 64, 6, 0.3), (5, 4, 4, 100.0)]:
        cfg = ep.make_config(T, 64, E, k, 1, cf)
        assert ep.ep_capacity(cfg) == min(orc.capacity(T, E, k, cf), T)


@pytest.mark.parametrize("bad", [
    dict(H=8), dict(H=24), dict(H=16400), dict(E=0), dict(E=1025), dict(k=0), dict(k=9, E=8),
    dict(k=33, E=64), dict(R=3), dict(R=0), dict(T=-1), dict(capacity_factor=float("nan")),
    dict(capacity_factor=float("inf")), dict(payload=7), dict(renormalize=2),
])
def test_config_check_rejects(ep, bad):
    base = dict(T=64, H=256, E=8, k=2, R=2, capacity_factor=0.0, renormalize=0, payload=0)
    base.update(bad)
    cfg = ep.ep_config_t(**{k: v for k, v in base.items()})
    assert ep.ep_config_check(cfg) == ep.EP_ERR_INVALID_ARG
    assert ep.ep_max_rows(cfg) == 0
    n = ctypes.c_size_t()
    assert ep.lib.ep_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == ep.EP_ERR_INVALID_ARG


def test_entry_points_reject_before_any_launch(ep):
    lib = ep.lib
    cfg = ep.make_config(64, 256, 8, 2, 2)
    ref = ctypes.byref(cfg)
    null = None
    # null pointers
    assert lib.ep_route(ref, null, null, null, null) == ep.EP_ERR_INVALID_ARG
    assert lib.ep_combine(ref, null, null, 0, null, null, null, null, 0, null) == ep.EP_ERR_WORKSPACE
    # misaligned fake addresses are rejected on the host, never dereferenced
    fake16 = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10004)
    assert lib.ep_route(ref, odd, fake16, fake16, null) == ep.EP_ERR_INVALID_ARG
    # workspace too small (all other pointers plausible, never touched)
    assert lib.ep_dispatch(ref, fake16, fake16, fake16, null, fake16, fake16, fake16, null, fake16, fake16, fake16,
                           fake16, 16, null) == ep.EP_ERR_WORKSPACE
    ws_misaligned = ctypes.c_void_p(0x10010)
    assert lib.ep_dispatch(ref, fake16, fake16, fake16, null, fake16, fake16, fake16, null, fake16, fake16, fake16,
                           ws_misaligned, 1 << 20, null) == ep.EP_ERR_WORKSPACE
    # int8 payload needs scales
    cfg8 = ep.make_config(64, 256, 8, 2, 2, payload=ep.EP_PAYLOAD_INT8)
    assert lib.ep_dispatch(ctypes.byref(cfg8), fake16, fake16, fake16, null, fake16, fake16, fake16, null, fake16,
                           fake16, fake16, fake16, 1 << 20, null) == ep.EP_ERR_INVALID_ARG
    # bad combine payload enum, bad quantize shapes
    assert lib.ep_combine(ref, fake16, null, 5, fake16, fake16, fake16, fake16, 1 << 20, null) == ep.EP_ERR_INVALID_ARG
    assert lib.ep_quantize_rows(fake16, 4, 24, fake16, fake16, null) == ep.EP_ERR_INVALID_ARG
    assert lib.ep_quantize_rows(fake16, -1, 64, fake16, fake16, null) == ep.EP_ERR_INVALID_ARG
    assert lib.ep_workspace_init(null, 1024, null) == ep.EP_ERR_WORKSPACE
    assert lib.ep_get_error(null, 1024, null) == ep.EP_ERR_WORKSPACE


def test_empty_batch_route_is_a_no_op(ep):
    cfg = ep.make_config(0, 256, 8, 2, 2)
    # T == 0: nothing to do, nothing enqueued, pointers may be null
    assert ep.lib.ep_route(ctypes.byref(cfg), None, None, None, None) == ep.EP_OK
    assert ep.lib.ep_quantize_rows(None, 0, 64, None, None, None) == ep.EP_OK


def test_load_stats_closed_forms(ep, orc):
    s = ep.ep_load_stats([5, 5, 5, 5])
    assert s["cv"] == 0.0 and s["mean"] == 5.0 and s["total"] == 20
    s = ep.ep_load_stats([0, 2])
    assert s["cv"] == 1.0 and s["min"] == 0 and s["max"] == 2
    c = np.random.default_rng(0).integers(0, 1000, 128).astype(np.int32)
    assert math.isclose(ep.ep_load_stats(c)["cv"], orc.count_cv(c), rel_tol=1e-12)


def test_int4_payload_needs_h_multiple_of_32(ep):
    ok = ep.make_config(64, 32, 8, 2, 2, payload=ep.EP_PAYLOAD_INT4)
    bad = ep.make_config(64, 48, 8, 2, 2, payload=ep.EP_PAYLOAD_INT4)
    assert ep.ep_config_check(ok) == ep.EP_OK
    assert ep.ep_config_check(bad) == ep.EP_ERR_INVALID_ARG
    assert ep.ep_config_check(ep.make_config(64, 48, 8, 2, 2, payload=4)) == ep.EP_ERR_INVALID_ARG


def test_debug_hooks_reject_unknown_options(ep):
    # only invalid values: a valid one would change process-wide state
    assert ep.lib.ep_debug_set(99, 0) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_debug_set(ep.EP_DEBUG_ROUTE_DISPATCH_FORM, 7) == ep.EP_ERR_INVALID_ARG
    assert ep.lib.ep_debug_set(ep.EP_DEBUG_ROUTE_DISPATCH_FORM, -1) == ep.EP_ERR_INVALID_ARG


def test_route_dispatch_kernels_checks_its_arguments(ep):
    bad = ep.make_config(16, 15, 8, 2, 2)  # H not a multiple of 16
    n = ctypes.c_int32(-1)
    assert ep.lib.ep_route_dispatch_kernels(ctypes.byref(bad), ctypes.byref(n)) == ep.EP_ERR_INVALID_ARG
    good = ep.make_config(16, 64, 8, 2, 2)
    assert ep.lib.ep_route_dispatch_kernels(ctypes.byref(good), None) == ep.EP_ERR_INVALID_ARG
    assert n.value == -1
