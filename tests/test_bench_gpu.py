"""The bench's JSON line on a small workload (GPU): every key the line
promises, with values consistent with each other and with the workload."""
import io
import json
from contextlib import redirect_stdout

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bench_line_on_decode_latency(monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import bench
    from combine_warp_top_fp32_b300 import workloads

    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    steps = 3
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--workload", "decode-latency", "--steps", str(steps), "--warmup", "3",
                         "--no-cpu-baseline", "--e2e-steps", "3"])
    assert rc == 0
    lines = [ln for ln in buf.getvalue().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    w = workloads.WORKLOADS["decode-latency"]

    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["value"] > 0
    assert d["value"] == pytest.approx(w.T / (d["ms_per_step"] / 1e3), rel=1e-6)
    # ep_route_dispatch as the library reports it (on this part, the decode
    # batch takes the single cooperative launch), then the combine
    from combine_warp_top_fp32_b300 import binding as ep

    kernels = ep.ep_route_dispatch_kernels(ep.config_from_workload(w, payload=ep.EP_PAYLOAD_INT8))
    assert kernels == 1
    assert d["gpu_launches"] == (kernels + 1) * steps
    assert d["config"]["workload"] == "decode-latency" and d["config"]["payload"] == "int8"

    roof = d["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["peak"] > 0
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])

    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "tokens/s"
    assert e2e["h2d_bytes_per_step"] == w.T * w.E * 4 + w.T * w.H * 2  # logits + x
    assert e2e["d2h_bytes_per_step"] == w.T * w.H * 2  # y
    link = e2e["link"]  # the host link's own bound, measured in the same run
    assert link["h2d_gbs"] > 0 and link["d2h_gbs"] > 0 and link["both_ms"] > 0
    assert link["bound_ms_per_step"] == pytest.approx(max(link["both_ms"], d["ms_per_step"]))
    assert 0 < link["frac_of_bound"] <= 1.05

    both = d["int8_both_directions"]
    assert both["value"] > 0 and both["bytes_per_step"] < d["hbm"]["bytes_per_step"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])


def test_combine_only_line(monkeypatch):
    """bench.py --combine-only: one line with every format asked for, its
    bytes per launch as the docstring counts them, and a positive time."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import bench
    from combine_warp_top_fp32_b300 import workloads

    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--workload", "prefill-mid", "--combine-only", "bf16,int8,fp8,int4", "--steps", "3",
                         "--warmup", "3"])
    assert rc == 0
    lines = [ln for ln in buf.getvalue().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    w = workloads.WORKLOADS["prefill-mid"]
    n = d["config"]["rows_dispatched"]
    assert n == w.T * w.k  # dropless
    per = {"bf16": 2, "int8": 1, "fp8": 1, "int4": 0.5}
    assert list(d["combine"]) == ["bf16", "int8", "fp8", "int4"]
    for fmt, rec in d["combine"].items():
        assert rec["us"] > 0
        assert rec["bytes"] == int(n * w.H * per[fmt]) + (n * 4 if fmt != "bf16" else 0) + w.T * w.H * 2
        assert rec["gbs"] == pytest.approx(rec["bytes"] / rec["us"] / 1e3)
    assert d["value"] == d["combine"]["bf16"]["us"]
