"""Host logic of bench.py without a GPU: byte accounting, the max-over-ranks
timing reduction on two gloo ranks, and the reference (oracle) arm."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parent.parent


def test_algorithmic_bytes_match_the_volume_formula():
    import bench
    from combine_warp_top_fp32_b300 import workloads

    g = json.loads((ROOT / "tests" / "golden" / "a2a_volume.json").read_text())
    w = workloads.WORKLOADS["large"]
    N = w.T * w.k  # dropless
    nb = bench.algorithmic_bytes(w.T, w.H, w.E, w.k, N, payload_int8=False)
    one_way = N * w.H * 2
    assert one_way == 17_179_869_184 and round(one_way / 1e9, 1) == g["one_direction_gb"]
    # dispatch writes one direction, combine reads the other; plus x, y, logits
    assert nb["dispatch"] == w.T * w.H * 2 + one_way
    assert nb["combine"] == one_way + w.T * w.H * 2
    assert nb["route"] == w.T * w.E * 4
    assert nb["total"] == nb["route"] + nb["dispatch"] + nb["combine"]
    nb8 = bench.algorithmic_bytes(w.T, w.H, w.E, w.k, N, payload_int8=True)
    assert nb8["dispatch"] == w.T * w.H * 2 + N * w.H + 4 * N


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, str(ROOT))
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(1.5 + rank)  # rank 1 is the slower one
        bench.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_max_over_ranks_without_a_group_is_identity():
    import bench

    assert bench.max_over_ranks(3.25) == 3.25


def test_reference_arm_prints_one_line(monkeypatch):
    import bench

    monkeypatch.delenv("RANK", raising=False)
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3",
                         "--reference-step-s", "0.02"])
    assert rc == 0
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_other_ranks_exit_quietly(monkeypatch):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"]) == 0
    assert buf.getvalue().strip() == ""


def test_warmup_below_three_is_rejected():
    import bench

    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])


def test_combine_only_arguments_and_bytes():
    """--combine-only parses a list of formats; with int8 expert outputs the
    combine's bytes are the combine term of algorithmic_bytes (N*H read, N*4
    scales, T*H*2 written), and int4 reads half the row bytes."""
    import bench
    from combine_warp_top_fp32_b300 import workloads

    a = bench.parse_args(["--combine-only", "bf16,int8,fp8,int4", "--workload", "capacity"])
    assert a.combine_only.split(",") == ["bf16", "int8", "fp8", "int4"]
    w = workloads.WORKLOADS["capacity"]
    N = 63_905
    per = bench.PAYLOAD_BYTES
    nb8 = bench.algorithmic_bytes(w.T, w.H, w.E, w.k, N, payload_int8=True, out_int8=True)
    assert int(N * w.H * per["int8"]) + N * 4 + w.T * w.H * 2 == nb8["combine"]
    nb16 = bench.algorithmic_bytes(w.T, w.H, w.E, w.k, N, payload_int8=True)
    assert int(N * w.H * per["bf16"]) + w.T * w.H * 2 == nb16["combine"]
    assert int(N * w.H * per["int4"]) * 2 == int(N * w.H * per["int8"])
