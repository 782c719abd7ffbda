"""Benchmark: MoE expert-parallel dispatch + combine on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload capacity] [--payload int8|bf16]
    python bench.py --impl reference ...      # the CPU oracle on a bounded sample

A step is one pass of the whole path over one batch: ep_route -> ep_dispatch
-> ep_combine on one stream, inputs resident in HBM. The headline workload is
T=16384 tokens, H=4096, E=128 experts, top-8, R=8 virtual ranks, capacity
factor 1.25, int8 payload. The metric is tokens/s; achieved HBM GB/s on the
algorithmic bytes (logits + x + payload + scales + expert outputs + y) is
reported beside it as a fraction of both the nominal 8 TB/s and the measured
copy bandwidth.

Under torchrun (N>1) every rank runs an independent replica of the workload
on its own GPU (the path has no exchange step on one node: its R ranks are
virtual), timing takes the max over ranks, and `value` counts all ranks'
tokens. Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6400.0
L2_BYTES = 126 * 1024 * 1024
METRIC = "dispatch+combine tokens/s and HBM GB/s as % of B300 peak (T=16384,H=4096)"
TRAFFIC_FILE = ROOT / "profiles" / "roofline_traffic.json"
PAYLOAD_MODE = {"bf16": 0, "int8": 1, "fp8": 2, "int4": 3}
PAYLOAD_BYTES = {"bf16": 2.0, "int8": 1.0, "fp8": 1.0, "int4": 0.5}  # per element


# ----------------------------------------------------------------------------
# algorithmic bytes (per step, per kernel)
# ----------------------------------------------------------------------------
def algorithmic_bytes(T, H, E, k, N, payload_int8, out_int8=False, payload_bytes=None):
    """Bytes each stage must move at least once, with N dispatched rows.

    route:    logits T*E*4 read
    dispatch: x T*H*2 read; payload N*H*b written (+ scales N*4 for int8 / FP8 / int4 codes)
    combine:  expert outputs N*H*b_out read (+ N*4 scales if coded); y T*H*2 written
    Routing metadata (indices, weights, slot maps: ~16*T*k bytes) is kept apart.
    b = payload_bytes per element when given (0.5 for int4), else 1 or 2.
    """
    b = payload_bytes if payload_bytes is not None else (1 if payload_int8 else 2)
    b_out = 1 if out_int8 else 2
    route = T * E * 4
    dispatch = T * H * 2 + int(N * H * b) + (N * 4 if payload_int8 else 0)
    combine = N * H * b_out + (N * 4 if out_int8 else 0) + T * H * 2
    meta = T * k * 4 * 4
    return dict(route=route, dispatch=dispatch, combine=combine, total=route + dispatch + combine, metadata=meta)


def measured_peak_gbs():
    p = ROOT / "MEASURED_PEAKS.json"
    try:
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(paths):
    h = hashlib.sha256()
    for p in paths:
        h.update(Path(p).read_bytes())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "combine": ["combine_warp_top_fp32_b300/csrc/combine.cu", "combine_warp_top_fp32_b300/csrc/ep_device.cuh"],
    "dispatch": ["combine_warp_top_fp32_b300/csrc/dispatch.cu", "combine_warp_top_fp32_b300/csrc/ep_device.cuh"],
    "route": ["combine_warp_top_fp32_b300/csrc/route.cu"],
}


def recorded_traffic(kernel, workload, payload):
    """DRAM bytes per launch from an ncu capture, only if the kernel's sources
    are unchanged since that capture (else None)."""
    try:
        d = json.loads(TRAFFIC_FILE.read_text())
        rec = d[f"{kernel}/{workload}/{payload}"]
        if rec["source_digest"] != source_digest(ROOT / p for p in KERNEL_SOURCES[kernel]):
            return None
        return int(rec["dram_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.error = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception as e:  # no nvidia-smi: report why
            self.error = f"nvidia-smi unavailable: {e}"

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"error": self.error}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"error": "no clock samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ----------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, group=None) -> float:
    """The slowest rank's time (a no-op without an initialised process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return value
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ----------------------------------------------------------------------------
# CPU oracle timing (reference arm and the cpu_baseline leg)
# ----------------------------------------------------------------------------
def oracle_sample_tokens(w, target_s=2.0, probe_tokens=256):
    """Tokens per oracle step so that one step takes about target_s seconds."""
    t = oracle_pass_seconds(w, min(probe_tokens, w.T))
    per_token = t / min(probe_tokens, w.T)
    return max(1, min(w.T, int(target_s / max(per_token, 1e-9))))


_oracle_cache = {}
_last_oracle_rows = [None]  # rows dispatched by the last oracle pass
_oracle_generator = [None]  # where the cached oracle inputs were drawn ("cuda": the GPU arm's bytes)


def _oracle_inputs(w, n_tokens):
    import torch

    from combine_warp_top_fp32_b300 import workloads

    key = (w.name, n_tokens)
    if key not in _oracle_cache:
        ws = w.replace(T=n_tokens)
        # the whole workload on a GPU machine: the device generator, as the GPU arm
        # draws it, copied to the host (the same bytes); else the host generator
        dev = "cuda" if n_tokens == w.T and torch.cuda.is_available() else "cpu"
        d = {k: v.cpu() for k, v in workloads.generate(ws, device=dev).items()}
        _oracle_cache.clear()
        _oracle_cache[key] = (ws, d["logits"].numpy(), workloads.bf16_bits(d["x"]), workloads.bf16_bits(d["expert_out"]))
        _oracle_generator[0] = dev
    return _oracle_cache[key]


def oracle_pass_seconds(w, n_tokens, payload_int8=None):
    import oracle

    ws, logits, x_bits, eo_bits = _oracle_inputs(w, n_tokens)
    orc = oracle.Oracle()
    p8 = int(w.payloads[0]) if payload_int8 is None else int(payload_int8)  # oracle payload mode
    t0 = time.perf_counter()
    out = orc.forward(logits, x_bits, eo_bits, ws.k, ws.R, ws.capacity_factor, ws.renormalize, p8)
    dt = time.perf_counter() - t0
    _last_oracle_rows[0] = int(out["N"])
    return dt


def run_reference(args):
    ws_, rank, _ = dist_env()
    if rank != 0:
        return 0
    from combine_warp_top_fp32_b300 import workloads

    w = workloads.WORKLOADS[args.workload]
    p8 = PAYLOAD_MODE[args.payload]
    n = oracle_sample_tokens(w, target_s=args.reference_step_s)
    for _ in range(args.warmup):
        oracle_pass_seconds(w, n, p8)
    times = [oracle_pass_seconds(w, n, p8) for _ in range(args.steps)]
    total = sum(times)
    value = n * args.steps / total
    cores = 1
    if n == w.T and _oracle_generator[0] == "cuda":
        sample = f"the whole '{w.name}' workload ({w.T} tokens) per step, the same bytes the GPU arm times"
    elif n == w.T:
        sample = (f"the whole '{w.name}' workload ({w.T} tokens) per step, drawn by the host generator "
                  f"(no GPU here: not the GPU arm's bytes)")
    else:
        sample = (f"first {n} of {w.T} tokens of the '{w.name}' workload per step "
                  f"(an instance of the same shape with T={n})")
    rows = _last_oracle_rows[0] if n == w.T else None
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32",
        "data": "synthetic", "config": dict(workload_config(w, args.payload, rows, False, args.path),
                                            path="CPU oracle (route, layout, payload, combine)", launch="host"),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
                         "cpu": cpu_model()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def cpu_model():
    try:
        for ln in Path("/proc/cpuinfo").read_text().splitlines():
            if ln.startswith("model name"):
                return ln.split(":", 1)[1].strip() + f" (nproc={os.cpu_count()})"
    except Exception:
        pass
    return f"unknown (nproc={os.cpu_count()})"


def workload_config(w, payload, n_rows, eager=False, path="fused"):
    rows = n_rows if n_rows is not None else w.max_rows()
    step_bytes = algorithmic_bytes(w.T, w.H, w.E, w.k, rows, payload != "bf16",
                                   payload_bytes=PAYLOAD_BYTES[payload])["total"]
    l2 = (f"no flush: each step moves {step_bytes / 1e9:.2f} GB, beyond the 126 MB L2" if step_bytes > L2_BYTES else
          f"not flushed: the {step_bytes / 1e6:.1f} MB step fits in the 126 MB L2 (latency-bound shape)")
    return {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "R": w.R,
            "capacity_factor": w.capacity_factor, "cap": w.capacity() if w.capacity_factor > 0 else None,
            "payload": payload, "expert_out": "bf16", "rows_dispatched": n_rows, "l2": l2,
            "parallelism": "replicas (R virtual ranks per GPU)",
            "path": ("ep_route_dispatch + ep_combine" if path == "fused" else "ep_route + ep_dispatch + ep_combine"),
            "launch": "eager" if eager else "one cuda graph of all timed steps; stage events on a side branch"}


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------
def graph_stage_ms(stage_fns, steps):
    """Total and per-stage ms per step of `steps` steps of the stage callables,
    replayed as one CUDA graph after an untimed replay; stage times from
    event-record nodes on a side branch (as in the headline measurement)."""
    import torch

    names = list(stage_fns)
    stream = torch.cuda.current_stream()
    ev_start = torch.cuda.Event(enable_timing=True, external=True)
    ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in names] for _ in range(steps)]
    side = torch.cuda.Stream()
    warm = torch.cuda.Stream()
    warm.wait_stream(stream)
    with torch.cuda.stream(warm):
        for fn in stage_fns.values():
            fn()
    stream.wait_stream(warm)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        main = torch.cuda.current_stream()
        ev_start.record(main)
        for i in range(steps):
            for j, n in enumerate(names):
                stage_fns[n]()
                side.wait_stream(main)
                ev[i][j].record(side)
        main.wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    ends = [e for step in ev for e in step]
    starts = [ev_start] + ends[:-1]
    stage_ms = {n: 0.0 for n in names}
    for q, (s0, s1) in enumerate(zip(starts, ends)):
        stage_ms[names[q % len(names)]] += s0.elapsed_time(s1) / steps
    del graph
    return t0.elapsed_time(t1) / steps, stage_ms


def large_records(steps, peak, peak_src):
    """The T=131072, H=8192 workload (the target's second config) timed beside
    the headline, int8 and bf16 payloads, ep_route_dispatch + ep_combine."""
    import torch

    from combine_warp_top_fp32_b300 import binding as ep
    from combine_warp_top_fp32_b300 import workloads

    w = workloads.WORKLOADS["large"]
    d = workloads.generate(w, device="cuda")
    out = {}
    for payload in ("int8", "bf16"):
        p8 = PAYLOAD_MODE[payload]
        cfg = ep.config_from_workload(w, payload=p8)
        buf = ep.EpBuffers.allocate(cfg)
        fns = {"route+dispatch": lambda: buf.route_dispatch(d["logits"], d["x"]),
               "combine": lambda: buf.combine(d["expert_out"])}
        ms, stage_ms = graph_stage_ms(fns, steps)
        assert ep.ep_get_error(buf.ws) == ep.EP_OK
        N = int(buf.rank_off[-1].item())
        nb = algorithmic_bytes(w.T, w.H, w.E, w.k, N, p8 != 0, payload_bytes=PAYLOAD_BYTES[payload])
        gbs = nb["total"] / (ms / 1e3) / 1e9
        comb_gbs = nb["combine"] / (stage_ms["combine"] / 1e3) / 1e9
        out[payload] = {
            "ms_per_step": ms, "value": w.T / (ms / 1e3), "unit": "tokens/s", "steps": steps,
            "bytes_per_step": nb["total"], "gbs": gbs, "frac_of_8000": gbs / NOMINAL_HBM_GBS,
            f"frac_of_{peak_src}": gbs / peak,
            "stages_ms": stage_ms,
            "roofline": {"bound": "hbm", "kernel": "combine_kernel<bf16>", "achieved": comb_gbs, "peak": peak,
                         "unit": "GB/s", "frac": comb_gbs / peak, "algorithmic_bytes_per_launch": nb["combine"]},
            "gpu_launches": (ep.ep_route_dispatch_kernels(cfg) + 1) * steps,
        }
        del buf, fns
        torch.cuda.empty_cache()
    del d
    torch.cuda.empty_cache()
    return out


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from combine_warp_top_fp32_b300 import binding as ep
    from combine_warp_top_fp32_b300 import workloads

    w = workloads.WORKLOADS[args.workload]
    p8 = PAYLOAD_MODE[args.payload]  # 0 bf16, 1 int8, 2 FP8 E4M3 (the library's EP_PAYLOAD_* values)
    cfg = ep.config_from_workload(w, payload=p8)
    d = workloads.generate(w, device=dev)
    logits, x, eo = d["logits"], d["x"], d["expert_out"]
    buf = ep.EpBuffers.allocate(cfg)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        if args.path == "fused":
            buf.route_dispatch(logits, x)
            buf.combine(eo)
        else:
            buf.step(logits, x, eo)
    torch.cuda.synchronize()
    assert ep.ep_get_error(buf.ws) == ep.EP_OK
    N = int(buf.rank_off[-1].item())
    if args.path == "fused":
        # ep_route_dispatch (as many kernels as the library reports for this
        # shape and device: one cooperative launch, or the cluster form, or
        # route+count, scan, scatter), then ep_combine (none for an empty batch)
        launches_per_step = ep.ep_route_dispatch_kernels(cfg) + (1 if w.T > 0 else 0)
    else:
        # ep_route; ep_dispatch (count, scan, scatter); ep_combine
        launches_per_step = 5 if w.T > 0 else 2

    # The timed region is one CUDA graph holding all K steps (the library's
    # calls neither synchronise nor allocate, so they capture as they are):
    # replaying it takes the host's per-call overhead off the GPU's critical
    # path (the Sparse-communication article's §4.2 suggestion), and the
    # library's programmatic dependent launches overlap each kernel's launch
    # with its predecessor's tail. Stage times are taken live by event-record
    # nodes on a side branch of the graph: after each call the side stream
    # waits on the main stream and records an event, and nothing waits on
    # those events, so they do not break the chain of dependent launches.
    # Stage i ends at its event; it starts where the previous stage ended.
    if args.path == "fused":
        stage_fns = {"route+dispatch": lambda: buf.route_dispatch(logits, x), "combine": lambda: buf.combine(eo)}
    else:
        stage_fns = {"route": lambda: buf.route(logits), "dispatch": lambda: buf.dispatch(x),
                     "combine": lambda: buf.combine(eo)}
    names = list(stage_fns)
    ev_start = torch.cuda.Event(enable_timing=True, external=not args.eager)
    ev = [[torch.cuda.Event(enable_timing=True, external=not args.eager) for _ in names] for _ in range(args.steps)]
    side = torch.cuda.Stream()

    def steps_with_events():
        main = torch.cuda.current_stream()
        ev_start.record(main)
        for i in range(args.steps):
            for j, n in enumerate(names):
                stage_fns[n]()
                if args.eager:
                    ev[i][j].record(main)
                else:
                    side.wait_stream(main)
                    ev[i][j].record(side)
        if not args.eager:
            main.wait_stream(side)

    graph = None
    if not args.eager:
        warm = torch.cuda.Stream()
        warm.wait_stream(stream)
        with torch.cuda.stream(warm):
            for fn in stage_fns.values():
                fn()
        stream.wait_stream(warm)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            steps_with_events()
        graph.replay()  # untimed warm-up pass of the captured steps
        torch.cuda.synchronize()
        assert ep.ep_get_error(buf.ws) == ep.EP_OK

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        steps_with_events()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    assert ep.ep_get_error(buf.ws) == ep.EP_OK
    clocks = sampler.stop()
    total_ms = t0.elapsed_time(t1)
    ends = [e for step in ev for e in step]
    starts = [ev_start] + ends[:-1]
    stage_ms = {n: 0.0 for n in names}
    for q, (s0, s1) in enumerate(zip(starts, ends)):
        stage_ms[names[q % len(names)]] += s0.elapsed_time(s1) / args.steps
    total_s = max_over_ranks(total_ms / 1e3)
    ms_per_step = 1e3 * total_s / args.steps
    tokens = w.T * args.steps * world
    value = tokens / total_s

    nb = algorithmic_bytes(w.T, w.H, w.E, w.k, N, p8 != 0, payload_bytes=PAYLOAD_BYTES[args.payload])
    nb["route+dispatch"] = nb["route"] + nb["dispatch"]
    peak, peak_src = measured_peak_gbs()
    step_gbs = nb["total"] / (ms_per_step / 1e3) / 1e9
    stage_gbs = {s: nb[s] / (stage_ms[s] / 1e3) / 1e9 for s in stage_ms}
    dominant = max(stage_ms, key=stage_ms.get)
    kernel_names = {"route": "route_topk_kernel", "dispatch": "count+scan+scatter_kernel",
                    "route+dispatch": ("route_dispatch_fused_kernel" if ep.ep_route_dispatch_kernels(cfg) == 1
                                       else "route_count+scan+scatter_kernel"),
                    "combine": "combine_kernel<bf16>"}
    traffic = recorded_traffic(dominant, w.name, args.payload)

    # int8 in both directions, beside the headline (not in place of it): the
    # experts return int8 rows + per-row scales (ep_quantize_rows of the same
    # expert outputs), which the combine dequantises. Same graph timing.
    both = None
    if p8 == PAYLOAD_MODE["int8"] and w.T > 0 and not args.no_int8_return:
        eo_q = torch.empty(eo.shape, dtype=torch.int8, device=dev)
        eo_s = torch.empty(eo.shape[0], dtype=torch.float32, device=dev)
        ep.ep_quantize_rows(eo, eo_q, eo_s)

        def step_q():
            if args.path == "fused":
                buf.route_dispatch(logits, x)
            else:
                buf.route(logits)
                buf.dispatch(x)
            buf.combine(eo_q, eo_s)

        warm = torch.cuda.Stream()
        warm.wait_stream(stream)
        with torch.cuda.stream(warm):
            step_q()
        stream.wait_stream(warm)
        gq = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gq):
            for _ in range(args.steps):
                step_q()
        gq.replay()
        torch.cuda.synchronize()
        q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        q0.record(stream)
        gq.replay()
        q1.record(stream)
        torch.cuda.synchronize()
        barrier()
        assert ep.ep_get_error(buf.ws) == ep.EP_OK
        q_s = max_over_ranks(q0.elapsed_time(q1) / 1e3)
        nbq = algorithmic_bytes(w.T, w.H, w.E, w.k, N, True, out_int8=True)
        q_gbs = nbq["total"] / (q_s / args.steps) / 1e9
        both = {"ms_per_step": 1e3 * q_s / args.steps, "value": w.T * args.steps * world / q_s, "unit": "tokens/s",
                "bytes_per_step": nbq["total"], "gbs": q_gbs, "frac_of_8000": q_gbs / NOMINAL_HBM_GBS,
                f"frac_of_{peak_src}": q_gbs / peak,
                "note": "expert outputs returned as int8 + fp32 row scales (ep_quantize_rows), dequantised by the combine"}
        del eo_q, eo_s, gq

    # end to end through the public API with host buffers: pinned H2D of the
    # step's inputs (logits, x), the calls, D2H of the result y, every step.
    # The expert outputs stay the device-resident stand-in of the timed steps:
    # in an MoE layer they are made on the GPU by the experts, between
    # dispatch and combine, and never cross the host link. Steps are double
    # buffered on three streams, as a serving loop would run them: step i's
    # D2H of y overlaps step i+1's H2D of its inputs (the two directions of
    # the link) and each step's kernels wait only for their own inputs.
    e2e = None
    if not args.no_e2e:
        h_logits = logits.cpu().pin_memory()
        h_x = x.cpu().pin_memory()
        bufs = [buf, ep.EpBuffers.allocate(cfg)]
        h_y = [torch.empty(buf.y.shape, dtype=buf.y.dtype).pin_memory() for _ in bufs]
        d_in = [(torch.empty_like(logits), torch.empty_like(x)) for _ in bufs]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in bufs]       # inputs of slot b copied
        ev_comp = [torch.cuda.Event() for _ in bufs]     # slot b's kernels done
        ev_out = [torch.cuda.Event() for _ in bufs]      # slot b's y copied out
        used = [False, False]

        def e2e_step(i):
            b = i % 2
            d_logits, d_x = d_in[b]
            with torch.cuda.stream(s_in):
                if used[b]:
                    s_in.wait_event(ev_comp[b])  # the kernels of step i-2 have read these inputs
                d_logits.copy_(h_logits, non_blocking=True)
                d_x.copy_(h_x, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if used[b]:
                stream.wait_event(ev_out[b])  # step i-2's y has left this slot
            if args.path == "fused":
                bufs[b].route_dispatch(d_logits, d_x)
                bufs[b].combine(eo)
            else:
                bufs[b].step(d_logits, d_x, eo)
            ev_comp[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b])
                h_y[b].copy_(bufs[b].y, non_blocking=True)
                ev_out[b].record(s_out)
            used[b] = True

        for i in range(max(2, min(args.warmup, 4))):
            e2e_step(i)
        torch.cuda.synchronize()
        k2 = max(1, min(args.steps, args.e2e_steps))
        barrier()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(s_in)
        for i in range(k2):
            e2e_step(i)
        s_in.wait_stream(s_out)  # the last step's y is on the host
        s1.record(s_in)
        torch.cuda.synchronize()
        barrier()
        assert all(ep.ep_get_error(bb.ws) == ep.EP_OK for bb in bufs)
        e2e_s = max_over_ranks(s0.elapsed_time(s1) / 1e3)
        h2d = logits.numel() * 4 + x.numel() * 2
        e2e = {"value": w.T * k2 * world / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": buf.y.numel() * 2, "steps": k2,
               "note": "H2D logits + x, D2H y each step, double buffered on three streams; "
                       "expert outputs are the device-resident stand-in"}
        # the host link's own bound for these copies, measured in this run:
        # the step's H2D alone, its D2H alone, and both at once on the two
        # copy streams; the loop cannot beat the slowest of (both copies at
        # once, the device step), so its fraction of that bound says how much
        # of the e2e time the schedule itself loses
        def copy_ms(do_h2d, do_d2h, reps=5):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            c0.record(s_in)
            s_out.wait_event(c0)
            for _ in range(reps):
                if do_h2d:
                    with torch.cuda.stream(s_in):
                        d_in[0][0].copy_(h_logits, non_blocking=True)
                        d_in[0][1].copy_(h_x, non_blocking=True)
                if do_d2h:
                    with torch.cuda.stream(s_out):
                        h_y[0].copy_(bufs[0].y, non_blocking=True)
            s_in.wait_stream(s_out)
            c1.record(s_in)
            torch.cuda.synchronize()
            return c0.elapsed_time(c1) / reps

        t_h2d, t_d2h, t_both = copy_ms(True, False), copy_ms(False, True), copy_ms(True, True)
        bound_ms = max(t_both, ms_per_step)
        e2e_ms = 1e3 * e2e_s / k2
        e2e["link"] = {"h2d_gbs": h2d / (t_h2d / 1e3) / 1e9, "d2h_gbs": buf.y.numel() * 2 / (t_d2h / 1e3) / 1e9,
                       "h2d_ms": t_h2d, "d2h_ms": t_d2h, "both_ms": t_both, "device_step_ms": ms_per_step,
                       "bound_ms_per_step": bound_ms, "e2e_ms_per_step": e2e_ms, "frac_of_bound": bound_ms / e2e_ms,
                       "note": "pinned host buffers; both = the step's H2D and D2H at once on two streams"}

    # the target's second configuration beside the headline (one GPU runs)
    large = None
    if args.workload == "capacity" and not args.no_large and world == 1:
        large = large_records(args.large_steps, peak, peak_src)

    cpu_baseline = None
    if rank == 0 and not args.no_cpu_baseline:
        n = oracle_sample_tokens(w, target_s=args.cpu_baseline_s / 3)
        reps = 3
        secs = sum(oracle_pass_seconds(w, n, p8) for _ in range(reps))
        cpu_baseline = {"value": n * reps / secs, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                        "sample": f"{reps} passes over the first {n} of {w.T} tokens (same shape, T={n})",
                        "cpu": cpu_model()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp32", "data": "synthetic", "config": workload_config(w, args.payload, N, args.eager, args.path),
            "hbm": {"bytes_per_step": nb["total"], "gbs": step_gbs, "frac_of_8000": step_gbs / NOMINAL_HBM_GBS,
                    f"frac_of_{peak_src}": step_gbs / peak, "metadata_bytes_per_step": nb["metadata"]},
            "stages": {s: {"ms": stage_ms[s], "bytes": nb[s], "gbs": stage_gbs[s]} for s in stage_ms},
            "roofline": {"bound": "hbm", "kernel": kernel_names[dominant], "achieved": stage_gbs[dominant],
                         "peak": peak, "unit": "GB/s", "frac": stage_gbs[dominant] / peak, "traffic": traffic,
                         "algorithmic_bytes_per_launch": nb[dominant], "peak_source": peak_src},
            "clocks": clocks,
            "gpu_launches": launches_per_step * args.steps,
            "e2e": e2e,
            "cpu_baseline": cpu_baseline,
        }
        if both is not None:
            line["int8_both_directions"] = both
        if large is not None:
            line["large"] = large
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------
# chunked pipeline (ThunderEP §2.2 overlap, §3.4 chunk sizes)
# ----------------------------------------------------------------------------
def run_pipeline(args):
    """Per chunk count C: one pass = ep_route_dispatch / stand-in expert GEMM /
    ep_combine over C chunks on two streams. Times, per step: e2e (with the
    GEMM experts), comm (the same pipeline with identity experts: dispatch and
    combine only) and compute (the GEMMs alone on the same chunk buffers);
    overlap shows as e2e < comm + compute. Each is one CUDA graph of K steps."""
    import torch

    from combine_warp_top_fp32_b300 import binding as ep
    from combine_warp_top_fp32_b300 import pipeline, workloads

    torch.cuda.set_device(0)
    w = workloads.WORKLOADS[args.workload]
    p8 = PAYLOAD_MODE[args.payload]
    cfg = ep.config_from_workload(w, payload=p8)
    d = workloads.generate(w, device="cuda", expert_out=False)
    g = torch.Generator(device="cuda").manual_seed(7)
    weight = (torch.randn(w.H, w.H, device="cuda", generator=g) / w.H ** 0.5).to(torch.bfloat16)
    gemm = pipeline.gemm_experts(weight)

    def identity(buf):
        if buf.payload.dtype == torch.bfloat16:
            return buf.payload
        return (buf.payload, buf.scales)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(args.steps):
                fn()
        graph.replay()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        graph.replay()
        t1.record()
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / args.steps

    table = {}
    for C in [int(c) for c in args.pipeline.split(",")]:
        pipe = pipeline.ChunkedPipeline(cfg, C)
        e2e = timed(lambda: pipe.run(d["logits"], d["x"], gemm))
        comm = timed(lambda: pipe.run(d["logits"], d["x"], identity))
        compute = timed(lambda: [gemm(ch.buf) for ch in pipe.chunks])
        for ch in pipe.chunks:
            assert ep.ep_get_error(ch.buf.ws) == ep.EP_OK
        table[str(C)] = {"chunks": len(pipe.chunks), "e2e_ms": e2e, "comm_ms": comm, "compute_ms": compute,
                         "overlap_saved_ms": comm + compute - e2e}
        del pipe
    best = min(table.values(), key=lambda r: r["e2e_ms"])
    line = {"metric": "chunked dispatch + expert GEMM + combine, ms per step", "value": best["e2e_ms"],
            "unit": "ms", "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "data": "synthetic", "config": dict(workload_config(w, args.payload, None, False, "fused"),
                                                expert="one bf16 [H, H] GEMM per dispatched row (cuBLAS)"),
            "pipeline": table}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------
# compact routing metadata (intelliparadigm §4.1: [bitmap, data])
# ----------------------------------------------------------------------------
def run_bitmap(args):
    """Metadata bytes per step as (expert id, position) pairs against one
    bitmap per token, and the device time of ep_bitmap_encode (sender) and
    ep_bitmap_layout (receiver rebuilding counts, offsets and row -> token),
    each one CUDA graph of K calls."""
    import torch

    from combine_warp_top_fp32_b300 import binding as ep
    from combine_warp_top_fp32_b300 import workloads

    torch.cuda.set_device(0)
    w = workloads.WORKLOADS[args.workload]
    cfg = ep.config_from_workload(w, payload=PAYLOAD_MODE[args.payload])
    d = workloads.generate(w, device="cuda", expert_out=False)
    buf = ep.EpBuffers.allocate(cfg)
    buf.route(d["logits"])
    words = ep.bitmap_words(w.E)
    bm = torch.empty((w.T, words), dtype=torch.int32, device="cuda")
    row_token = torch.empty((max(ep.ep_max_rows(cfg), 1),), dtype=torch.int32, device="cuda")
    i32 = dict(dtype=torch.int32, device="cuda")
    outs = [torch.empty(w.E, **i32), torch.empty(w.E, **i32), torch.empty(w.E + 1, **i32),
            torch.empty(w.R + 1, **i32), torch.empty(1, **i32)]

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(args.steps):
                fn()
        g.replay()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        g.replay()
        t1.record()
        torch.cuda.synchronize()
        return 1e3 * t0.elapsed_time(t1) / args.steps

    enc = timed(lambda: ep.ep_bitmap_encode(cfg, buf.topk_idx, bm, buf.ws))
    lay = timed(lambda: ep.ep_bitmap_layout(cfg, bm, row_token, *outs, buf.ws))
    assert ep.ep_get_error(buf.ws) == ep.EP_OK
    pairs_bytes = w.T * w.k * 8
    bitmap_bytes = w.T * words * 4
    line = {"metric": "routing metadata bytes per step, bitmap against (expert, position) pairs",
            "value": bitmap_bytes, "unit": "bytes", "higher_is_better": False, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "data": "synthetic",
            "config": workload_config(w, args.payload, None, False, "fused"),
            "bitmap": {"pairs_bytes": pairs_bytes, "bitmap_bytes": bitmap_bytes,
                       "saved_frac": 1 - bitmap_bytes / pairs_bytes, "encode_us": enc, "layout_us": lay}}
    print(json.dumps(line))
    return 0


def run_combine_only(args):
    """ep_combine alone on the workload's layout, for each expert-output
    format asked for (bf16 rows, or int8 / E4M3 / int4 codes with per-row
    scales made by ep_quantize_rows*): each one CUDA graph of K launches.
    Bytes per launch: N*H*b_out (+ N*4 scales) read, T*H*2 written."""
    import torch

    from combine_warp_top_fp32_b300 import binding as ep
    from combine_warp_top_fp32_b300 import workloads

    torch.cuda.set_device(0)
    w = workloads.WORKLOADS[args.workload]
    cfg = ep.config_from_workload(w, payload=PAYLOAD_MODE[args.payload])
    d = workloads.generate(w, device="cuda")
    buf = ep.EpBuffers.allocate(cfg)
    buf.route_dispatch(d["logits"], d["x"])
    torch.cuda.synchronize()
    n_rows = int(buf.expert_off[-1].item())
    eo = d["expert_out"]
    rows, H = eo.shape
    peak, peak_src = measured_peak_gbs()

    def coded(fmt):
        if fmt == "bf16":
            return eo, None
        q = torch.empty((rows, H // 2 if fmt == "int4" else H), dtype=torch.int8 if fmt == "int8" else torch.uint8,
                        device="cuda")
        sc = torch.empty(rows, dtype=torch.float32, device="cuda")
        {"int8": ep.ep_quantize_rows, "fp8": ep.ep_quantize_rows_fp8, "int4": ep.ep_quantize_rows_int4}[fmt](eo, q, sc)
        return q, sc

    out = {}
    for fmt in args.combine_only.split(","):
        o, sc = coded(fmt)
        for _ in range(args.warmup):
            buf.combine(o, sc)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(args.steps):
                buf.combine(o, sc)
        g.replay()
        best = float("inf")
        for _ in range(3):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record()
            g.replay()
            t1.record()
            torch.cuda.synchronize()
            best = min(best, 1e3 * t0.elapsed_time(t1) / args.steps)
        if ep.ep_get_error(buf.ws) != ep.EP_OK:
            raise RuntimeError("ep_combine reported a device error")
        nbytes = int(n_rows * H * PAYLOAD_BYTES[fmt]) + (n_rows * 4 if fmt != "bf16" else 0) + w.T * H * 2
        out[fmt] = {"us": best, "bytes": nbytes, "gbs": nbytes / best / 1e3, "frac_of_" + peak_src: nbytes / best / 1e3 / peak,
                    "elements_per_s": n_rows * H / (best * 1e-6)}
    first = next(iter(out.values()))
    line = {"metric": "ep_combine alone, by expert-output format", "value": first["us"], "unit": "us per launch",
            "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "data": "synthetic",
            "config": dict(workload_config(w, args.payload, n_rows, False, "fused"), expert_out=args.combine_only,
                           path="ep_combine alone (layout from ep_route_dispatch)"),
            "combine": out}
    print(json.dumps(line))
    return 0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description="MoE dispatch+combine benchmark")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="capacity")
    ap.add_argument("--payload", choices=["int8", "bf16", "fp8", "int4"], default=None)
    ap.add_argument("--path", choices=["calls", "fused"], default="fused",
                    help="fused: ep_route_dispatch + ep_combine; calls: ep_route, ep_dispatch, ep_combine")
    ap.add_argument("--pipeline", default=None,
                    help="comma-separated chunk counts: time the chunked pipeline with stand-in GEMM experts")
    ap.add_argument("--combine-only", default=None, metavar="FMTS",
                    help="comma-separated expert-output formats (bf16,int8,fp8,int4): time ep_combine alone")
    ap.add_argument("--bitmap", action="store_true",
                    help="report the bitmap routing metadata (bytes saved, encode and layout times)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-large", action="store_true",
                    help="skip the T=131072, H=8192 record that the capacity line carries beside the headline")
    ap.add_argument("--large-steps", type=int, default=5)
    ap.add_argument("--eager", action="store_true", help="launch through the binding each step (no CUDA graph)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-int8-return", action="store_true",
                    help="skip the extra line with int8 expert outputs (int8 payload only)")
    ap.add_argument("--cpu-baseline-s", type=float, default=15.0)
    ap.add_argument("--reference-step-s", type=float, default=4.0,
                    help="longest oracle pass per reference step; the whole workload when it fits (capacity: ~2 s)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    from combine_warp_top_fp32_b300 import workloads

    w = workloads.WORKLOADS[args.workload]
    if args.payload is None:
        args.payload = "int8" if w.payloads[0] == 1 else "bf16"
    return args


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.pipeline:
        return run_pipeline(args)
    if args.bitmap:
        return run_bitmap(args)
    if args.combine_only:
        return run_combine_only(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
