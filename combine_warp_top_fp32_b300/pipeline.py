"""Chunked dispatch -> experts -> combine with communication / compute overlap.

The chunked pipeline of ThunderEP on consumer GPUs (bjdmk.com.cn, §2.2 and
the chunk_size sweep of §3.4): the batch is cut into C chunks of consecutive
tokens; every chunk is aggregated on its own (its own rank-major send buffer,
counts and capacity), so that while the experts work on chunk c the next
chunk is already being dispatched and the previous one combined. Two CUDA
streams carry the two kinds of work and CUDA events order them, with no
device-wide synchronisation (ThunderEP §2.2: event record + stream wait).

Schedule for C chunks (D = ep_route_dispatch, X = experts, K = ep_combine):

    dispatch stream:  D0 D1 K0 D2 K1 ... D(C-1) K(C-2) K(C-1)
    expert stream:       X0    X1    ...        X(C-1)

Kc waits for Xc, Xc waits for Dc; everything else is stream order. Every
kernel on the dispatch stream is the library's (argument marshalling only
here); the experts are the caller's function.

Semantics: each chunk is an independent batch for routing, capacity
(cap = ceil(cf * T_c * k / E) per chunk) and layout, as the article's
per-chunk aggregation implies. With no capacity limit the combined output of
a row-wise expert function is the same for every C.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as ep


def chunk_bounds(T: int, n_chunks: int) -> list[int]:
    """Token bounds [0, b1, ..., T] of at most n_chunks non-empty chunks of
    nearly equal size, on multiples of 4 tokens (so every chunk's fp32 logit
    rows start 16-byte aligned whatever E is); [0, 0] for an empty batch."""
    if T <= 0:
        return [0, 0]
    b = sorted({min(T, 4 * ((T * c // n_chunks + 3) // 4)) for c in range(n_chunks)} | {T})
    return b if b[0] == 0 else [0] + b


@dataclass
class Chunk:
    t0: int
    t1: int
    cfg: ep.ep_config_t
    buf: ep.EpBuffers


class ChunkedPipeline:
    """C chunks of a [T, H] batch with their own buffers (allocated once)."""

    def __init__(self, cfg: ep.ep_config_t, n_chunks: int, device="cuda"):
        if n_chunks < 1:
            raise ValueError("n_chunks must be >= 1")
        self.cfg = cfg
        T = cfg.T
        bounds = chunk_bounds(T, n_chunks)
        self.y = torch.empty((T, cfg.H), dtype=torch.bfloat16, device=device)
        self.chunks = []
        for t0, t1 in zip(bounds[:-1], bounds[1:]):
            ccfg = ep.make_config(t1 - t0, cfg.H, cfg.E, cfg.k, cfg.R, cfg.capacity_factor, cfg.renormalize,
                                  cfg.payload)
            buf = ep.EpBuffers.allocate(ccfg, device)
            buf.y = self.y[t0:t1]  # each chunk's combine writes its rows of y in place
            self.chunks.append(Chunk(t0, t1, ccfg, buf))
        self.dispatch_stream = torch.cuda.Stream(device)
        self.expert_stream = torch.cuda.Stream(device)

    def run(self, logits: torch.Tensor, x: torch.Tensor, experts):
        """One pass over the batch. `experts(buf)` is called on the expert
        stream once per chunk with that chunk's EpBuffers (payload, scales,
        counts and offsets on the device) and returns the chunk's expert
        outputs [max_rows, H] (bf16, or int8 / E4M3 codes with their scales
        as a tuple (codes, scales)). Returns y [T, H] bf16 (written on the
        dispatch stream; the caller's current stream waits for it)."""
        caller = torch.cuda.current_stream()
        ds, xs = self.dispatch_stream, self.expert_stream
        ds.wait_stream(caller)
        xs.wait_stream(caller)
        C = len(self.chunks)
        dispatched = [torch.cuda.Event() for _ in range(C)]
        computed = [torch.cuda.Event() for _ in range(C)]
        outputs = [None] * C

        def dispatch(c):
            ch = self.chunks[c]
            with torch.cuda.stream(ds):
                ch.buf.route_dispatch(logits[ch.t0:ch.t1], x[ch.t0:ch.t1])
                dispatched[c].record(ds)
            with torch.cuda.stream(xs):
                xs.wait_event(dispatched[c])
                outputs[c] = experts(ch.buf)
                computed[c].record(xs)

        def combine(c):
            ch = self.chunks[c]
            with torch.cuda.stream(ds):
                ds.wait_event(computed[c])
                eo = outputs[c]
                scales = None
                if isinstance(eo, tuple):
                    eo, scales = eo
                ch.buf.combine(eo, scales)

        dispatch(0)
        for c in range(1, C):
            dispatch(c)
            combine(c - 1)
        combine(C - 1)
        caller.wait_stream(ds)
        return self.y


def gemm_experts(weight: torch.Tensor):
    """A stand-in for the expert FFNs: every dispatched row times one [H, H]
    bf16 matrix (a plain cuBLAS GEMM through torch), on the rows [0, N) the
    dispatch wrote. Codes are widened with their row scales first. Returns
    bf16 expert outputs of the buffer's row count."""

    def run(buf: ep.EpBuffers):
        rows = buf.payload.shape[0]
        p = buf.payload
        if p.dtype == torch.bfloat16:
            a = p
        elif p.dtype == torch.int8:
            a = (p.float() * buf.scales[:, None]).to(torch.bfloat16)
        else:  # E4M3 codes
            a = (p.view(torch.float8_e4m3fn).float() * buf.scales[:, None]).to(torch.bfloat16)
        out = torch.empty((rows, weight.shape[1]), dtype=torch.bfloat16, device=p.device)
        torch.matmul(a, weight, out=out)
        return out

    return run
