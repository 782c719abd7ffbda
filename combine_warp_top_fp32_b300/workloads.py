"""Seeded synthetic workloads for MoE expert-parallel dispatch/combine.

This module holds the five workload shapes and the seeded generators that both
the CUDA path and the CPU oracle consume. It holds none of the method's
arithmetic (no routing, counting, quantisation or combining) and imports
neither the CUDA binding nor the oracle.

Recipe (one ``torch.Generator`` per call, seeded with the workload's seed;
every draw is made in this order):

1. ``bias[E] = sigma_bias * N(0,1)`` — one per expert, drawn before the logits
   (only when ``sigma_bias > 0``);
2. ``logits[T,E] = N(0,1) + bias`` in fp32;
3. ``x[T,H]`` in bf16: ``N(0,1)``, or for ``decode-latency`` a Student-t with
   3 degrees of freedom scaled by 0.5, built as ``z0 / sqrt((z1²+z2²+z3²)/3)``
   from four standard normals (heavy tails stress the per-token int8 scale);
4. ``expert_out[max_rows,H]`` in bf16 ``N(0,1)`` — the synthetic expert
   outputs that the combine gathers (identity-free: they are not the payload).

"N(0,s)" means standard deviation s. Generated values depend on the device
(CPU and CUDA generators draw different streams), so a test generates once
and copies the same bytes to the other side.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

PAYLOAD_BF16 = 0
PAYLOAD_INT8 = 1


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    R: int
    capacity_factor: float  # <= 0: dropless
    payloads: tuple  # payload modes exercised by this workload
    seed: int
    x_dist: str = "normal"  # "normal" | "student_t3_half"
    sigma_bias: float = 0.0
    renormalize: bool = False
    notes: str = field(default="", compare=False)

    def capacity(self) -> int:
        """Per-expert cap ceil(cf*T*k/E) evaluated in double; T when dropless."""
        if not self.capacity_factor > 0:
            return self.T
        return int(math.ceil(float(self.capacity_factor) * self.T * self.k / self.E))

    def max_rows(self) -> int:
        """Upper bound on dispatched rows: T*k, or min(T*k, E*cap) with a cap."""
        if not self.capacity_factor > 0:
            return self.T * self.k
        return min(self.T * self.k, self.E * self.capacity())

    def replace(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The five shapes: a tiny case that the oracle finishes instantly, a decode
# step with heavy-tailed activations, a mid prefill, a capacity-limited batch
# (the headline shape T=16384, H=4096) and a large all-to-all
# (T=131072, H=8192, k=8: 17.2 GB per direction in bf16).
WORKLOADS = {
    "tiny": Workload("tiny", T=256, H=512, E=8, k=2, R=2, capacity_factor=0.0,
                     payloads=(PAYLOAD_BF16,), seed=0),
    "decode-latency": Workload("decode-latency", T=128, H=7168, E=256, k=8, R=64, capacity_factor=0.0,
                               payloads=(PAYLOAD_INT8,), seed=1, x_dist="student_t3_half", sigma_bias=0.5),
    "prefill-mid": Workload("prefill-mid", T=4096, H=2048, E=64, k=6, R=8, capacity_factor=0.0,
                            payloads=(PAYLOAD_BF16, PAYLOAD_INT8), seed=2, sigma_bias=1.0),
    "capacity": Workload("capacity", T=16384, H=4096, E=128, k=8, R=8, capacity_factor=1.25,
                         payloads=(PAYLOAD_INT8,), seed=3, sigma_bias=1.0),
    "large": Workload("large", T=131072, H=8192, E=256, k=8, R=8, capacity_factor=0.0,
                      payloads=(PAYLOAD_BF16, PAYLOAD_INT8), seed=4, sigma_bias=0.5),
}

HEADLINE = "capacity"


def _randn(gen: torch.Generator, shape, device, dtype=torch.float32) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, device=device, dtype=dtype)


def generate_logits(w: Workload, gen: torch.Generator, device) -> torch.Tensor:
    if w.sigma_bias > 0:
        bias = _randn(gen, (w.E,), device) * w.sigma_bias
    else:
        bias = None
    logits = _randn(gen, (w.T, w.E), device)
    if bias is not None:
        logits += bias
    return logits


def generate_x(w: Workload, gen: torch.Generator, device, chunk_rows: int = 8192) -> torch.Tensor:
    x = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=device)
    for r0 in range(0, w.T, chunk_rows):
        r1 = min(w.T, r0 + chunk_rows)
        if w.x_dist == "normal":
            x[r0:r1] = _randn(gen, (r1 - r0, w.H), device).to(torch.bfloat16)
        elif w.x_dist == "student_t3_half":
            z = _randn(gen, (4, r1 - r0, w.H), device)
            t3 = z[0] / torch.sqrt((z[1] * z[1] + z[2] * z[2] + z[3] * z[3]) / 3.0)
            x[r0:r1] = (0.5 * t3).to(torch.bfloat16)
        else:
            raise ValueError(f"unknown x distribution {w.x_dist!r}")
    return x


def generate_expert_out(w: Workload, gen: torch.Generator, device, rows: int | None = None,
                        chunk_rows: int = 65536) -> torch.Tensor:
    rows = w.max_rows() if rows is None else rows
    out = torch.empty((rows, w.H), dtype=torch.bfloat16, device=device)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = _randn(gen, (r1 - r0, w.H), device).to(torch.bfloat16)
    return out


def generate(w: Workload, device="cpu", seed: int | None = None, expert_out: bool = True) -> dict:
    """Draw logits, x and (optionally) expert outputs for workload ``w``."""
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    d = {"logits": generate_logits(w, gen, device), "x": generate_x(w, gen, device)}
    if expert_out:
        d["expert_out"] = generate_expert_out(w, gen, device)
    return d


def bf16_bits(t: torch.Tensor):
    """View a bf16 tensor's storage as uint16 numpy bits (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
