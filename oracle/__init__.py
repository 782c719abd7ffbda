"""CPU oracle for MoE expert-parallel dispatch and combine — TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg
may import this package. The product path (the CUDA library and its binding)
never does. The arithmetic lives in ``ep_oracle.cpp`` (plain single-threaded
C++); this module only marshals numpy arrays to it through ctypes.

Functions and the passages they follow:

* :func:`route` — softmax over router logits, then top-k (MoE sparse-
  communication article, intelliparadigm.com, §2.1 Router listing).
* :func:`expert_rank` — expert e lives on rank e // (E/R) (MoE communication-
  wall explainer, juhe.plus, "64 experts on 8 GPUs" example).
* :func:`layout` — per-expert counts, capacity cap, offsets as running sums and
  the rank-major row order (NCCL EP article, hotelren.com, §3.3 flat sendbuff;
  ThunderEP on consumer GPUs, bjdmk.com.cn, §2.1 aggregation).
* :func:`quantize_rows` / :func:`payload` — per-token int8 code (ThunderEP §2.3),
  or the same per-token scheme with an FP8 E4M3 or a 4-bit code (ThunderEP
  §5.2; NCCL EP article §6.3).
* :func:`combine` — gate-weighted sum of the k expert outputs (ThunderEP §1.3).
"""
from __future__ import annotations

import ctypes
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "ep_oracle.cpp"
_LIB = _HERE / "libep_oracle.so"

# -ffp-contract=off: no fused multiply-add beyond the explicit fmaf calls.
CXXFLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(out: Path | None = None, extra_flags: list[str] | None = None) -> Path:
    """Compile ep_oracle.cpp with g++ into a shared library and return its path."""
    out = Path(out) if out is not None else _LIB
    cmd = ["g++", *CXXFLAGS, *(extra_flags or []), str(_SRC), "-o", str(out)]
    subprocess.run(cmd, check=True)
    return out


_lib = None


def _load(path: Path | None = None):
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(str(path)))
    if _lib is None:
        if not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
            build()
        _lib = _bind(ctypes.CDLL(str(_LIB)))
    return _lib


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.oracle_route.argtypes = [I, I, I, I, P, P, P]
    lib.oracle_expert_rank.argtypes = [I, I, I]
    lib.oracle_capacity.argtypes = [I, I, I, ctypes.c_float]
    lib.oracle_capacity.restype = ctypes.c_int64
    lib.oracle_layout.argtypes = [I, I, I, I, ctypes.c_float, P, P, P, P, P, P, P, P]
    lib.oracle_quantize_row.argtypes = [I, P, P, P]
    lib.oracle_quantize_rows.argtypes = [I, I, P, P, P]
    lib.oracle_payload.argtypes = [I, I, I, I, I, P, P, P, P]
    lib.oracle_dequant.argtypes = [ctypes.c_int8, ctypes.c_float]
    lib.oracle_dequant.restype = ctypes.c_float
    lib.oracle_dequant_fp8.argtypes = [ctypes.c_uint8, ctypes.c_float]
    lib.oracle_dequant_fp8.restype = ctypes.c_float
    lib.oracle_quantize_row_fp8.argtypes = [I, P, P, P]
    lib.oracle_quantize_rows_fp8.argtypes = [I, I, P, P, P]
    lib.oracle_quantize_row_int4.argtypes = [I, P, P, P]
    lib.oracle_quantize_rows_int4.argtypes = [I, I, P, P, P]
    lib.oracle_dequant_int4.argtypes = [P, I, ctypes.c_float]
    lib.oracle_dequant_int4.restype = ctypes.c_float
    lib.oracle_float_to_e4m3.argtypes = [ctypes.c_float]
    lib.oracle_float_to_e4m3.restype = ctypes.c_uint8
    lib.oracle_e4m3_to_float.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_float.restype = ctypes.c_float
    lib.oracle_combine.argtypes = [I, I, I, I, P, P, P, P, P]
    lib.oracle_combine_tokens.argtypes = [I, P, I, I, I, P, P, P, P, P]
    lib.oracle_count_cv.argtypes = [I, P]
    lib.oracle_count_cv.restype = ctypes.c_double
    lib.oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_float.restype = ctypes.c_float
    lib.oracle_float_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_float_to_bf16.restype = ctypes.c_uint16
    return lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def _out_mode(expert_out: np.ndarray) -> int:
    """Expert-output format from the array's dtype: uint16 bf16 bits, int8 codes, uint8 E4M3 codes."""
    modes = {np.dtype(np.uint16): 0, np.dtype(np.int8): 1, np.dtype(np.uint8): 2}
    if expert_out.dtype not in modes:
        raise ValueError(f"unsupported expert output dtype {expert_out.dtype}")
    return modes[expert_out.dtype]


class Oracle:
    """Thin numpy front end over one loaded copy of the oracle library."""

    def __init__(self, lib_path: Path | None = None):
        self.lib = _load(lib_path)

    # step 1
    def route(self, logits: np.ndarray, k: int, renormalize: bool = False):
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        T, E = logits.shape
        idx = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float32)
        _check(self.lib.oracle_route(T, E, k, int(bool(renormalize)), _p(logits), _p(idx), _p(w)), "route")
        return idx, w

    # step 2
    def expert_rank(self, E: int, R: int, e: int) -> int:
        r = self.lib.oracle_expert_rank(E, R, e)
        if r < 0:
            raise ValueError("bad expert/rank arguments")
        return r

    def capacity(self, T: int, E: int, k: int, capacity_factor: float) -> int:
        return int(self.lib.oracle_capacity(T, E, k, float(capacity_factor)))

    # steps 3-4
    def layout(self, idx: np.ndarray, E: int, R: int, capacity_factor: float = 0.0):
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        T, k = idx.shape
        counts = np.empty(E, np.int32)
        raw = np.empty(E, np.int32)
        eoff = np.empty(E + 1, np.int32)
        roff = np.empty(R + 1, np.int32)
        slot_row = np.empty(T * k, np.int32)
        row_slot = np.full(max(T * k, 1), -1, np.int32)
        nd = np.zeros(1, np.int32)
        _check(self.lib.oracle_layout(T, E, k, R, float(capacity_factor), _p(idx), _p(counts), _p(raw),
                                      _p(eoff), _p(roff), _p(slot_row), _p(row_slot), _p(nd)), "layout")
        N = int(eoff[E])
        return dict(expert_counts=counts, expert_raw=raw, expert_off=eoff, rank_off=roff,
                    slot_row=slot_row, row_slot=row_slot[:N].copy(), n_dropped=int(nd[0]), N=N)

    # step 5
    def quantize_rows(self, x_bits: np.ndarray, fp8: bool = False, int4: bool = False):
        """Per-row int8 codes (int8 array), E4M3 codes (uint8 array) with fp8=True,
        or packed int4 codes ([n, H/2] uint8 array) with int4=True."""
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        n, H = x_bits.shape
        s = np.empty(n, np.float32)
        if int4:
            q = np.empty((n, H // 2), np.uint8)
            _check(self.lib.oracle_quantize_rows_int4(n, H, _p(x_bits), _p(q), _p(s)), "quantize_rows_int4")
        elif fp8:
            q = np.empty((n, H), np.uint8)
            _check(self.lib.oracle_quantize_rows_fp8(n, H, _p(x_bits), _p(q), _p(s)), "quantize_rows_fp8")
        else:
            q = np.empty((n, H), np.int8)
            _check(self.lib.oracle_quantize_rows(n, H, _p(x_bits), _p(q), _p(s)), "quantize_rows")
        return q, s

    def payload(self, x_bits: np.ndarray, row_slot: np.ndarray, k: int, mode):
        """mode: 0/False bf16 bytes, 1/True int8 code, 2 FP8 E4M3 code (uint8),
        3 packed int4 code ([N, H/2] uint8)."""
        mode = int(mode)
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        row_slot = np.ascontiguousarray(row_slot, dtype=np.int32)
        T, H = x_bits.shape
        N = row_slot.shape[0]
        if mode == 1:
            pl = np.empty((N, H), np.int8)
            sc = np.empty(N, np.float32)
        elif mode == 2:
            pl = np.empty((N, H), np.uint8)
            sc = np.empty(N, np.float32)
        elif mode == 3:
            pl = np.empty((N, H // 2), np.uint8)
            sc = np.empty(N, np.float32)
        else:
            pl = np.empty((N, H), np.uint16)
            sc = None
        _check(self.lib.oracle_payload(T, H, k, N, mode, _p(x_bits), _p(row_slot), _p(pl), _p(sc)), "payload")
        return pl, sc

    def dequant(self, q: int, scale: float) -> float:
        return float(self.lib.oracle_dequant(int(q), float(scale)))

    def dequant_int4(self, q_row: np.ndarray, h: int, scale: float) -> float:
        q_row = np.ascontiguousarray(q_row, dtype=np.uint8)
        return float(self.lib.oracle_dequant_int4(_p(q_row), int(h), float(scale)))

    def dequant_fp8(self, code: int, scale: float) -> float:
        return float(self.lib.oracle_dequant_fp8(int(code), float(scale)))

    def float_to_e4m3(self, v: float) -> int:
        return int(self.lib.oracle_float_to_e4m3(float(v)))

    def e4m3_to_float(self, code: int) -> float:
        return float(self.lib.oracle_e4m3_to_float(int(code)))

    # step 7
    def combine(self, expert_out: np.ndarray, out_scales: np.ndarray | None, slot_row: np.ndarray,
                topk_w: np.ndarray, T: int, k: int, int4: bool = False):
        """int4=True: expert_out is [*, H/2] packed int4 codes (uint8)."""
        expert_out = np.ascontiguousarray(expert_out)
        H = expert_out.shape[1] * (2 if int4 else 1)
        out_mode = 3 if int4 else _out_mode(expert_out)
        slot_row = np.ascontiguousarray(slot_row, dtype=np.int32).reshape(-1)
        topk_w = np.ascontiguousarray(topk_w, dtype=np.float32).reshape(-1)
        sc = None if out_scales is None else np.ascontiguousarray(out_scales, dtype=np.float32)
        y = np.empty((T, H), np.uint16)
        _check(self.lib.oracle_combine(T, H, k, out_mode, _p(expert_out), _p(sc), _p(slot_row),
                                       _p(topk_w), _p(y)), "combine")
        return y

    def combine_tokens(self, tokens: np.ndarray, expert_out: np.ndarray, out_scales, slot_row, topk_w, k: int,
                       int4: bool = False):
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        expert_out = np.ascontiguousarray(expert_out)
        H = expert_out.shape[1] * (2 if int4 else 1)
        out_mode = 3 if int4 else _out_mode(expert_out)
        slot_row = np.ascontiguousarray(slot_row, dtype=np.int32).reshape(-1)
        topk_w = np.ascontiguousarray(topk_w, dtype=np.float32).reshape(-1)
        sc = None if out_scales is None else np.ascontiguousarray(out_scales, dtype=np.float32)
        y = np.empty((tokens.shape[0], H), np.uint16)
        _check(self.lib.oracle_combine_tokens(tokens.shape[0], _p(tokens), H, k, out_mode, _p(expert_out),
                                              _p(sc), _p(slot_row), _p(topk_w), _p(y)), "combine_tokens")
        return y

    def count_cv(self, counts: np.ndarray) -> float:
        counts = np.ascontiguousarray(counts, dtype=np.int32)
        return float(self.lib.oracle_count_cv(counts.shape[0], _p(counts)))

    def bf16_to_float(self, b: int) -> float:
        return float(self.lib.oracle_bf16_to_float(int(b)))

    def float_to_bf16(self, f: float) -> int:
        return int(self.lib.oracle_float_to_bf16(float(f)))

    # the whole pass, in the pages' order
    def forward(self, logits, x_bits, expert_out, k: int, R: int, capacity_factor: float = 0.0,
                renormalize: bool = False, payload_int8: bool = False, out_scales=None):
        T, E = logits.shape
        idx, w = self.route(logits, k, renormalize)
        lay = self.layout(idx, E, R, capacity_factor)
        pl, sc = self.payload(x_bits, lay["row_slot"], k, int(payload_int8))
        y = self.combine(expert_out, out_scales, lay["slot_row"], w, T, k)
        return dict(topk_idx=idx, topk_w=w, payload=pl, scales=sc, y=y, **lay)


def default() -> Oracle:
    return Oracle()

