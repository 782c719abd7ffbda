"""ctypes binding of libep_b300 (the C ABI in include/ep.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. The entry points keep the C names (``ep_route``, ``ep_dispatch``,
``ep_combine``, ...) and take torch CUDA tensors; a non-OK status raises
:class:`EpError`. If the library has not been built this module raises on
import — there is no fallback path.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from pathlib import Path

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libep_b300.so"

EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_WORKSPACE = 2
EP_ERR_CUDA = 3
EP_ERR_TIMEOUT = 4
EP_ERR_DEVICE_INDEX = 5

EP_PAYLOAD_BF16 = 0
EP_PAYLOAD_INT8 = 1
EP_PAYLOAD_FP8 = 2  # FP8 E4M3 codes (bytes) + one fp32 scale per row
EP_PAYLOAD_INT4 = 3  # 4-bit codes, two per byte ([rows, H/2] bytes) + one fp32 scale per row

# Every symbol include/ep.h declares.
EXPORTS = (
    "ep_status_string", "ep_config_check", "ep_capacity", "ep_max_rows", "ep_workspace_size",
    "ep_workspace_init", "ep_route", "ep_dispatch", "ep_combine", "ep_quantize_rows", "ep_get_error",
    "ep_load_stats", "ep_dispatch_static", "ep_route_dispatch", "ep_quantize_rows_fp8", "ep_bitmap_encode",
    "ep_bitmap_layout", "ep_quantize_rows_int4", "ep_debug_set", "ep_route_dispatch_kernels",
)


def _header_constant(name: str) -> int:
    """An integer #define of include/ep.h (an expression of integer literals)."""
    import re

    text = (_PKG.parent / "include" / "ep.h").read_text()
    m = re.search(rf"#define\s+{name}\s+\(([0-9u*+ ]+)\)", text)
    if m is None:
        raise ImportError(f"{name} not found in include/ep.h")
    value = 1
    for factor in m.group(1).replace("u", "").split("*"):
        value *= int(factor)
    return value


# Size of ep_dispatch_static's fixed scratch array.
EP_STATIC_SCRATCH_BYTES = _header_constant("EP_STATIC_SCRATCH_BYTES")


class EpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {ep_status_string(status)} (status {status})")


class ep_config_t(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("R", ctypes.c_int32), ("capacity_factor", ctypes.c_float), ("renormalize", ctypes.c_int32),
                ("payload", ctypes.c_int32)]

    def __repr__(self):
        return (f"ep_config_t(T={self.T}, H={self.H}, E={self.E}, k={self.k}, R={self.R}, "
                f"capacity_factor={self.capacity_factor}, renormalize={self.renormalize}, payload={self.payload})")


class ep_load_stats_t(ctypes.Structure):
    _fields_ = [("mean", ctypes.c_double), ("stddev", ctypes.c_double), ("cv", ctypes.c_double),
                ("min", ctypes.c_int32), ("max", ctypes.c_int32), ("total", ctypes.c_int64)]


def _load():
    if not LIB_PATH.exists():
        raise ImportError(f"{LIB_PATH.name} is not built; run `python -m combine_warp_top_fp32_b300.build` "
                          "(the CUDA library is required: there is no CPU fallback)")
    lib = ctypes.CDLL(str(LIB_PATH))
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    CFG = ctypes.POINTER(ep_config_t)
    lib.ep_status_string.argtypes = [ctypes.c_int]
    lib.ep_status_string.restype = ctypes.c_char_p
    lib.ep_config_check.argtypes = [CFG]
    lib.ep_capacity.argtypes = [CFG, ctypes.POINTER(I32)]
    lib.ep_max_rows.argtypes = [CFG]
    lib.ep_max_rows.restype = I64
    lib.ep_workspace_size.argtypes = [CFG, ctypes.POINTER(SZ)]
    lib.ep_workspace_init.argtypes = [P, SZ, P]
    lib.ep_route.argtypes = [CFG, P, P, P, P]
    lib.ep_dispatch.argtypes = [CFG, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]
    lib.ep_combine.argtypes = [CFG, P, P, I32, P, P, P, P, SZ, P]
    lib.ep_quantize_rows.argtypes = [P, I64, I32, P, P, P]
    lib.ep_quantize_rows_fp8.argtypes = [P, I64, I32, P, P, P]
    lib.ep_quantize_rows_int4.argtypes = [P, I64, I32, P, P, P]
    lib.ep_bitmap_encode.argtypes = [CFG, P, P, P, SZ, P]
    lib.ep_bitmap_layout.argtypes = [CFG, P, P, P, P, P, P, P, P, SZ, P]
    lib.ep_get_error.argtypes = [P, SZ, P]
    lib.ep_load_stats.argtypes = [P, I32, ctypes.POINTER(ep_load_stats_t)]
    lib.ep_dispatch_static.argtypes = [CFG, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.ep_route_dispatch.argtypes = [CFG, P, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]
    lib.ep_debug_set.argtypes = [I32, I32]
    lib.ep_route_dispatch_kernels.argtypes = [CFG, ctypes.POINTER(I32)]
    for name in EXPORTS:
        if name not in ("ep_status_string", "ep_max_rows"):
            getattr(lib, name).restype = ctypes.c_int
    return lib


lib = _load()


def ep_status_string(status: int) -> str:
    return lib.ep_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != EP_OK:
        raise EpError(status, where)


def make_config(T, H, E, k, R, capacity_factor=0.0, renormalize=False, payload=EP_PAYLOAD_BF16) -> ep_config_t:
    return ep_config_t(int(T), int(H), int(E), int(k), int(R), float(capacity_factor), int(bool(renormalize)),
                       int(payload))


def config_from_workload(w, payload=None, renormalize=None) -> ep_config_t:
    return make_config(w.T, w.H, w.E, w.k, w.R, w.capacity_factor,
                       w.renormalize if renormalize is None else renormalize,
                       w.payloads[0] if payload is None else payload)


# bf16 rows, int8 codes, FP8 E4M3 codes (as bytes or as torch.float8_e4m3fn)
_PAYLOAD_DTYPES = (torch.bfloat16, torch.int8, torch.uint8, torch.float8_e4m3fn)


def payload_kind(t: torch.Tensor, H: int | None = None) -> int:
    """EP_PAYLOAD_* of a payload / expert-output tensor from its dtype (and,
    for bytes, its width: H/2 columns are packed int4, H columns E4M3)."""
    if t.dtype == torch.bfloat16:
        return EP_PAYLOAD_BF16
    if t.dtype == torch.int8:
        return EP_PAYLOAD_INT8
    if t.dtype == torch.float8_e4m3fn:
        return EP_PAYLOAD_FP8
    if t.dtype == torch.uint8:
        return EP_PAYLOAD_INT4 if H is not None and t.shape[-1] * 2 == H else EP_PAYLOAD_FP8
    raise ValueError(f"unsupported payload dtype {t.dtype}")


def _ptr(t: torch.Tensor | None, dtype=None, what=""):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what}: expected a contiguous tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{what}: expected {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


# ---- host-only queries ------------------------------------------------------
def ep_config_check(cfg: ep_config_t) -> int:
    return lib.ep_config_check(ctypes.byref(cfg))


def ep_capacity(cfg: ep_config_t) -> int:
    cap = ctypes.c_int32()
    _check(lib.ep_capacity(ctypes.byref(cfg), ctypes.byref(cap)), "ep_capacity")
    return cap.value


def ep_max_rows(cfg: ep_config_t) -> int:
    return int(lib.ep_max_rows(ctypes.byref(cfg)))


def ep_route_dispatch_kernels(cfg: ep_config_t) -> int:
    """Kernels ep_route_dispatch launches for cfg on the current device."""
    n = ctypes.c_int32()
    _check(lib.ep_route_dispatch_kernels(ctypes.byref(cfg), ctypes.byref(n)), "ep_route_dispatch_kernels")
    return n.value


def ep_workspace_size(cfg: ep_config_t) -> int:
    n = ctypes.c_size_t()
    _check(lib.ep_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "ep_workspace_size")
    return n.value


def ep_load_stats(counts) -> dict:
    import numpy as np

    c = np.ascontiguousarray(np.asarray(counts, dtype=np.int32))
    out = ep_load_stats_t()
    _check(lib.ep_load_stats(c.ctypes.data_as(ctypes.c_void_p), int(c.shape[0]), ctypes.byref(out)),
           "ep_load_stats")
    return dict(mean=out.mean, stddev=out.stddev, cv=out.cv, min=out.min, max=out.max, total=out.total)


# ---- device calls -------------------------------------------------------------
def ep_workspace_init(ws: torch.Tensor, stream=None):
    _check(lib.ep_workspace_init(_ptr(ws, what="ws"), ws.numel() * ws.element_size(), _stream(stream)),
           "ep_workspace_init")


def ep_route(cfg, logits, topk_idx, topk_w, stream=None):
    _check(lib.ep_route(ctypes.byref(cfg), _ptr(logits, torch.float32, "logits"),
                        _ptr(topk_idx, torch.int32, "topk_idx"), _ptr(topk_w, torch.float32, "topk_w"),
                        _stream(stream)), "ep_route")


def ep_dispatch(cfg, x, topk_idx, payload, scales, row_slot, slot_row, expert_counts, expert_raw, expert_off,
                rank_off, n_dropped, ws, stream=None):
    _check(lib.ep_dispatch(ctypes.byref(cfg), _ptr(x, torch.bfloat16, "x"), _ptr(topk_idx, torch.int32, "topk_idx"),
                           _ptr(payload, _PAYLOAD_DTYPES, "payload"),
                           _ptr(scales, torch.float32, "scales"), _ptr(row_slot, torch.int32, "row_slot"),
                           _ptr(slot_row, torch.int32, "slot_row"), _ptr(expert_counts, torch.int32, "expert_counts"),
                           _ptr(expert_raw, torch.int32, "expert_raw"), _ptr(expert_off, torch.int32, "expert_off"),
                           _ptr(rank_off, torch.int32, "rank_off"), _ptr(n_dropped, torch.int32, "n_dropped"),
                           _ptr(ws, what="ws"), ws.numel() * ws.element_size(), _stream(stream)), "ep_dispatch")


def ep_route_dispatch(cfg, logits, x, topk_idx, topk_w, payload, scales, row_slot, slot_row, expert_counts,
                      expert_raw, expert_off, rank_off, n_dropped, ws, stream=None):
    _check(lib.ep_route_dispatch(ctypes.byref(cfg), _ptr(logits, torch.float32, "logits"),
                                 _ptr(x, torch.bfloat16, "x"), _ptr(topk_idx, torch.int32, "topk_idx"),
                                 _ptr(topk_w, torch.float32, "topk_w"),
                                 _ptr(payload, _PAYLOAD_DTYPES, "payload"),
                                 _ptr(scales, torch.float32, "scales"), _ptr(row_slot, torch.int32, "row_slot"),
                                 _ptr(slot_row, torch.int32, "slot_row"),
                                 _ptr(expert_counts, torch.int32, "expert_counts"),
                                 _ptr(expert_raw, torch.int32, "expert_raw"),
                                 _ptr(expert_off, torch.int32, "expert_off"), _ptr(rank_off, torch.int32, "rank_off"),
                                 _ptr(n_dropped, torch.int32, "n_dropped"), _ptr(ws, what="ws"),
                                 ws.numel() * ws.element_size(), _stream(stream)), "ep_route_dispatch")


def ep_combine(cfg, expert_out, out_scales, out_payload, slot_row, topk_w, y, ws, stream=None):
    _check(lib.ep_combine(ctypes.byref(cfg), _ptr(expert_out, _PAYLOAD_DTYPES, "expert_out"),
                          _ptr(out_scales, torch.float32, "out_scales"), int(out_payload),
                          _ptr(slot_row, torch.int32, "slot_row"), _ptr(topk_w, torch.float32, "topk_w"),
                          _ptr(y, torch.bfloat16, "y"), _ptr(ws, what="ws"), ws.numel() * ws.element_size(),
                          _stream(stream)), "ep_combine")


def ep_quantize_rows(inp, q, scales, stream=None):
    n, H = inp.shape
    _check(lib.ep_quantize_rows(_ptr(inp, torch.bfloat16, "in"), int(n), int(H), _ptr(q, torch.int8, "q"),
                                _ptr(scales, torch.float32, "scales"), _stream(stream)), "ep_quantize_rows")


def ep_quantize_rows_fp8(inp, q, scales, stream=None):
    n, H = inp.shape
    _check(lib.ep_quantize_rows_fp8(_ptr(inp, torch.bfloat16, "in"), int(n), int(H),
                                    _ptr(q, (torch.uint8, torch.float8_e4m3fn), "q"),
                                    _ptr(scales, torch.float32, "scales"), _stream(stream)), "ep_quantize_rows_fp8")


def bitmap_words(E: int) -> int:
    """32-bit words per token of an expert bitmap."""
    return (int(E) + 31) // 32


def ep_bitmap_encode(cfg, topk_idx, bitmap, ws, stream=None):
    _check(lib.ep_bitmap_encode(ctypes.byref(cfg), _ptr(topk_idx, torch.int32, "topk_idx"),
                                _ptr(bitmap, (torch.int32, torch.uint32), "bitmap"), _ptr(ws, what="ws"),
                                ws.numel() * ws.element_size(), _stream(stream)), "ep_bitmap_encode")


def ep_bitmap_layout(cfg, bitmap, row_token, expert_counts, expert_raw, expert_off, rank_off, n_dropped, ws,
                     stream=None):
    _check(lib.ep_bitmap_layout(ctypes.byref(cfg), _ptr(bitmap, (torch.int32, torch.uint32), "bitmap"),
                                _ptr(row_token, torch.int32, "row_token"),
                                _ptr(expert_counts, torch.int32, "expert_counts"),
                                _ptr(expert_raw, torch.int32, "expert_raw"),
                                _ptr(expert_off, torch.int32, "expert_off"), _ptr(rank_off, torch.int32, "rank_off"),
                                _ptr(n_dropped, torch.int32, "n_dropped"), _ptr(ws, what="ws"),
                                ws.numel() * ws.element_size(), _stream(stream)), "ep_bitmap_layout")


def ep_quantize_rows_int4(inp, q, scales, stream=None):
    n, H = inp.shape
    _check(lib.ep_quantize_rows_int4(_ptr(inp, torch.bfloat16, "in"), int(n), int(H), _ptr(q, torch.uint8, "q"),
                                     _ptr(scales, torch.float32, "scales"), _stream(stream)), "ep_quantize_rows_int4")


EP_DEBUG_FORCE_WAIT_TIMEOUT = 1
EP_DEBUG_ROUTE_DISPATCH_FORM = 2
EP_FORM_AUTO, EP_FORM_SINGLE, EP_FORM_CHAIN = 0, 1, 2


def ep_debug_set(option: int, value: int):
    """Process-wide test hooks (include/ep.h): force the single-launch form's
    device-wide wait to time out, or choose the form of ep_route_dispatch."""
    _check(lib.ep_debug_set(int(option), int(value)), "ep_debug_set")


def ep_get_error(ws, stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return lib.ep_get_error(_ptr(ws, what="ws"), ws.numel() * ws.element_size(), _stream(stream))


# ---- buffers for one configuration (plumbing: torch allocates, the library computes)
@dataclass
class EpBuffers:
    cfg: ep_config_t
    topk_idx: torch.Tensor
    topk_w: torch.Tensor
    payload: torch.Tensor
    scales: torch.Tensor | None
    row_slot: torch.Tensor
    slot_row: torch.Tensor
    expert_counts: torch.Tensor
    expert_raw: torch.Tensor
    expert_off: torch.Tensor
    rank_off: torch.Tensor
    n_dropped: torch.Tensor
    ws: torch.Tensor
    y: torch.Tensor

    @staticmethod
    def allocate(cfg: ep_config_t, device="cuda", stream=None) -> "EpBuffers":
        T, H, E, k, R = cfg.T, cfg.H, cfg.E, cfg.k, cfg.R
        rows = ep_max_rows(cfg)
        coded = cfg.payload != EP_PAYLOAD_BF16
        pdtype = {EP_PAYLOAD_BF16: torch.bfloat16, EP_PAYLOAD_INT8: torch.int8, EP_PAYLOAD_FP8: torch.uint8,
                  EP_PAYLOAD_INT4: torch.uint8}[cfg.payload]
        pcols = H // 2 if cfg.payload == EP_PAYLOAD_INT4 else H
        i32 = dict(dtype=torch.int32, device=device)
        b = EpBuffers(
            cfg=cfg,
            topk_idx=torch.empty((T, k), **i32),
            topk_w=torch.empty((T, k), dtype=torch.float32, device=device),
            payload=torch.empty((rows, pcols), dtype=pdtype, device=device),
            scales=torch.empty((rows,), dtype=torch.float32, device=device) if coded else None,
            row_slot=torch.empty((rows,), **i32),
            slot_row=torch.empty((T * k,), **i32),
            expert_counts=torch.empty((E,), **i32),
            expert_raw=torch.empty((E,), **i32),
            expert_off=torch.empty((E + 1,), **i32),
            rank_off=torch.empty((R + 1,), **i32),
            n_dropped=torch.empty((1,), **i32),
            ws=torch.empty((max(ep_workspace_size(cfg), 256),), dtype=torch.uint8, device=device),
            y=torch.empty((T, H), dtype=torch.bfloat16, device=device),
        )
        ep_workspace_init(b.ws, stream)
        return b

    def route(self, logits, stream=None):
        ep_route(self.cfg, logits, self.topk_idx, self.topk_w, stream)

    def dispatch(self, x, stream=None):
        ep_dispatch(self.cfg, x, self.topk_idx, self.payload, self.scales, self.row_slot, self.slot_row,
                    self.expert_counts, self.expert_raw, self.expert_off, self.rank_off, self.n_dropped, self.ws,
                    stream)

    def route_dispatch(self, logits, x, stream=None):
        """ep_route + ep_dispatch as one call (routing fused with the count)."""
        ep_route_dispatch(self.cfg, logits, x, self.topk_idx, self.topk_w, self.payload, self.scales, self.row_slot,
                          self.slot_row, self.expert_counts, self.expert_raw, self.expert_off, self.rank_off,
                          self.n_dropped, self.ws, stream)

    def combine(self, expert_out, out_scales=None, stream=None):
        out_payload = payload_kind(expert_out, self.cfg.H)
        ep_combine(self.cfg, expert_out, out_scales, out_payload, self.slot_row, self.topk_w, self.y, self.ws, stream)

    def step(self, logits, x, expert_out, out_scales=None, stream=None):
        """One pass of the path: route -> dispatch -> combine, all on `stream`."""
        self.route(logits, stream)
        self.dispatch(x, stream)
        self.combine(expert_out, out_scales, stream)
        return self.y
