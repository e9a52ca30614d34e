"""Thin ctypes binding of libmoe_nvfp4 (see include/moe_nvfp4.h for the contract).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are torch tensors (device memory and streams come from
PyTorch); their ``data_ptr()`` and the current CUDA stream are passed through.
The library is loaded on first use and a missing build raises immediately --
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CAPACITY",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_BAD_ROUTING", 6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_NO_DEVICE"}
DEVFLAG_BAD_ROUTING = 0x1
DEVFLAG_TIMEOUT = 0x2

# every entry point declared in include/moe_nvfp4.h
ENTRY_POINTS = ("moe_nvfp4_status_string", "moe_nvfp4_create", "moe_nvfp4_destroy", "moe_nvfp4_forward",
                "moe_nvfp4_forward_host", "moe_nvfp4_get_device_error", "moe_nvfp4_debug_routing",
                "moe_nvfp4_debug_intermediates", "moe_nvfp4_set_timing", "moe_nvfp4_kernel_times",
                "nvfp4_matmul", "weighted_row_sum", "moe_nvfp4_forward_noalloc", "moe_router_topk",
                "moe_nvfp4_shared_expert_forward", "moe_nvfp4_debug_offset_grid_barrier")

_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status_string(status)})")


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("max_tokens", ctypes.c_int32), ("gemv_max_rows", ctypes.c_int32),
                ("single_max_tokens", ctypes.c_int32), ("activation", ctypes.c_int32)]


ACT_RELU2, ACT_SWIGLU = 0, 1


class Weights(ctypes.Structure):
    _fields_ = [("up_codes", ctypes.c_void_p), ("up_scales", ctypes.c_void_p), ("down_codes", ctypes.c_void_p),
                ("down_scales", ctypes.c_void_p), ("up_global", ctypes.c_void_p), ("down_global", ctypes.c_void_p),
                ("gate_codes", ctypes.c_void_p), ("gate_scales", ctypes.c_void_p), ("gate_global", ctypes.c_void_p)]


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libmoe_nvfp4.so; raise if it is not built (no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and not os.path.exists(path):
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libmoe_nvfp4 is not built ({path}); run __graft_entry__.build() or "
                               "python -m nvfp4_quantized_moe_topk_gb300.build")
        L = ctypes.CDLL(path)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.moe_nvfp4_status_string.argtypes = [ctypes.c_int]
        L.moe_nvfp4_status_string.restype = ctypes.c_char_p
        L.moe_nvfp4_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), vp, ctypes.POINTER(vp)]
        L.moe_nvfp4_destroy.argtypes = [vp]
        L.moe_nvfp4_forward.argtypes = [vp, vp, vp, vp, vp, i32, vp]
        L.moe_nvfp4_forward_host.argtypes = [vp, vp, vp, vp, vp, i32, vp]
        L.moe_nvfp4_shared_expert_forward.argtypes = [vp, vp, vp, i32, vp]
        L.moe_nvfp4_debug_offset_grid_barrier.argtypes = [vp, ctypes.c_int64]
        L.moe_nvfp4_get_device_error.argtypes = [vp, ctypes.POINTER(i32)]
        L.moe_nvfp4_debug_routing.argtypes = [vp, vp, vp, vp, vp, vp]
        L.moe_nvfp4_debug_intermediates.argtypes = [vp, vp, vp, vp]
        L.moe_nvfp4_set_timing.argtypes = [vp, i32]
        L.moe_nvfp4_kernel_times.argtypes = [vp, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_double),
                                             ctypes.POINTER(i64), i32, ctypes.POINTER(i32)]
        L.nvfp4_matmul.argtypes = [vp, vp, vp, ctypes.c_float, vp, i32, i32, i32, i32, vp]
        L.weighted_row_sum.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp]
        L.moe_router_topk.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp]
        L.moe_nvfp4_forward_noalloc.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), vp, vp, vp, vp,
                                                i32, vp]
        for name in ENTRY_POINTS:
            if name != "moe_nvfp4_status_string":
                getattr(L, name).restype = ctypes.c_int
        _lib = L
        return L


def status_string(status: int) -> str:
    try:
        return load().moe_nvfp4_status_string(status).decode()
    except Exception:  # pragma: no cover - only when the library itself is missing
        return STATUS.get(status, "unknown")


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream):
    import torch

    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


class MoeLayer:
    """A created layer (``moe_nvfp4_create``); weights are copied into the handle.

    Passing gate weights (``gate_codes``, ``gate_scales``, ``gate_global``)
    makes the experts gated: a = bf16(silu(gate) * up) instead of relu^2."""

    def __init__(self, hidden, inter, n_experts, top_k, max_tokens, up_codes, up_scales, down_codes, down_scales,
                 up_global, down_global, gemv_max_rows: int = 0, single_max_tokens: int = 0, stream=None,
                 gate_codes=None, gate_scales=None, gate_global=None):
        L = load()
        self.hidden, self.inter, self.n_experts, self.top_k = hidden, inter, n_experts, top_k
        self.max_tokens = max_tokens
        self.gated = gate_codes is not None
        cfg = Config(hidden, inter, n_experts, top_k, max_tokens, gemv_max_rows, single_max_tokens,
                     ACT_SWIGLU if self.gated else ACT_RELU2)
        w = Weights(_ptr(up_codes), _ptr(up_scales), _ptr(down_codes), _ptr(down_scales), _ptr(up_global),
                    _ptr(down_global), _ptr(gate_codes), _ptr(gate_scales), _ptr(gate_global))
        h = ctypes.c_void_p()
        _check(L.moe_nvfp4_create(ctypes.byref(cfg), ctypes.byref(w), _stream(stream), ctypes.byref(h)),
               "moe_nvfp4_create")
        self._h = h

    @property
    def handle(self):
        return self._h

    def forward(self, x, topk_ids, topk_weights, dst, n_tokens: int | None = None, stream=None):
        n = x.shape[0] if n_tokens is None else n_tokens
        _check(load().moe_nvfp4_forward(self._h, _ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(dst), n,
                                        _stream(stream)), "moe_nvfp4_forward")
        return dst

    def debug_offset_grid_barrier(self, arrivals: int):
        """Test hook: offset the streaming kernel's barrier count (the next
        single-launch forward then times out, bounded; see the C header)."""
        _check(load().moe_nvfp4_debug_offset_grid_barrier(self._h, int(arrivals)),
               "moe_nvfp4_debug_offset_grid_barrier")

    def shared_expert_forward(self, x, dst, n_tokens: int | None = None, stream=None):
        """dst = bf16(expert 0's FFN of x) for a 1-expert top-1 layer (the shared expert)."""
        n = x.shape[0] if n_tokens is None else n_tokens
        _check(load().moe_nvfp4_shared_expert_forward(self._h, _ptr(x), _ptr(dst), n, _stream(stream)),
               "moe_nvfp4_shared_expert_forward")
        return dst

    def forward_host(self, x, topk_ids, topk_weights, dst, n_tokens: int | None = None, stream=None):
        n = x.shape[0] if n_tokens is None else n_tokens
        _check(load().moe_nvfp4_forward_host(self._h, _ptr(x), _ptr(topk_ids), _ptr(topk_weights), _ptr(dst), n,
                                             _stream(stream)), "moe_nvfp4_forward_host")
        return dst

    def device_error(self) -> int:
        f = ctypes.c_int32()
        _check(load().moe_nvfp4_get_device_error(self._h, ctypes.byref(f)), "moe_nvfp4_get_device_error")
        return f.value

    def debug_routing(self, counts=None, offsets=None, perm_pair=None, inv=None, stream=None):
        _check(load().moe_nvfp4_debug_routing(self._h, _ptr(counts), _ptr(offsets), _ptr(perm_pair), _ptr(inv),
                                              _stream(stream)), "moe_nvfp4_debug_routing")

    def debug_intermediates(self, a_rows=None, y_rows=None, stream=None):
        _check(load().moe_nvfp4_debug_intermediates(self._h, _ptr(a_rows), _ptr(y_rows), _stream(stream)),
               "moe_nvfp4_debug_intermediates")

    def set_timing(self, enable: bool):
        _check(load().moe_nvfp4_set_timing(self._h, 1 if enable else 0), "moe_nvfp4_set_timing")

    def kernel_times(self) -> dict:
        cap = 16
        names = (ctypes.c_char_p * cap)()
        ms = (ctypes.c_double * cap)()
        launches = (ctypes.c_int64 * cap)()
        count = ctypes.c_int32()
        _check(load().moe_nvfp4_kernel_times(self._h, names, ms, launches, cap, ctypes.byref(count)),
               "moe_nvfp4_kernel_times")
        return {names[i].decode(): (ms[i], launches[i]) for i in range(min(count.value, cap))}

    def close(self):
        if getattr(self, "_h", None):
            load().moe_nvfp4_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def nvfp4_matmul(A, codes, scales, global_scale: float, C, epilogue: int, stream=None):
    M, K = A.shape
    N = codes.shape[0]
    _check(load().nvfp4_matmul(_ptr(A), _ptr(codes), _ptr(scales), float(global_scale), _ptr(C), M, N, K,
                               epilogue, _stream(stream)), "nvfp4_matmul")
    return C


def router_topk(logits, bias, topk_ids, topk_weights, counts=None, stream=None):
    """moe_router_topk: fills topk_ids [n,k] / topk_weights [n,k] (and counts [E]) from logits [n,E]."""
    n, E = logits.shape
    k = topk_ids.shape[1]
    _check(load().moe_router_topk(_ptr(logits), _ptr(bias), n, E, k, _ptr(topk_ids), _ptr(topk_weights),
                                  _ptr(counts), _stream(stream)), "moe_router_topk")
    return topk_ids, topk_weights


def weighted_row_sum(dst, src, rows, w, stream=None):
    n, cols = dst.shape
    k = rows.shape[1]
    _check(load().weighted_row_sum(_ptr(dst), _ptr(src), _ptr(rows), _ptr(w), n, k, cols, src.shape[0],
                                   _stream(stream)), "weighted_row_sum")
    return dst


def forward_noalloc(hidden, inter, n_experts, top_k, up_codes, up_scales, down_codes, down_scales, up_global,
                    down_global, x, topk_ids, topk_weights, dst, n_tokens: int | None = None, stream=None,
                    gate_codes=None, gate_scales=None, gate_global=None):
    """``moe_nvfp4_forward_noalloc``: the layer without a handle and without any
    device allocation (weights read in place; intermediates in the library's
    fixed device array).  Gate weights make the experts gated."""
    n = x.shape[0] if n_tokens is None else n_tokens
    cfg = Config(hidden, inter, n_experts, top_k, n, 0, 0, ACT_SWIGLU if gate_codes is not None else ACT_RELU2)
    w = Weights(_ptr(up_codes), _ptr(up_scales), _ptr(down_codes), _ptr(down_scales), _ptr(up_global),
                _ptr(down_global), _ptr(gate_codes), _ptr(gate_scales), _ptr(gate_global))
    _check(load().moe_nvfp4_forward_noalloc(ctypes.byref(cfg), ctypes.byref(w), _ptr(x), _ptr(topk_ids),
                                            _ptr(topk_weights), _ptr(dst), n, _stream(stream)),
           "moe_nvfp4_forward_noalloc")
    return dst
