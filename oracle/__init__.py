"""fp64 CPU oracle for the NVFP4 MoE expert layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product (the CUDA library and its Python
binding) never imports, links or runs anything here, and this package never
imports the product: the two share only the seeded input generator, which
holds none of the layer's arithmetic.

``moe_oracle.c`` is the oracle proper (plain C, fp64, OpenMP over independent
output values); this module compiles it with gcc into ``oracle/_build/`` and
wraps it with ctypes.  ``numpy_ref`` is an independent restatement (dense-masked form,
numpy fp64) used to pin the C oracle.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_int = ctypes.c_int
_ptr = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2 -fopenmp, portable flags: x86 and Arm)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(L):
    L.or_e2m1.argtypes = [ctypes.c_uint]
    L.or_e2m1.restype = ctypes.c_double
    L.or_e4m3.argtypes = [ctypes.c_uint, ctypes.POINTER(ctypes.c_double)]
    L.or_e4m3.restype = _int
    L.or_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.or_bf16_to_double.restype = ctypes.c_double
    L.or_bf16_from_double.argtypes = [ctypes.c_double]
    L.or_bf16_from_double.restype = ctypes.c_uint16
    L.or_dequant.argtypes = [_ptr, _ptr, _i64, _i64, _ptr]
    L.or_dequant.restype = _int
    L.or_routing.argtypes = [_ptr, _i64, _int, _int, _ptr, _ptr, _ptr, _ptr]
    L.or_routing.restype = _i64
    L.or_nvfp4_matmul.argtypes = [_ptr, _ptr, _ptr, ctypes.c_double, _i64, _i64, _i64, _int, _ptr, _ptr]
    L.or_nvfp4_matmul.restype = _int
    L.or_weighted_row_sum.argtypes = [_ptr, _ptr, _ptr, _ptr, _i64, _int, _i64, _i64]
    L.or_weighted_row_sum.restype = _i64
    L.or_moe_forward.argtypes = [_i64, _int, _int, _int, _int] + [_ptr] * 14 + [_i64, _i64]
    L.or_moe_forward.restype = _int
    L.or_moe_forward_act.argtypes = [_i64, _int, _int, _int, _int] + [_ptr] * 9 + [_int] + [_ptr] * 8 + [_i64, _i64]
    L.or_moe_forward_act.restype = _int
    L.or_router_topk.argtypes = [_ptr, _ptr, _i64, _int, _int, _ptr, _ptr, _ptr]
    L.or_router_topk.restype = _int
    L.or_num_threads.argtypes = []
    L.or_num_threads.restype = _int
    return L


def lib():
    """The oracle library; a test may swap in a deliberately broken build with ``use_library``."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def build_variant(src_text: str, tag: str) -> str:
    """Compile an edited copy of the oracle source (tests plant mistakes this way)."""
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_BUILD, f"variant_{tag}.c")
    out = os.path.join(_BUILD, f"libvariant_{tag}_{os.getpid()}.so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", src,
                    "-o", out, "-lm"], check=True)
    return out


class use_library:
    """Context manager: route every oracle call through another build of moe_oracle.c."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        lib()
        with _lock:
            self.saved = _lib
            _lib = _bind(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _p(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ formats
def e2m1(code: int) -> float:
    return lib().or_e2m1(code)


def e4m3(byte: int) -> float | None:
    """Decoded value, or None for the NaN bytes 0x7F / 0xFF."""
    v = ctypes.c_double()
    return None if lib().or_e4m3(byte, ctypes.byref(v)) != 0 else v.value


def bf16_to_double(bits: int) -> float:
    return lib().or_bf16_to_double(bits)


def bf16_from_double(v: float) -> int:
    return int(lib().or_bf16_from_double(float(v)))


def dequant(codes: np.ndarray, scales: np.ndarray, rows: int, K: int) -> np.ndarray:
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    out = np.empty((rows, K), np.float64)
    rc = lib().or_dequant(_p(codes), _p(scales), rows, K, _p(out))
    if rc != 0:
        raise ValueError(f"or_dequant failed ({rc})")
    return out


# ------------------------------------------------------------------ routing
def routing(ids: np.ndarray, E: int):
    """-> counts [E], offsets [E+1], perm_pair [R_kept], inv [n*k], dropped."""
    ids = _c(ids, np.int32)
    n, k = ids.shape
    R = n * k
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.full(max(R, 1), -1, np.int32)
    inv = np.empty(max(R, 1), np.int32)
    dropped = lib().or_routing(_p(ids), n, k, E, _p(counts), _p(offsets), _p(perm), _p(inv))
    if dropped < 0:
        raise ValueError(f"or_routing failed ({dropped})")
    kept = R - dropped
    return counts, offsets, perm[:kept].copy(), inv[:R].copy(), int(dropped)


# ------------------------------------------------------------------ matmul
def nvfp4_matmul(A_bf16: np.ndarray, codes: np.ndarray, scales: np.ndarray, g: float, epilogue: int):
    A_bf16 = _c(A_bf16, np.uint16)
    M, K = A_bf16.shape
    N = codes.shape[0]
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    if epilogue == 0:
        out = np.empty((M, N), np.float64)
        rc = lib().or_nvfp4_matmul(_p(A_bf16), _p(codes), _p(scales), g, M, N, K, 0, _p(out), None)
    else:
        out = np.empty((M, N), np.uint16)
        rc = lib().or_nvfp4_matmul(_p(A_bf16), _p(codes), _p(scales), g, M, N, K, 1, None, _p(out))
    if rc != 0:
        raise ValueError(f"or_nvfp4_matmul failed ({rc})")
    return out


# ---------------------------------------------------------- WeightedRowSum
def weighted_row_sum(dst_bf16: np.ndarray, src: np.ndarray, rows: np.ndarray, w: np.ndarray):
    """Returns (new dst bf16 bits, skipped count); dst is not modified."""
    dst = _c(dst_bf16, np.uint16).copy()
    src = _c(src, np.float64)
    rows = _c(rows, np.int32)
    w = _c(w, np.float32)
    n, k = rows.shape
    cols = dst.shape[1]
    skipped = lib().or_weighted_row_sum(_p(dst), _p(src), _p(rows), _p(w), n, k, cols, src.shape[0])
    return dst, int(skipped)


# ------------------------------------------------------------- whole layer
class Result:
    """Oracle output: final dst (bf16 bits), and optional intermediates.

    a_rows are the bf16 intermediates (relu^2 or silu * up) by packed row,
    a_f64 the same values before their bf16 rounding, y_rows the fp64 down
    rows, out_f64 the layer output before its final rounding."""

    def __init__(self, dst, a_rows, y_rows, out_f64, a_f64=None):
        self.dst, self.a_rows, self.y_rows, self.out_f64 = dst, a_rows, y_rows, out_f64
        self.a_f64 = a_f64


def moe_forward(wl, *, intermediates: bool = False, out_f64: bool = False,
                tok_range: tuple[int, int] | None = None) -> Result:
    """Run the layer on a ``workload.Workload``; wl.dst is not modified.

    A workload with gate weights (``wl.gate_codes`` not None) runs the gated
    (silu(gate) * up) form, otherwise relu^2."""
    n, H, I, E, k = wl.n, wl.H, wl.I, wl.E, wl.k
    x = _c(wl.x, np.uint16)
    ids = _c(wl.topk_ids, np.int32)
    w = _c(wl.topk_weights, np.float32)
    arrs = [_c(a, np.uint8) for a in (wl.up_codes, wl.up_scales, wl.down_codes, wl.down_scales)]
    ug, dg = _c(wl.up_global, np.float32), _c(wl.down_global, np.float32)
    dst = _c(wl.dst, np.uint16).copy()
    R = n * k
    a_rows = np.zeros((R, I), np.uint16) if intermediates else None
    a_f64 = np.zeros((R, I), np.float64) if intermediates else None
    y_rows = np.zeros((R, H), np.float64) if intermediates else None
    of = np.zeros((n, H), np.float64) if out_f64 else None
    t0, t1 = tok_range if tok_range is not None else (0, n)
    gated = getattr(wl, "gate_codes", None) is not None
    if gated:
        gc, gs = _c(wl.gate_codes, np.uint8), _c(wl.gate_scales, np.uint8)
        gg = _c(wl.gate_global, np.float32)
        rc = lib().or_moe_forward_act(n, H, I, E, k, _p(x), _p(ids), _p(w), *[_p(a) for a in arrs], _p(ug),
                                      _p(dg), 1, _p(gc), _p(gs), _p(gg), _p(dst), _p(a_rows), _p(a_f64), _p(y_rows),
                                      _p(of), t0, t1)
    else:
        rc = lib().or_moe_forward(n, H, I, E, k, _p(x), _p(ids), _p(w), *[_p(a) for a in arrs], _p(ug), _p(dg),
                                  _p(dst), _p(a_rows), _p(a_f64), _p(y_rows), _p(of), t0, t1)
    if rc != 0:
        raise ValueError(f"or_moe_forward failed ({rc})")
    return Result(dst, a_rows, y_rows, of, a_f64)


def router_topk(logits: np.ndarray, bias: np.ndarray | None, k: int):
    """(ids int32 [n,k], weights fp32 [n,k], counts int32 [E]) of the router."""
    logits = _c(logits, np.float32)
    n, E = logits.shape
    b = None if bias is None else _c(bias, np.float32)
    ids = np.zeros((n, k), np.int32)
    w = np.zeros((n, k), np.float32)
    counts = np.zeros(E, np.int32)
    rc = lib().or_router_topk(_p(logits), _p(b), n, E, k, _p(ids), _p(w), _p(counts))
    if rc != 0:
        raise ValueError(f"or_router_topk failed ({rc})")
    return ids, w, counts


def num_threads() -> int:
    return int(lib().or_num_threads())
