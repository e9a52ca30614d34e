"""Seeded synthetic inputs for the NVFP4 MoE expert layer.

This module only *draws* inputs.  It holds none of the layer's arithmetic
(no dequantisation, no GEMM, no relu², no combine), so the CPU oracle and the
CUDA path can both take their inputs from it without sharing any of the
computation they are compared on.

Workloads follow the configurations the layer is specified on (tiny,
decode-1, decode-32, prefill-4314, prefill-16384).  The recipe, in draw
order, from ``numpy.random.Generator(PCG64(seed))`` with
``seed = 1000 + config index`` unless overridden:

1. ``x``: fp32 N(0,1) of shape [n, H], rounded to bf16 (round to nearest even).
2. router logits: fp32 N(0,1) of shape [n, E].
3. per-expert router bias (only where the config gives a sigma): fp32 N(0, sigma) [E],
   added to every token's logits.
4. up codes: uniform random bytes [E, I, H/2]; each byte holds two independent
   uniform 4-bit e2m1 codes (element 2i in the low nibble, 2i+1 in the high one).
5. up block-scale exponents: uniform integers in [-4, 2], shape [E, I, H/16];
   stored as the e4m3 byte of 2^u (mantissa 0).
6. down codes: uniform bytes [E, H, I/2].
7. down block-scale exponents: as 5, shape [E, H, I/16].
8. ``dst`` (the pre-filled shared-expert output): fp32 N(0,1) [n, H] -> bf16.

Gated (silu(gate) * up) workloads draw, after all of the above and from the
same generator, 9. gate codes [E, I, H/2] and 10. gate scale exponents
[E, I, H/16] as in 4 and 5, so the draws 1-8 are the same with or without a
gate.

Per-tensor globals are 2^-4 for every expert and matrix.

Parity tests also draw the weights over the whole NVFP4 contract rather than
the configs' narrow recipe (``scales=`` and ``globals=`` of ``small_custom``
and ``generate``): block scales uniform over every finite E4M3FN byte of both
signs (``"full"``: zero, subnormals, every mantissa), or over the bytes whose
exponent field is 0..3 (``"low"``: zero, all subnormals and the smallest
normals of both signs, so that the subnormal scales carry a large share of the
result), and one fp32 global per (expert, matrix), all different and none a
power of two (``"distinct"``).  The distinct globals are drawn after every
other array (up, then down, then gate), so a workload's codes, routing and
activations do not depend on the globals chosen.

Top-k takes the k
largest biased logits of each token (ties to the lower expert index) in
descending order; the k routing weights are a softmax over those k biased
logits, computed in fp64 on the host and stored as fp32.  That routing is the
step *before* the layer: the layer takes ``topk_ids``/``topk_weights`` as given.
"""
from __future__ import annotations

import dataclasses

import numpy as np

# name -> shape parameters.  "index" is the position in the specified config
# list (it fixes the default seed); "bias_sigma" skews the routing.
CONFIGS = {
    "tiny": dict(index=0, n=32, H=256, I=128, E=8, k=2, bias_sigma=0.0),
    "decode-1": dict(index=1, n=1, H=2688, I=1856, E=128, k=6, bias_sigma=0.0),
    "decode-32": dict(index=2, n=32, H=2688, I=1856, E=128, k=6, bias_sigma=0.0),
    "prefill-4314": dict(index=3, n=4314, H=2688, I=1856, E=128, k=6, bias_sigma=1.5),
    "prefill-16384": dict(index=4, n=16384, H=4096, I=2048, E=128, k=8, bias_sigma=2.0),
}

GLOBAL_SCALE = 2.0 ** -4


@dataclasses.dataclass
class Workload:
    """One seeded instance of the layer's inputs (host numpy arrays)."""

    name: str
    n: int
    H: int
    I: int
    E: int
    k: int
    x: np.ndarray  # uint16 [n, H] (bf16 bit patterns)
    topk_ids: np.ndarray  # int32 [n, k]
    topk_weights: np.ndarray  # float32 [n, k]
    up_codes: np.ndarray  # uint8 [E, I, H/2]
    up_scales: np.ndarray  # uint8 [E, I, H/16]  (e4m3 bytes)
    down_codes: np.ndarray  # uint8 [E, H, I/2]
    down_scales: np.ndarray  # uint8 [E, H, I/16]
    up_global: np.ndarray  # float32 [E]
    down_global: np.ndarray  # float32 [E]
    dst: np.ndarray  # uint16 [n, H] (bf16 bit patterns), the pre-filled output
    gate_codes: np.ndarray | None = None  # uint8 [E, I, H/2] (gated workloads only)
    gate_scales: np.ndarray | None = None  # uint8 [E, I, H/16]
    gate_global: np.ndarray | None = None  # float32 [E]

    @property
    def gated(self) -> bool:
        return self.gate_codes is not None

    @property
    def R(self) -> int:
        return self.n * self.k


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact widening)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def e4m3_byte_of_pow2(u: np.ndarray) -> np.ndarray:
    """e4m3 (E4M3FN, bias 7) byte of 2^u for integer u in [-6, 8] (normal range)."""
    return ((np.asarray(u, dtype=np.int32) + 7) << 3).astype(np.uint8)


SCALE_MODES = ("pow2", "full", "low")
GLOBAL_MODES = ("const", "distinct")


def draw_scales(rng, shape, mode: str = "pow2", exp_range=(-4, 2)) -> np.ndarray:
    """e4m3 block-scale bytes of the given shape.

    ``pow2``: 2^u with u a uniform integer in ``exp_range`` (the configs' recipe);
    ``full``: uniform over all 254 finite E4M3FN bytes (every byte but the
    NaNs 0x7F and 0xFF); ``low``: uniform over the 64 bytes whose exponent
    field is 0..3, both signs."""
    if mode == "pow2":
        lo, hi = exp_range
        return e4m3_byte_of_pow2(rng.integers(lo, hi + 1, size=shape, dtype=np.int32))
    if mode == "full":
        i = rng.integers(0, 254, size=shape, dtype=np.int32)
        return np.where(i < 0x7F, i, i + 1).astype(np.uint8)  # skip 0x7F; 253 -> 0xFE
    if mode == "low":
        i = rng.integers(0, 64, size=shape, dtype=np.int32)  # sign | exponent 0..3 | mantissa
        return (((i >> 5) << 7) | (i & 31)).astype(np.uint8)
    raise ValueError(f"unknown scale mode {mode!r}")


def draw_globals(rng, E: int, base: float) -> np.ndarray:
    """One fp32 global per expert: base * u, u uniform in [0.5, 2), never a power of two."""
    g = (np.float64(base) * rng.uniform(0.5, 2.0, size=E)).astype(np.float32)
    m, _ = np.frexp(g.astype(np.float64))
    g = np.where(m == 0.5, np.float32(base) * np.float32(1.375), g).astype(np.float32)
    return g


def global_base(scales: str) -> float:
    """Global magnitude that keeps the layer output well above the N(0,1) dst
    for the given scale distribution (small scales need larger globals)."""
    return 4.0 if scales == "low" else GLOBAL_SCALE


def _apply_globals(wl, rng, globals_: str, scales: str):
    if globals_ == "const":
        return
    if globals_ != "distinct":
        raise ValueError(f"unknown globals mode {globals_!r}")
    base = global_base(scales)
    wl.up_global = draw_globals(rng, wl.E, base)
    wl.down_global = draw_globals(rng, wl.E, base)
    if wl.gate_codes is not None:
        wl.gate_global = draw_globals(rng, wl.E, base)


def route_topk(logits: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """Top-k by descending logit (ties to the lower index), softmax over the k picked.

    This is the router that *precedes* the layer; the layer consumes its output.
    """
    n, E = logits.shape
    order = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :k]
    picked = np.take_along_axis(logits.astype(np.float64), order, axis=1)
    z = picked - picked.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    return order.astype(np.int32), p.astype(np.float32)


def make_routing(n: int, E: int, k: int, bias_sigma: float, seed: int) -> tuple[np.ndarray, np.ndarray]:
    """Routing only (ids, weights) from its own seed: used to rotate routings in timing."""
    rng = np.random.Generator(np.random.PCG64(seed))
    logits = rng.standard_normal((n, E), dtype=np.float32)
    if bias_sigma > 0:
        logits = logits + (rng.standard_normal(E, dtype=np.float32) * np.float32(bias_sigma))[None, :]
    return route_topk(logits, k)


def _draw_gate(rng, E: int, H: int, I: int, lo: int = -4, hi: int = 2, scales: str = "pow2"):
    codes = rng.integers(0, 256, size=(E, I, H // 2), dtype=np.uint8)
    sc = draw_scales(rng, (E, I, H // 16), scales, (lo, hi))
    return codes, sc, np.full(E, GLOBAL_SCALE, dtype=np.float32)


def generate(name: str, seed: int | None = None, *, n: int | None = None, weights: bool = True,
             gated: bool = False, scales: str = "pow2", globals_: str = "const") -> Workload:
    """Draw the named workload.  ``n`` overrides the token count (same recipe);
    ``gated`` adds gate weights (drawn last); ``scales`` / ``globals_`` widen
    the weight draws (see the module docstring; the defaults are the configs'
    recipe)."""
    cfg = dict(CONFIGS[name])
    if n is not None:
        cfg["n"] = int(n)
    if seed is None:
        seed = 1000 + cfg["index"]
    n_, H, I, E, k = cfg["n"], cfg["H"], cfg["I"], cfg["E"], cfg["k"]
    rng = np.random.Generator(np.random.PCG64(seed))
    x = f32_to_bf16_bits(rng.standard_normal((n_, H), dtype=np.float32))
    logits = rng.standard_normal((n_, E), dtype=np.float32)
    if cfg["bias_sigma"] > 0:
        logits = logits + (rng.standard_normal(E, dtype=np.float32) * np.float32(cfg["bias_sigma"]))[None, :]
    ids, w = route_topk(logits, k)
    if weights:
        up_codes = rng.integers(0, 256, size=(E, I, H // 2), dtype=np.uint8)
        up_scales = draw_scales(rng, (E, I, H // 16), scales)
        down_codes = rng.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8)
        down_scales = draw_scales(rng, (E, H, I // 16), scales)
    else:
        up_codes = np.zeros((0,), np.uint8)
        up_scales = down_codes = down_scales = up_codes
    dst = f32_to_bf16_bits(rng.standard_normal((n_, H), dtype=np.float32))
    g = np.full(E, GLOBAL_SCALE, dtype=np.float32)
    wl = Workload(name, n_, H, I, E, k, x, ids, w, up_codes, up_scales, down_codes, down_scales,
                  g.copy(), g.copy(), dst)
    if gated and weights:
        wl.gate_codes, wl.gate_scales, wl.gate_global = _draw_gate(rng, E, H, I, scales=scales)
    if weights:
        _apply_globals(wl, rng, globals_, scales)
    return wl


def small_custom(n: int, H: int, I: int, E: int, k: int, seed: int, *, bias_sigma: float = 0.0,
                 scale_exp=(-4, 2), gated: bool = False, scales: str = "pow2",
                 globals_: str = "const") -> Workload:
    """Same recipe at arbitrary (small) shapes, for parity and edge-case tests."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = f32_to_bf16_bits(rng.standard_normal((n, H), dtype=np.float32))
    logits = rng.standard_normal((n, E), dtype=np.float32)
    if bias_sigma > 0:
        logits = logits + (rng.standard_normal(E, dtype=np.float32) * np.float32(bias_sigma))[None, :]
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    ids, w = route_topk(logits, k)
    lo, hi = scale_exp
    up_codes = rng.integers(0, 256, size=(E, I, H // 2), dtype=np.uint8)
    up_scales = draw_scales(rng, (E, I, H // 16), scales, (lo, hi))
    down_codes = rng.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8)
    down_scales = draw_scales(rng, (E, H, I // 16), scales, (lo, hi))
    dst = f32_to_bf16_bits(rng.standard_normal((n, H), dtype=np.float32))
    g = np.full(E, GLOBAL_SCALE, dtype=np.float32)
    wl = Workload("custom", n, H, I, E, k, x, ids, w, up_codes, up_scales, down_codes, down_scales,
                  g.copy(), g.copy(), dst)
    if gated:
        wl.gate_codes, wl.gate_scales, wl.gate_global = _draw_gate(rng, E, H, I, lo, hi, scales)
    _apply_globals(wl, rng, globals_, scales)
    return wl


def expected_rows(name: str) -> int:
    c = CONFIGS[name]
    return c["n"] * c["k"]


def weight_bytes_per_expert(H: int, I: int, gated: bool = False) -> int:
    """Packed NVFP4 bytes of one expert's matrices (codes + block scales): up and
    down, plus the gate when gated."""
    return (3 if gated else 2) * (H * I // 2 + H * I // 16)


def l2_flush_bytes() -> int:
    """A write larger than the 129 MB L2 (twice it, rounded)."""
    return 256 * 1024 * 1024


__all__ = [
    "CONFIGS", "GLOBAL_SCALE", "SCALE_MODES", "GLOBAL_MODES", "Workload", "generate", "small_custom",
    "make_routing", "route_topk", "draw_scales", "draw_globals", "global_base",
    "f32_to_bf16_bits", "bf16_bits_to_f32", "e4m3_byte_of_pow2", "expected_rows",
    "weight_bytes_per_expert", "l2_flush_bytes",
]
