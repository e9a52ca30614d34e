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

Per-tensor globals are 2^-4 for every expert and matrix.  Top-k takes the k
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


def _draw_gate(rng, E: int, H: int, I: int, lo: int = -4, hi: int = 2):
    codes = rng.integers(0, 256, size=(E, I, H // 2), dtype=np.uint8)
    scales = e4m3_byte_of_pow2(rng.integers(lo, hi + 1, size=(E, I, H // 16), dtype=np.int32))
    return codes, scales, np.full(E, GLOBAL_SCALE, dtype=np.float32)


def generate(name: str, seed: int | None = None, *, n: int | None = None, weights: bool = True,
             gated: bool = False) -> Workload:
    """Draw the named workload.  ``n`` overrides the token count (same recipe);
    ``gated`` adds gate weights (drawn last)."""
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
        up_scales = e4m3_byte_of_pow2(rng.integers(-4, 3, size=(E, I, H // 16), dtype=np.int32))
        down_codes = rng.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8)
        down_scales = e4m3_byte_of_pow2(rng.integers(-4, 3, size=(E, H, I // 16), dtype=np.int32))
    else:
        up_codes = np.zeros((0,), np.uint8)
        up_scales = down_codes = down_scales = up_codes
    dst = f32_to_bf16_bits(rng.standard_normal((n_, H), dtype=np.float32))
    g = np.full(E, GLOBAL_SCALE, dtype=np.float32)
    wl = Workload(name, n_, H, I, E, k, x, ids, w, up_codes, up_scales, down_codes, down_scales,
                  g.copy(), g.copy(), dst)
    if gated and weights:
        wl.gate_codes, wl.gate_scales, wl.gate_global = _draw_gate(rng, E, H, I)
    return wl


def small_custom(n: int, H: int, I: int, E: int, k: int, seed: int, *, bias_sigma: float = 0.0,
                 scale_exp=(-4, 2), gated: bool = False) -> Workload:
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
    up_scales = e4m3_byte_of_pow2(rng.integers(lo, hi + 1, size=(E, I, H // 16), dtype=np.int32))
    down_codes = rng.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8)
    down_scales = e4m3_byte_of_pow2(rng.integers(lo, hi + 1, size=(E, H, I // 16), dtype=np.int32))
    dst = f32_to_bf16_bits(rng.standard_normal((n, H), dtype=np.float32))
    g = np.full(E, GLOBAL_SCALE, dtype=np.float32)
    wl = Workload("custom", n, H, I, E, k, x, ids, w, up_codes, up_scales, down_codes, down_scales,
                  g.copy(), g.copy(), dst)
    if gated:
        wl.gate_codes, wl.gate_scales, wl.gate_global = _draw_gate(rng, E, H, I, lo, hi)
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
    "CONFIGS", "GLOBAL_SCALE", "Workload", "generate", "small_custom", "make_routing", "route_topk",
    "f32_to_bf16_bits", "bf16_bits_to_f32", "e4m3_byte_of_pow2", "expected_rows",
    "weight_bytes_per_expert", "l2_flush_bytes",
]
