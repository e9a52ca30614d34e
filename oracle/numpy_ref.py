"""Independent restatement of the layer in numpy fp64 -- TEST INFRASTRUCTURE ONLY.

It shares no code with ``moe_oracle.c`` and is written in the *other* form the
pages describe: the dense-masked execution that pull request #91 ("What the
profile showed", item 1) replaced, where every expert runs over every token
and a token that did not pick the expert weighs it zero.  Since gathering only
skips work whose weight is zero, this form must agree with the C oracle's
per-pair evaluation (up to fp64 summation order) -- the gather-vs-dense-masked
pin.  Decoding uses independent sources: the e2m1 value table of the OCP
Microscaling (MX) specification and torch's float8_e4m3fn conversion; the
gated form's logistic function is scipy's ``expit``.
"""
from __future__ import annotations

import numpy as np
import torch
from scipy.special import expit

# OCP MX specification, FP4 (E2M1) element values for codes 0..7; codes 8..15
# are the same magnitudes with the sign bit set.
OCP_E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e2m1_table() -> np.ndarray:
    mags = np.array(OCP_E2M1_MAGNITUDES, dtype=np.float64)
    return np.concatenate([mags, -mags])


def e4m3_values(bytes_: np.ndarray) -> np.ndarray:
    """e4m3 bytes -> fp64 through torch's float8_e4m3fn (a library decoder)."""
    t = torch.from_numpy(np.ascontiguousarray(bytes_, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] 4-bit codes, element 2i from the low nibble."""
    lo = np.bitwise_and(codes, 0x0F)
    hi = np.right_shift(codes, 4)
    return np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)


def dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """NVFP4 matrix [rows, K] in fp64 (global not applied)."""
    vals = e2m1_table()[unpack_codes(codes)]
    s = e4m3_values(scales)
    return vals * np.repeat(s, 16, axis=-1)


def bf16_round(a: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 value (ties to even), returned as fp64.

    Written independently of the C oracle: scale each value by its bf16
    spacing and use numpy's half-to-even ``round``.
    """
    a = np.asarray(a, dtype=np.float64)
    mag = np.abs(a)
    _, ex = np.frexp(np.where(mag > 0, mag, 1.0))
    binade = np.maximum(ex - 1, -126)
    q = np.ldexp(1.0, binade - 7)
    r = np.round(mag / q) * q
    return np.where(mag > 0, np.copysign(r, a), a)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """bf16-representable fp64 values -> bit patterns (exact through fp32)."""
    return (np.asarray(v, np.float64).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def moe_dense_masked(wl) -> dict:
    """Dense-masked layer: every expert over every token, weight 0 where unpicked.

    Returns the unrounded fp64 output, its bf16 rounding, and per-(token,
    expert) intermediates (relu^2, or g * logistic(g) * u for a workload with
    gate weights), rounded to bf16 ("a") and before that rounding ("a_f64").
    """
    n, H, I, E, k = wl.n, wl.H, wl.I, wl.E, wl.k
    X = bf16_bits_to_f64(wl.x)
    out = bf16_bits_to_f64(wl.dst).copy()
    mask_w = np.zeros((n, E), np.float64)
    for t in range(n):
        for j in range(k):
            e = int(wl.topk_ids[t, j])
            if 0 <= e < E:
                mask_w[t, e] += float(wl.topk_weights[t, j])
    a_all, a_raw = {}, {}
    for e in range(E):
        Wu = dequant(wl.up_codes[e], wl.up_scales[e])  # [I, H]
        Wd = dequant(wl.down_codes[e], wl.down_scales[e])  # [H, I]
        h = (X @ Wu.T) * float(wl.up_global[e])  # [n, I] over *all* tokens
        if getattr(wl, "gate_codes", None) is not None:
            Wg = dequant(wl.gate_codes[e], wl.gate_scales[e])
            gt = (X @ Wg.T) * float(wl.gate_global[e])
            a_raw[e] = gt * expit(gt) * h
        else:
            a_raw[e] = np.maximum(h, 0.0) ** 2
        a = bf16_round(a_raw[e])
        y = (a @ Wd.T) * float(wl.down_global[e])  # [n, H]
        out += mask_w[:, e:e + 1] * y
        a_all[e] = a
    return {"out_f64": out, "dst": f64_to_bf16_bits(bf16_round(out)), "a": a_all, "a_f64": a_raw}


def matvec_chain(x_bf16: np.ndarray, up_codes, up_scales, dn_codes, dn_scales, g_up: float, g_dn: float):
    """n = 1, k = 1, w = 1: two textbook matrix-vector products around relu^2."""
    x = bf16_bits_to_f64(x_bf16)
    Wu = dequant(up_codes, up_scales)
    Wd = dequant(dn_codes, dn_scales)
    a = bf16_round(np.maximum(g_up * (Wu @ x), 0.0) ** 2)
    return g_dn * (Wd @ a), a
