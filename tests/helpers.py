"""Shared helpers for the parity tests: upload seeded workloads, compare to the oracle."""
import numpy as np

from nvfp4_quantized_moe_topk_gb300 import workload as W


def to_dev(a, dev):
    import torch

    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(dev)


def bf16_from_dev(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def make_layer(wl, dev, max_tokens=None, gemv_max_rows=0, stream=None, single_max_tokens=0):
    """single_max_tokens=-1 forces the multi-kernel path (routing, gather,
    streaming kernel for small experts, grouped GEMMs, combine).  A workload
    with gate weights makes a gated layer."""
    from nvfp4_quantized_moe_topk_gb300 import api

    gate = {}
    if getattr(wl, "gate_codes", None) is not None:
        gate = dict(gate_codes=to_dev(wl.gate_codes, dev), gate_scales=to_dev(wl.gate_scales, dev),
                    gate_global=to_dev(wl.gate_global, dev))
    return api.MoeLayer(wl.H, wl.I, wl.E, wl.k, wl.n if max_tokens is None else max_tokens,
                        to_dev(wl.up_codes, dev), to_dev(wl.up_scales, dev), to_dev(wl.down_codes, dev),
                        to_dev(wl.down_scales, dev), to_dev(wl.up_global, dev), to_dev(wl.down_global, dev),
                        gemv_max_rows=gemv_max_rows, single_max_tokens=single_max_tokens, stream=stream, **gate)


def run_forward(layer, wl, dev, stream=None):
    """Upload x / ids / weights / dst, run the layer, return the new dst (bf16 bits)."""
    import torch

    x = to_dev(wl.x, dev)
    ids = to_dev(wl.topk_ids, dev)
    w = to_dev(wl.topk_weights, dev)
    dst = to_dev(wl.dst, dev)
    layer.forward(x, ids, w, dst, stream=stream)
    torch.cuda.synchronize()
    return bf16_from_dev(dst)


def half_ulp_bf16(vals) -> np.ndarray:
    """Half the bf16 spacing at each (bf16-representable) value: the most a
    round-to-nearest into bf16 can move a number that lands on that value."""
    v = np.abs(np.asarray(vals, np.float64))
    _, ex = np.frexp(np.where(v > 0, v, 1.0))
    binade = np.maximum(ex - 1, -126)
    return np.where(v > 0, np.ldexp(1.0, binade - 8), np.ldexp(1.0, -134))


def layer_tolerance_check(got_bits, ref_f64, rows=None, extra=None):
    """The layer bound against the oracle's UNROUNDED fp64 result:

        |y_gpu - y_ref| <= 1e-2 * RMS(y_ref) + 1/2 ulp(y_gpu)   for every element

    y_gpu is one bf16 rounding of an fp32 result, so the half ulp is that
    rounding; the 1e-2 * RMS term is the layer's stated tolerance.  Used for
    the layer output (against ``out_f64``) and for the bf16 intermediates
    (against ``a_f64``).  ``extra`` (elementwise, same shape) widens the bound
    by the propagated intermediate rounding difference (``flip_allowance``).
    Returns (ok, max_err, rms)."""
    if not isinstance(ref_f64, np.ndarray) or ref_f64.dtype != np.float64:
        raise TypeError("layer_tolerance_check compares with the oracle's unrounded fp64 values")
    g = W.bf16_bits_to_f32(got_bits).astype(np.float64)
    r = ref_f64
    if r.shape != g.shape:
        raise ValueError(f"shape mismatch {g.shape} vs {r.shape}")
    x = 0.0 if extra is None else np.asarray(extra, np.float64)
    if rows is not None:
        g, r = g[rows], r[rows]
        if extra is not None:
            x = x[rows]
    if r.size == 0:
        return True, 0.0, 0.0
    rms = float(np.sqrt(np.mean(r * r)))
    err = np.abs(g - r)
    ok = bool(np.all(err <= 1e-2 * rms + half_ulp_bf16(g) + x))
    return ok, float(err.max()), rms


def flip_allowance(wl, a_gpu_bits, a_ref_bits, rows=None):
    """How far a one-step rounding difference in the bf16 intermediate moves
    the down rows.

    Both sides round the intermediate (relu^2, or silu * up) to bf16 once, the
    GPU from an fp32 sum and the oracle from an fp64 one; where the two sums
    straddle a rounding boundary the intermediates differ by one bf16 step
    (the intermediate check bounds that).  The down projection then carries
    the difference into its rows: |dy[r, c]| <= |g_dn,e| * sum_i |W_dn,e[c, i]|
    * |a_gpu[r, i] - a_ref[r, i]|, with W decoded by the oracle.  Returns that
    bound for every packed row [R][H] (zero where the intermediates agree) and
    its weighted sum over each token's slots [n][H], the same for the layer
    output.  ``rows``: only these packed rows are compared (others zero)."""
    import oracle

    a_g = W.bf16_bits_to_f32(a_gpu_bits).astype(np.float64)
    a_r = W.bf16_bits_to_f32(a_ref_bits).astype(np.float64)
    d = np.abs(a_g - a_r)
    if rows is not None:
        keep = np.zeros(d.shape[0], bool)
        keep[rows] = True
        d[~keep] = 0.0
    R = d.shape[0]
    E_rows = np.zeros((R, wl.H), np.float64)
    out = np.zeros((wl.n, wl.H), np.float64)
    bad = np.nonzero(d.any(axis=1))[0]
    if bad.size == 0:
        return E_rows, out
    _, _, perm, _, _ = oracle.routing(wl.topk_ids, wl.E)
    ids = np.asarray(wl.topk_ids).ravel()
    by_expert = {}
    for r in bad:
        by_expert.setdefault(int(ids[perm[r]]), []).append(int(r))
    for e, rs in by_expert.items():
        Wd = np.abs(oracle.dequant(wl.down_codes[e], wl.down_scales[e], wl.H, wl.I))
        E_rows[rs] = abs(float(wl.down_global[e])) * (d[rs] @ Wd.T)
    w = np.abs(np.asarray(wl.topk_weights, np.float64)).ravel()
    for r in bad:
        p = int(perm[r])
        out[p // wl.k] += w[p] * E_rows[r]
    return E_rows, out


def fp_tolerance_check(got, ref, extra=None):
    """|y - y_ref| <= 1e-2 * RMS(y_ref) (+ ``extra``, elementwise) for fp32
    results against fp64.  Returns (ok, max_err, rms)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if not ref.size:
        return True, 0.0, 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(got - ref)
    bound = 1e-2 * rms + (0.0 if extra is None else extra)
    return bool(np.all(err <= bound)), float(err.max()), rms
