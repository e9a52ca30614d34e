"""Pins for the oracle's gated (silu(gate) * up) expert form.

The gated expert is the "gate-up" kernel of "nvfp4 experts cuda: decode
kernels stall on load latency ... #2265" (section "What ncu shows": each warp
reads both rows' inputs per output).  The page does not print the activation;
the reading taken is SwiGLU, a_i = bf16(silu(g_i) * u_i) with
silu(g) = g * logistic(g).  What pins it, without re-typing the oracle:
  * textbook values of the logistic function at +-1 (``golden/silu_points.json``);
  * the limits silu(g) -> g and silu(-g) -> 0 for large g, with the up
    projection taken from the oracle's separately pinned NVFP4 matmul;
  * the identity silu(g) - silu(-g) = g (logistic(g) + logistic(-g) = 1),
    within the two bf16 roundings;
  * the independent dense-masked numpy restatement (scipy's ``expit``).
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import numpy_ref
from nvfp4_quantized_moe_topk_gb300 import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ONE_CODE, SCALE_ONE = 0x2, 0x38  # e2m1 1.0, e4m3 1.0
E2M1_CODE = {1.0: 0x2, -1.0: 0xA, 2.0: 0x4, -2.0: 0xC}


def _one_expert(n, H, I, seed=0):
    wl = W.small_custom(n, H, I, 1, 1, seed=seed, gated=True)
    wl.topk_ids[:] = 0
    wl.topk_weights[:] = 1.0
    return wl


def test_logistic_points_from_fixture():
    """g_i and u_i set exactly by one nonzero weight per row; a_i must be the
    bf16 of silu(g) * u at the textbook logistic values."""
    fx = json.load(open(os.path.join(GOLDEN, "silu_points.json")))
    H, I = 64, 32
    wl = _one_expert(1, H, I)
    x = np.zeros((1, H), np.float32)
    x[0, 0] = 1.0
    wl.x[:] = W.f32_to_bf16_bits(x)
    for arr in (wl.gate_codes, wl.up_codes):
        arr[:] = 0
    wl.gate_scales[:] = SCALE_ONE
    wl.up_scales[:] = SCALE_ONE
    wl.gate_global[:] = 1.0
    wl.up_global[:] = 1.0
    cases = fx["cases"]
    for i in range(I):
        c = cases[i % len(cases)]
        wl.gate_codes[0, i, 0] = E2M1_CODE[c["g"]]  # element 0 = low nibble of byte 0
        wl.up_codes[0, i, 0] = E2M1_CODE[c["u"]]
    res = oracle.moe_forward(wl, intermediates=True)
    for i in range(I):
        c = cases[i % len(cases)]
        assert int(res.a_rows[0, i]) == int(c["a_bf16_bits"], 16), (i, c)
        assert numpy_ref.bf16_bits_to_f64(res.a_rows[0, i]) == c["a_value"]


def _saturated_gate(sign):
    """x = 1, every gate weight 1.0, gate global 2 * sign: g = 128 * sign exactly."""
    H, I = 64, 32
    wl = _one_expert(3, H, I, seed=41)
    wl.x[:] = W.f32_to_bf16_bits(np.ones((3, H), np.float32))
    wl.gate_codes[:] = ONE_CODE | (ONE_CODE << 4)
    wl.gate_scales[:] = SCALE_ONE
    wl.gate_global[:] = 2.0 * sign
    return wl


def test_large_positive_gate_passes_the_up_projection():
    """silu(128) = 128 in fp64, so a = bf16(128 * u), u from the pinned matmul."""
    wl = _saturated_gate(+1)
    res = oracle.moe_forward(wl, intermediates=True)
    u = oracle.nvfp4_matmul(wl.x, wl.up_codes[0], wl.up_scales[0], float(wl.up_global[0]), 0)
    want = numpy_ref.bf16_round(128.0 * u)
    assert np.array_equal(numpy_ref.bf16_bits_to_f64(res.a_rows), want)
    assert np.count_nonzero(want) > 0


def test_large_negative_gate_closes_the_expert():
    """silu(-128) ~ -3e-54 underflows bf16: a = 0, the output is dst exactly."""
    wl = _saturated_gate(-1)
    res = oracle.moe_forward(wl, intermediates=True)
    assert not np.any(numpy_ref.bf16_bits_to_f64(res.a_rows))
    assert np.array_equal(res.dst, wl.dst)


def test_silu_odd_part_is_the_product():
    """silu(g) * u - silu(-g) * u = g * u; the gate negated by flipping every
    code's sign bit.  Each side carries one bf16 rounding (<= 2^-9 relative)."""
    wl = W.small_custom(4, 64, 32, 3, 2, seed=43, gated=True)
    pos = oracle.moe_forward(wl, intermediates=True)
    wl_neg = W.small_custom(4, 64, 32, 3, 2, seed=43, gated=True)
    wl_neg.gate_codes ^= 0x88
    neg = oracle.moe_forward(wl_neg, intermediates=True)
    counts, offsets, perm, inv, _ = oracle.routing(wl.topk_ids, wl.E)
    ap = numpy_ref.bf16_bits_to_f64(pos.a_rows)
    an = numpy_ref.bf16_bits_to_f64(neg.a_rows)
    for r, p in enumerate(perm):
        t, e = p // wl.k, int(wl.topk_ids.ravel()[p])
        xt = wl.x[t:t + 1]
        g = oracle.nvfp4_matmul(xt, wl.gate_codes[e], wl.gate_scales[e], float(wl.gate_global[e]), 0)[0]
        u = oracle.nvfp4_matmul(xt, wl.up_codes[e], wl.up_scales[e], float(wl.up_global[e]), 0)[0]
        bound = 2.0 ** -8 * (np.abs(ap[r]) + np.abs(an[r])) + 1e-30
        assert np.all(np.abs(ap[r] - an[r] - g * u) <= bound)


@pytest.mark.parametrize("shape", [(5, 64, 32, 4, 3, 51), (9, 128, 96, 6, 2, 52), ("tiny",)])
def test_gated_gather_equals_dense_masked(shape):
    """Per-pair gated oracle vs the independent dense-masked numpy form."""
    wl = W.generate("tiny", gated=True) if shape == ("tiny",) else W.small_custom(*shape[:5], seed=shape[5],
                                                                                    gated=True)
    res = oracle.moe_forward(wl, intermediates=True, out_f64=True)
    dense = numpy_ref.moe_dense_masked(wl)
    scale = np.abs(dense["out_f64"]).max()
    assert np.allclose(res.out_f64, dense["out_f64"], rtol=1e-12, atol=1e-12 * scale)
    assert np.count_nonzero(res.dst != dense["dst"]) == 0
    counts, offsets, perm, inv, _ = oracle.routing(wl.topk_ids, wl.E)
    for r, p in enumerate(perm):
        t, e = p // wl.k, int(wl.topk_ids.ravel()[p])
        assert np.array_equal(numpy_ref.bf16_bits_to_f64(res.a_rows[r]), dense["a"][e][t])


def test_gate_draws_leave_the_ungated_workload_unchanged():
    a = W.generate("tiny")
    b = W.generate("tiny", gated=True)
    for f in ("x", "topk_ids", "topk_weights", "up_codes", "up_scales", "down_codes", "down_scales", "dst"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    assert b.gate_codes.shape == b.up_codes.shape and b.gate_scales.shape == b.up_scales.shape
