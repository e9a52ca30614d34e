"""Pins for the fp64 CPU oracle: each test ties it to something other than itself.

Sources of truth used here (none of them re-types the oracle's formulas):
  * the OCP MX e2m1 value table and torch's float8_e4m3fn decoder (formats);
  * exact rational arithmetic (``fractions.Fraction``) for bf16 rounding and
    for dyadic matmul cases, and torch's fp32->bf16 conversion;
  * numpy ``argsort(kind="stable")`` / ``bincount`` for the routing;
  * hand-worked fixtures under ``tests/golden/``;
  * an independent numpy restatement in the dense-masked form the pages
    replaced, and textbook numpy matvecs for the n = k = 1 special case;
  * closed forms (power-of-two globals) and degenerate cases.
"""
import json
import os
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import numpy_ref
from nvfp4_quantized_moe_topk_gb300 import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ formats
def test_e2m1_matches_ocp_table():
    table = numpy_ref.e2m1_table()
    for c in range(16):
        assert oracle.e2m1(c) == table[c], c
    # the -0 code is a zero
    assert oracle.e2m1(8) == 0.0


def test_e4m3_matches_torch_for_every_byte():
    ref = numpy_ref.e4m3_values(np.arange(256, dtype=np.uint8))
    for b in range(256):
        v = oracle.e4m3(b)
        if b in (0x7F, 0xFF):
            assert v is None and np.isnan(ref[b])
        else:
            assert v == ref[b], hex(b)


def _sig_bits(fr: Fraction) -> int:
    """Number of significant bits of a dyadic rational."""
    if fr == 0:
        return 0
    num, den = abs(fr.numerator), fr.denominator
    assert den & (den - 1) == 0, "not dyadic"
    while num % 2 == 0:
        num //= 2
    return num.bit_length()


def test_code_times_scale_is_exact_in_bf16():
    """Every e2m1 code times every finite e4m3 byte has <= 6 significant bits and
    survives a round trip through bf16 unchanged (pull request #91, "What
    changes", bf16 NVFP4 GEMM: the unpacked weight is exact in bf16)."""
    checked = 0
    for c in range(16):
        for b in range(256):
            if b in (0x7F, 0xFF):
                continue
            v = oracle.e2m1(c) * oracle.e4m3(b)
            assert _sig_bits(Fraction(v)) <= 6
            assert oracle.bf16_to_double(oracle.bf16_from_double(v)) == v
            checked += 1
    assert checked == 16 * 254


def _exact_bf16_round(v: float) -> float:
    """Round-to-nearest-even to bf16 in exact rational arithmetic (reference)."""
    fr = Fraction(v)
    if fr == 0:
        return 0.0
    s = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    q = Fraction(2) ** (e - 7)
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return float(s * fl * q)


def _rounding_samples(count=4000, seed=7):
    rng = random.Random(seed)
    out = []
    for _ in range(count):
        e = rng.randint(-140, 120)
        m = rng.random() + 1.0
        out.append(rng.choice([-1, 1]) * m * 2.0 ** e)
    # exact ties and near-ties around bf16 neighbours, incl. subnormal range
    for _ in range(2000):
        e = rng.randint(-133, 100)
        base = rng.randint(128, 255) * 2.0 ** (e - 7)
        half = 2.0 ** (e - 8)
        for d in (half, half * (1 + 2 ** -40), half * (1 - 2 ** -40)):
            out.append(base + d)
    return out


def test_bf16_rounding_matches_exact_rationals():
    for v in _rounding_samples():
        got = oracle.bf16_to_double(oracle.bf16_from_double(v))
        assert got == _exact_bf16_round(v), v


def test_bf16_rounding_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(3)
    a = (rng.standard_normal(20000) * np.exp2(rng.integers(-30, 30, 20000))).astype(np.float32)
    t = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    ours = np.array([oracle.bf16_from_double(float(v)) for v in a], dtype=np.uint16)
    assert np.array_equal(ours, t)


def test_numpy_ref_rounding_matches_exact_rationals():
    s = _rounding_samples(count=1000, seed=11)
    got = numpy_ref.bf16_round(np.array(s))
    exp = np.array([_exact_bf16_round(v) for v in s])
    assert np.array_equal(got, exp)


# ------------------------------------------------------------------ routing
def test_routing_hand_fixtures():
    for case in _load("routing_hand.json")["cases"]:
        counts, offsets, perm, inv, dropped = oracle.routing(np.array(case["ids"], np.int32), case["E"])
        assert counts.tolist() == case["counts"], case["name"]
        assert offsets.tolist() == case["offsets"], case["name"]
        assert perm.tolist() == case["perm_pair"], case["name"]
        assert inv.tolist() == case["inv"], case["name"]
        assert dropped == sum(1 for r in case["inv"] if r < 0)


@pytest.mark.parametrize("n,k,E,seed", [(1, 6, 128, 0), (32, 6, 128, 1), (200, 8, 16, 2), (1000, 3, 5, 3)])
def test_routing_matches_numpy_stable_argsort(n, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(n, k)).astype(np.int32)  # duplicates allowed
    counts, offsets, perm, inv, dropped = oracle.routing(ids, E)
    flat = ids.ravel()
    assert dropped == 0
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    assert np.array_equal(inv[perm], np.arange(n * k))


@pytest.mark.parametrize("name", ["tiny", "decode-1", "decode-32", "prefill-4314", "prefill-16384"])
def test_row_counts_sum_to_n_times_topk(name):
    wl = W.generate(name, weights=False)
    counts, offsets, perm, inv, dropped = oracle.routing(wl.topk_ids, wl.E)
    assert dropped == 0
    assert int(counts.sum()) == wl.n * wl.k == offsets[-1]
    if name == "prefill-4314":
        # pull request #91, "What the profile showed", item 1: ~26k routed rows
        # at topK 6 against ~552k dense-masked rows over 128 experts
        assert wl.n * wl.k == 25884 and wl.n * wl.E == 552192
    if name == "prefill-16384":
        assert wl.n * wl.k == 131072


# ------------------------------------------------------- WeightedRowSum
def test_weighted_row_sum_hand_fixtures():
    for case in _load("weighted_row_sum_hand.json")["cases"]:
        dst = W.f32_to_bf16_bits(np.array(case["dst"], np.float32))
        out, skipped = oracle.weighted_row_sum(dst, np.array(case["src"], np.float64),
                                               np.array(case["rows"], np.int32), np.array(case["w"], np.float32))
        got = W.bf16_bits_to_f32(out).astype(np.float64)
        assert np.array_equal(got, np.array(case["expected"])), case["name"]
        assert skipped == 0


def test_weighted_row_sum_skips_out_of_range_rows():
    dst = W.f32_to_bf16_bits(np.array([[1.0, 2.0]], np.float32))
    out, skipped = oracle.weighted_row_sum(dst, np.array([[4.0, 8.0]]), np.array([[0, 5, -1]], np.int32),
                                           np.array([[0.5, 1.0, 1.0]], np.float32))
    assert skipped == 2
    assert W.bf16_bits_to_f32(out).tolist() == [[3.0, 6.0]]


# ------------------------------------------------------------------ matmul
def _hand_matmul_case():
    g = _load("nvfp4_matmul_hand.json")
    K = g["K"]
    codes = np.zeros((2, K // 2), np.uint8)
    scales = np.zeros((2, K // 16), np.uint8)
    codes[0] = np.frombuffer(bytes.fromhex(g["codes_row0_hex"]), np.uint8)
    scales[0] = np.frombuffer(bytes.fromhex(g["scales_row0_hex"]), np.uint8)
    # row 1: the mirror image (nibbles swapped, blocks swapped) must give a different value
    codes[1] = ((codes[0] & 0x0F) << 4) | (codes[0] >> 4)
    scales[1] = scales[0][::-1]
    x = np.zeros((1, K), np.float32)
    for i, v in g["x"].items():
        x[0, int(i)] = v
    return g, W.f32_to_bf16_bits(x), codes, scales


def test_nvfp4_matmul_hand_fixture():
    g, xb, codes, scales = _hand_matmul_case()
    out = oracle.nvfp4_matmul(xb, codes, scales, g["global"], 0)
    assert out[0, 0] == g["expected_fp32"]
    assert out[0, 1] != g["expected_fp32"]  # nibble order and block index matter
    o1 = oracle.nvfp4_matmul(xb, codes, scales, g["global"], 1)
    assert int(o1[0, 0]) == int(g["expected_relu2_bf16_bits"], 16)


def test_nvfp4_matmul_matches_numpy_dequant():
    rng = np.random.default_rng(5)
    M, N, K = 7, 48, 96
    A = W.f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, (N, K // 16)).astype(np.uint8)  # any finite positive e4m3
    g = 0.37
    ref = (numpy_ref.bf16_bits_to_f64(A) @ numpy_ref.dequant(codes, scales).T) * g
    out = oracle.nvfp4_matmul(A, codes, scales, g, 0)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.array_equal(oracle.dequant(codes, scales, N, K), numpy_ref.dequant(codes, scales))


def test_nvfp4_matmul_dyadic_is_exact():
    """x in {0, +-1, +-2}/4, scales in {1/2, 1, 2}, global 2^-4: every partial sum
    is dyadic and exact, so the fp64 result equals exact rational arithmetic."""
    rng = np.random.default_rng(9)
    M, N, K = 5, 16, 64
    xv = rng.choice(np.array([0, 1, -1, 2, -2], np.float32) / 4, size=(M, K))
    A = W.f32_to_bf16_bits(xv)
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scales = W.e4m3_byte_of_pow2(rng.integers(-1, 2, (N, K // 16)))
    Wd = numpy_ref.dequant(codes, scales)
    out = oracle.nvfp4_matmul(A, codes, scales, 2.0 ** -4, 0)
    for m in range(M):
        for j in range(N):
            exact = sum(Fraction(float(xv[m, c])) * Fraction(float(Wd[j, c])) for c in range(K)) * Fraction(1, 16)
            assert Fraction(out[m, j]) == exact


def test_global_scaling_closed_form():
    """Doubling the up global multiplies relu^2's input square by 4; doubling the
    down global doubles the down output (exact for power-of-two globals)."""
    wl = W.small_custom(4, 64, 32, 3, 2, seed=21)
    wl.dst[:] = 0
    base = oracle.moe_forward(wl, intermediates=True)
    wl2 = W.small_custom(4, 64, 32, 3, 2, seed=21)
    wl2.dst[:] = 0
    wl2.down_global *= 2
    dbl = oracle.moe_forward(wl2, intermediates=True)
    assert np.array_equal(dbl.y_rows, 2 * base.y_rows)
    assert np.array_equal(dbl.a_rows, base.a_rows)
    wl3 = W.small_custom(4, 64, 32, 3, 2, seed=21)
    wl3.dst[:] = 0
    wl3.up_global *= 2
    up2 = oracle.moe_forward(wl3, intermediates=True)
    a0 = numpy_ref.bf16_bits_to_f64(base.a_rows)
    a1 = numpy_ref.bf16_bits_to_f64(up2.a_rows)
    assert np.array_equal(a1, 4 * a0)  # x4 is a power of two: rounding commutes


# ------------------------------------------------------------ whole layer
def test_zero_weights_leave_dst_unchanged():
    wl = W.small_custom(6, 64, 32, 4, 2, seed=1)
    wl.topk_weights[:] = 0
    assert np.array_equal(oracle.moe_forward(wl).dst, wl.dst)


def test_zero_codes_leave_dst_unchanged():
    wl = W.small_custom(6, 64, 32, 4, 2, seed=2)
    wl.up_codes[:] = 0
    assert np.array_equal(oracle.moe_forward(wl).dst, wl.dst)
    wl = W.small_custom(6, 64, 32, 4, 2, seed=2)
    wl.down_codes[:] = 0x88  # -0 in both nibbles
    assert np.array_equal(oracle.moe_forward(wl).dst, wl.dst)


def test_all_negative_preactivations_leave_dst_unchanged():
    wl = W.small_custom(3, 64, 32, 2, 1, seed=3)
    wl.x[:] = W.f32_to_bf16_bits(np.ones((3, 64), np.float32))
    wl.up_codes[:] = 0xAA  # every code 0xA = -1.0: h < 0 everywhere
    assert np.array_equal(oracle.moe_forward(wl).dst, wl.dst)


def test_single_pair_reduces_to_two_matvecs():
    """n = 1, k = 1, w = 1: the layer is two textbook matvecs around relu^2."""
    wl = W.small_custom(1, 96, 64, 3, 1, seed=4)
    wl.topk_weights[:] = 1.0
    e = int(wl.topk_ids[0, 0])
    res = oracle.moe_forward(wl, intermediates=True, out_f64=True)
    y, a = numpy_ref.matvec_chain(wl.x[0], wl.up_codes[e], wl.up_scales[e], wl.down_codes[e], wl.down_scales[e],
                                  float(wl.up_global[e]), float(wl.down_global[e]))
    assert np.array_equal(numpy_ref.bf16_bits_to_f64(res.a_rows[0]), a)
    assert np.allclose(res.y_rows[0], y, rtol=1e-12, atol=1e-12 * np.abs(y).max())
    dst0 = numpy_ref.bf16_bits_to_f64(wl.dst[0])
    assert np.allclose(res.out_f64[0], dst0 + y, rtol=1e-12, atol=1e-12 * np.abs(y).max())


@pytest.mark.parametrize("shape", [("tiny",), (5, 64, 32, 4, 3, 31), (9, 128, 96, 6, 2, 32), (3, 32, 64, 2, 2, 33)])
def test_gather_equals_dense_masked(shape):
    """The per-pair (gathered) oracle agrees with the independent dense-masked
    restatement (pull request #91, "What the profile showed", item 1)."""
    wl = W.generate("tiny") if shape == ("tiny",) else W.small_custom(*shape[:5], seed=shape[5])
    res = oracle.moe_forward(wl, intermediates=True, out_f64=True)
    dense = numpy_ref.moe_dense_masked(wl)
    scale = np.abs(dense["out_f64"]).max()
    assert np.allclose(res.out_f64, dense["out_f64"], rtol=1e-12, atol=1e-12 * scale)
    mismatch = np.count_nonzero(res.dst != dense["dst"])
    assert mismatch == 0
    counts, offsets, perm, inv, _ = oracle.routing(wl.topk_ids, wl.E)
    for r, p in enumerate(perm):
        t, e = p // wl.k, int(wl.topk_ids.ravel()[p])
        assert np.array_equal(numpy_ref.bf16_bits_to_f64(res.a_rows[r]), dense["a"][e][t])
        # the unrounded intermediate: the restatement's value up to fp64 summation order,
        # and the bf16 row is its one rounding
        raw = dense["a_f64"][e][t]
        assert np.allclose(res.a_f64[r], raw, rtol=1e-12, atol=1e-12 * max(np.abs(raw).max(), 1e-300))
        assert np.array_equal(numpy_ref.bf16_round(res.a_f64[r]), numpy_ref.bf16_bits_to_f64(res.a_rows[r]))


def test_duplicate_expert_in_one_token():
    """A token may pick the same expert twice; each pair is its own row."""
    wl = W.small_custom(2, 64, 32, 3, 2, seed=5)
    wl.topk_ids[0] = [1, 1]
    res = oracle.moe_forward(wl, intermediates=True, out_f64=True)
    dense = numpy_ref.moe_dense_masked(wl)
    assert np.allclose(res.out_f64, dense["out_f64"], rtol=1e-12)
    counts, *_ = oracle.routing(wl.topk_ids, wl.E)
    assert counts[1] >= 2


def test_out_of_range_id_drops_the_pair():
    wl = W.small_custom(2, 64, 32, 3, 2, seed=6)
    keep = oracle.moe_forward(wl, out_f64=True)
    wl.topk_ids[1, 1] = 99
    wl.topk_weights[1, 1] = 0.0  # weight-0 pair == dropped pair
    ref = oracle.moe_forward(wl, out_f64=True)
    wl.topk_weights[1, 1] = 0.7
    dropped = oracle.moe_forward(wl, out_f64=True)
    assert np.array_equal(dropped.out_f64, ref.out_f64)
    assert np.array_equal(dropped.out_f64[0], keep.out_f64[0])


def test_token_range_sample_matches_full_run():
    wl = W.small_custom(8, 64, 32, 4, 2, seed=8)
    full = oracle.moe_forward(wl)
    part = oracle.moe_forward(wl, tok_range=(3, 6))
    assert np.array_equal(part.dst[3:6], full.dst[3:6])
    assert np.array_equal(part.dst[:3], wl.dst[:3])


# ----------------------------------------------------------------- router
def _biased(logits, bias):
    return logits if bias is None else (logits + bias[None, :]).astype(np.float32)


@pytest.mark.parametrize("n,E,k,sigma,seed", [(200, 128, 8, 0.0, 1), (300, 128, 6, 1.5, 2), (64, 1024, 32, 2.0, 3),
                                              (17, 8, 8, 0.0, 4), (5, 3, 1, 1.0, 5)])
def test_router_matches_argsort_and_softmax(n, E, k, sigma, seed):
    """Top-k equals numpy's stable argsort of the fp32 biased logits (descending,
    ties to the lower index); weights equal scipy's softmax of the picked ones;
    counts equal bincount."""
    from scipy.special import softmax

    rng = np.random.Generator(np.random.PCG64(seed))
    logits = rng.standard_normal((n, E), dtype=np.float32)
    bias = (rng.standard_normal(E, dtype=np.float32) * np.float32(sigma)) if sigma > 0 else None
    ids, w, counts = oracle.router_topk(logits, bias, k)
    z = _biased(logits, bias)
    ref_ids = np.argsort(-z.astype(np.float64), axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, ref_ids)
    picked = np.take_along_axis(z.astype(np.float64), ref_ids, axis=1)
    assert np.allclose(w, softmax(picked, axis=1), rtol=1e-6, atol=0)
    assert np.array_equal(counts, np.bincount(ref_ids.ravel(), minlength=E))


def test_router_hand_fixture_with_ties_and_bias():
    g = json.load(open(os.path.join(GOLDEN, "router_hand.json")))
    ids, w, counts = oracle.router_topk(np.array(g["logits"], np.float32), np.array(g["bias"], np.float32), g["k"])
    assert ids.tolist() == g["ids"]
    assert np.allclose(w, np.array(g["weights"]), rtol=1e-6, atol=0)
    assert counts.tolist() == g["counts"]


def test_router_closed_forms():
    rng = np.random.Generator(np.random.PCG64(9))
    logits = rng.standard_normal((50, 16), dtype=np.float32)
    _, w1, _ = oracle.router_topk(logits, None, 1)
    assert np.all(w1 == 1.0)  # a single pick gets the whole weight
    _, w, _ = oracle.router_topk(logits, None, 5)
    assert np.allclose(w.astype(np.float64).sum(axis=1), 1.0, atol=1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)  # descending logits give descending weights
    with pytest.raises(ValueError):
        oracle.router_topk(logits, None, 17)
