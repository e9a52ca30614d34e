"""The seeded input recipe that both the oracle and the GPU path consume (CPU).

The generator holds none of the layer's arithmetic; these tests check that it
draws what the input recipe states: reproducible from the seed, uniform code
bytes, block scales 2^u with u uniform in {-4, ..., 2}, a routing that is the
top-k of the (biased) logits with softmax weights over the k picks, and gate
draws appended after the ungated draws."""
import numpy as np
import pytest

from nvfp4_quantized_moe_topk_gb300 import workload as W


def test_same_seed_same_arrays():
    a, b = W.generate("tiny"), W.generate("tiny")
    for f in ("x", "topk_ids", "topk_weights", "up_codes", "up_scales", "down_codes", "down_scales", "dst"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    c = W.generate("tiny", seed=7)
    assert not np.array_equal(a.up_codes, c.up_codes)


def test_scale_bytes_are_powers_of_two_in_range():
    wl = W.generate("tiny")
    allowed = {((u + 7) << 3) for u in range(-4, 3)}  # e4m3 of 2^u: exponent field u + 7, mantissa 0
    for s in (wl.up_scales, wl.down_scales):
        vals, counts = np.unique(s, return_counts=True)
        assert set(vals.tolist()) == allowed  # all seven exponents drawn, nothing else
        assert counts.min() > 0.8 * s.size / 7 and counts.max() < 1.2 * s.size / 7


def test_code_nibbles_are_uniform():
    wl = W.generate("tiny")
    nib = np.concatenate([(wl.up_codes & 15).ravel(), (wl.up_codes >> 4).ravel()])
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * nib.size / 16 and counts.max() < 1.1 * nib.size / 16


@pytest.mark.parametrize("name", ["tiny", "decode-32"])
def test_routing_is_topk_of_logits_with_softmax_weights(name):
    wl = W.generate(name, weights=False)
    ids, w = wl.topk_ids, wl.topk_weights.astype(np.float64)
    assert ids.shape == (wl.n, wl.k) and ids.min() >= 0 and ids.max() < wl.E
    assert all(len(set(r.tolist())) == wl.k for r in ids)  # k distinct experts per token
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6)
    assert np.all(np.diff(w, axis=1) <= 0) and np.all(w > 0)


def test_activations_and_dst_are_finite_bf16():
    wl = W.generate("tiny")
    for a in (wl.x, wl.dst):
        v = W.bf16_bits_to_f32(a)
        assert np.all(np.isfinite(v))
        assert abs(float(v.mean())) < 0.1 and 0.9 < float(v.std()) < 1.1  # standard normal draws


def test_gate_draws_come_after_the_shared_ones():
    plain, gated = W.generate("tiny"), W.generate("tiny", gated=True)
    for f in ("x", "topk_ids", "topk_weights", "up_codes", "up_scales", "down_codes", "down_scales", "dst"):
        assert np.array_equal(getattr(plain, f), getattr(gated, f)), f
    assert gated.gate_codes.shape == plain.up_codes.shape
    assert gated.gate_scales.shape == plain.up_scales.shape
    assert not np.array_equal(gated.gate_codes, gated.up_codes)


def test_bias_skews_expert_counts():
    # the prefill recipe adds a per-expert bias (sigma 1.5) to the logits: the row counts then spread far
    # wider than the unbiased multinomial's
    skewed = np.bincount(W.generate("prefill-4314", weights=False).topk_ids.ravel(), minlength=128)
    unbiased = np.bincount(W.make_routing(4314, 128, 6, 0.0, seed=5)[0].ravel(), minlength=128)
    assert skewed.sum() == unbiased.sum() == 4314 * 6
    assert skewed.std() > 3 * unbiased.std()


def test_full_contract_scale_draws():
    """'full' draws every finite E4M3FN byte (both signs, zero, subnormals) and
    never a NaN byte; 'low' draws exactly the bytes with exponent field 0..3."""
    rng = np.random.Generator(np.random.PCG64(3))
    full = W.draw_scales(rng, (200000,), "full")
    seen = set(np.unique(full).tolist())
    assert seen == set(range(256)) - {0x7F, 0xFF}
    low = W.draw_scales(rng, (50000,), "low")
    want = {(s << 7) | (e << 3) | m for s in (0, 1) for e in range(4) for m in range(8)}
    assert set(np.unique(low).tolist()) == want
    assert np.any(low & 0x80) and np.any((low & 0x78) == 0)  # negative and subnormal scales occur


def test_distinct_globals_and_unchanged_shared_draws():
    base = W.small_custom(6, 64, 32, 5, 2, seed=9)
    wide = W.small_custom(6, 64, 32, 5, 2, seed=9, globals_="distinct", gated=True)
    for g in (wide.up_global, wide.down_global, wide.gate_global):
        m, _ = np.frexp(g.astype(np.float64))
        assert not np.any(m == 0.5), "a global is a power of two"
    allg = np.concatenate([wide.up_global, wide.down_global, wide.gate_global])
    assert len(np.unique(allg)) == allg.size
    # the globals are drawn last: codes, scales, routing and activations are the recipe's
    for name in ("x", "topk_ids", "topk_weights", "up_codes", "up_scales", "down_codes", "down_scales", "dst"):
        assert np.array_equal(getattr(base, name), getattr(wide, name)), name
