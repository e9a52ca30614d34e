"""The streaming kernel's two sources of activation rows, in one launch.

When every expert holds at most 8 tokens, a CTA copies the activation rows of
the experts its work items belong to once per phase into a shared stage (the x
rows of their tokens for the up projection, their packed relu^2 / silu * up
rows for the down projection); otherwise, or when those rows would not fit,
each weight chunk brings its own activation row segments.  The choice is made
per CTA after the in-kernel routing.

Here all 8 tokens pick all 7 experts (k = E) at H = 4096: a CTA whose items lie
in one expert stages 8 rows of 8 KB, one whose items straddle two experts would
need 16 rows (128 KB) and takes the per-chunk copies instead, so both kinds run
side by side in every launch, for relu^2 and gated experts.  The bound is the
layer's (output and intermediates against the oracle's unrounded fp64 values,
down rows with the propagated intermediate rounding difference), and a second
forward must give the same bits."""
import numpy as np
import pytest

import oracle
from nvfp4_quantized_moe_topk_gb300 import workload as W
from helpers import flip_allowance, fp_tolerance_check, layer_tolerance_check, make_layer, run_forward

pytestmark = pytest.mark.gpu

STAGE_MAX = 96 * 1024  # bytes of staged rows a CTA may hold


@pytest.fixture(scope="module")
def dev():
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    return torch.device("cuda:0")


def _cta_stage_bytes(wl, num_sms):
    """Per CTA, the staged bytes of the larger phase (items cut evenly over
    the grid, two 16-row tiles per item since experts hold several tokens)."""
    counts = np.bincount(wl.topk_ids.ravel(), minlength=wl.E)
    act = [e for e in range(wl.E) if counts[e] > 0]
    n_act = len(act)
    out = []
    for b in range(num_sms):
        need = 0
        for NP, K in (((2 * wl.I if wl.gated else wl.I) // 32, wl.H), (wl.H // 32, wl.I)):
            U = n_act * NP
            lo, hi = U * b // num_sms, U * (b + 1) // num_sms
            if hi > lo:
                rows = sum(int(counts[act[j]]) for j in range(lo // NP, (hi - 1) // NP + 1))
                need = max(need, rows * (2 * K + 16))
        out.append(need)
    return out


@pytest.mark.parametrize("gated", [False, True])
def test_staged_and_per_chunk_ctas_in_one_launch(dev, gated):
    import torch

    wl = W.small_custom(8, 4096, 1920, 7, 7, seed=71, gated=gated, scales="full", globals_="distinct")
    need = _cta_stage_bytes(wl, torch.cuda.get_device_properties(dev).multi_processor_count)
    assert min(need) <= STAGE_MAX < max(need), "want CTAs on both sides of the stage limit"
    layer = make_layer(wl, dev)
    got = run_forward(layer, wl, dev)
    assert layer.device_error() == 0
    ref = oracle.moe_forward(wl, intermediates=True, out_f64=True)
    a = torch.empty((wl.R, wl.I), dtype=torch.int16, device=dev)
    y = torch.empty((wl.R, wl.H), dtype=torch.float32, device=dev)
    layer.debug_intermediates(a, y)
    torch.cuda.synchronize()
    a = a.cpu().numpy().view(np.uint16)
    y = y.cpu().numpy()
    ok_a, ea, ra = layer_tolerance_check(a, ref.a_f64)
    assert ok_a, f"intermediate rows: max|err| {ea:.4g} vs rms {ra:.4g}"
    e_rows, extra_out = flip_allowance(wl, a, ref.a_rows)
    ok_y, ey, ry = fp_tolerance_check(y, ref.y_rows, extra=e_rows)
    assert ok_y, f"down rows: max|err| {ey:.4g} vs rms {ry:.4g}"
    ok, err, rms = layer_tolerance_check(got, ref.out_f64, extra=extra_out)
    assert ok, f"layer output: max|err| {err:.4g} vs rms {rms:.4g}"
    again = run_forward(layer, wl, dev)
    assert np.array_equal(got, again), "repeated forward changed bits"
    layer.close()


def _scale_rows_pow2(bits, exps):
    """bf16 rows times 2^exps[row], exactly (the values stay normal bf16)."""
    v = W.bf16_bits_to_f32(bits).astype(np.float64) * np.ldexp(1.0, np.asarray(exps))[:, None]
    out = W.f32_to_bf16_bits(v.astype(np.float32))
    assert np.array_equal(W.bf16_bits_to_f32(out).astype(np.float64), v), "scaling must be exact"
    return out


@pytest.mark.parametrize("gated", [False, True])
def test_staged_f16_rows_across_the_bf16_range(dev, gated):
    """The staged path computes in f16 after scaling each activation row by a
    power of two; rows 2^-40 .. 2^50 (their relu^2 / silu * up rows spanning
    roughly 2^-75 .. 2^105) would leave f16's range without that scaling.
    One row also holds values 2^-36 below the rest, which land among f16's
    subnormals.  Each token's output, and each packed row's intermediate and
    down row, is held to the layer bound against its own RMS."""
    import torch

    wl = W.small_custom(8, 512, 256, 4, 2, seed=72, gated=gated, scales="full", globals_="distinct")
    exps = np.array([-40, -24, -8, 0, 8, 16, 24, 36])
    wl.x = _scale_rows_pow2(wl.x, exps)
    x0 = W.bf16_bits_to_f32(wl.x).astype(np.float64)
    x0[0, ::7] *= 2.0 ** -36
    wl.x = W.f32_to_bf16_bits(x0.astype(np.float32))
    wl.dst = _scale_rows_pow2(wl.dst, exps)
    counts = np.bincount(wl.topk_ids.ravel(), minlength=wl.E)
    assert counts.max() <= 8
    layer = make_layer(wl, dev)
    got = run_forward(layer, wl, dev)
    assert layer.device_error() == 0
    ref = oracle.moe_forward(wl, intermediates=True, out_f64=True)
    a = torch.empty((wl.R, wl.I), dtype=torch.int16, device=dev)
    y = torch.empty((wl.R, wl.H), dtype=torch.float32, device=dev)
    layer.debug_intermediates(a, y)
    torch.cuda.synchronize()
    a = a.cpu().numpy().view(np.uint16)
    y = y.cpu().numpy()
    layer.close()
    assert np.all(np.isfinite(W.bf16_bits_to_f32(got)))
    e_rows, extra_out = flip_allowance(wl, a, ref.a_rows)
    for r in range(wl.R):
        ok_a, ea, ra = layer_tolerance_check(a, ref.a_f64, rows=[r])
        assert ok_a, f"packed row {r}: intermediate max|err| {ea:.4g} vs rms {ra:.4g}"
        ok_y, ey, ry = fp_tolerance_check(y[r:r + 1], ref.y_rows[r:r + 1], extra=e_rows[r:r + 1])
        assert ok_y, f"packed row {r}: down row max|err| {ey:.4g} vs rms {ry:.4g}"
    for t in range(wl.n):
        ok, err, rms = layer_tolerance_check(got, ref.out_f64, rows=[t], extra=extra_out)
        assert ok, f"token {t} (x 2^{exps[t]}): output max|err| {err:.4g} vs rms {rms:.4g}"


@pytest.mark.parametrize("gated", [False, True])
def test_staged_path_with_many_experts_per_cta(dev, gated):
    """The single launch at its pair bound (64 tokens x top-16 = 1024 pairs)
    over 1024 experts: every expert holds at most a few tokens, so CTAs stage,
    each for five or six experts (small H and I: six or eight items per
    expert).  Layer output and intermediates against the oracle."""
    import torch

    wl = W.small_custom(64, 256, 192, 1024, 16, seed=73, gated=gated, scales="full", globals_="distinct")
    counts = np.bincount(wl.topk_ids.ravel(), minlength=wl.E)
    assert wl.R == 1024 and 2 <= counts.max() <= 8
    layer = make_layer(wl, dev)
    got = run_forward(layer, wl, dev)
    assert layer.device_error() == 0
    ref = oracle.moe_forward(wl, intermediates=True, out_f64=True)
    a = torch.empty((wl.R, wl.I), dtype=torch.int16, device=dev)
    y = torch.empty((wl.R, wl.H), dtype=torch.float32, device=dev)
    layer.debug_intermediates(a, y)
    torch.cuda.synchronize()
    a = a.cpu().numpy().view(np.uint16)
    y = y.cpu().numpy()
    layer.close()
    ok_a, ea, ra = layer_tolerance_check(a, ref.a_f64)
    assert ok_a, f"intermediate rows: max|err| {ea:.4g} vs rms {ra:.4g}"
    e_rows, extra_out = flip_allowance(wl, a, ref.a_rows)
    ok_y, ey, ry = fp_tolerance_check(y, ref.y_rows, extra=e_rows)
    assert ok_y, f"down rows: max|err| {ey:.4g} vs rms {ry:.4g}"
    ok, err, rms = layer_tolerance_check(got, ref.out_f64, extra=extra_out)
    assert ok, f"layer output: max|err| {err:.4g} vs rms {rms:.4g}"
