"""Every layer kernel on weights drawn over the whole NVFP4 contract, against the oracle.

The configs' own recipe draws block scales that are powers of two in
[2^-4, 2^2] and one global 2^-4 for every expert and matrix.  The format the
layer takes is wider (gllm pull request #91, "What changes", bf16 NVFP4 GEMM:
a code times its e4m3 block scale, the per-tensor global as the GEMM's
alpha): any finite E4M3FN scale byte -- zero, subnormal, any mantissa, either
sign -- and a separate fp32 global per (expert, matrix).  Here every path
that runs the layer sees such weights:

  * the single-launch streaming kernel (routing, both projections and the
    combine in one launch; up to 8 tokens combine per column block, more
    after a second grid barrier);
  * the multi-kernel path: routing, gather, the streaming kernel in
    external-routing mode for experts at or below the threshold, the
    tcgen05 grouped GEMMs for the larger ones, WeightedRowSum;
  * the matrix-vector fallback (more pairs than one launch takes, threshold
    above every expert);
  * the shared expert (one expert, top-1, weight 1, written to dst);
  * the standalone NVFP4 matmul;

each for relu^2 and gated experts where the path has both, with scales over
all finite bytes ("full") and over the subnormal-heavy low range ("low",
where a flushed subnormal or a dropped mantissa bit moves the result by far
more than the tolerance), and distinct non-power-of-two globals throughout.

The bound is the layer's: |y_gpu - y_ref| <= 1e-2 * RMS(y_ref) + 1/2 ulp(y_gpu)
against the oracle's unrounded fp64 output, the same for the intermediates
(relu^2 or silu * up rows against their unrounded values), and
1e-2 * RMS for the fp32 down rows -- the down rows and the output plus the
intermediate's own rounding difference carried through |W_down| (see
``_check``).

The last tests show the bound has teeth on these inputs: mistakes a kernel
could plausibly make (up and down globals swapped, another expert's global,
the scale's mantissa or sign ignored, subnormal scales flushed) are planted
in copies of the ORACLE on the CPU, and the GPU's correct output must fail
against every one of them -- so the same mistake in a kernel would fail
against the real oracle."""
import os

import numpy as np
import pytest

import oracle
from nvfp4_quantized_moe_topk_gb300 import workload as W
from helpers import (bf16_from_dev, flip_allowance, fp_tolerance_check, layer_tolerance_check, make_layer,
                     run_forward, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    return torch.device("cuda:0")


def _intermediates(layer, wl, dev):
    import torch

    a = torch.empty((wl.R, wl.I), dtype=torch.int16, device=dev)
    y = torch.empty((wl.R, wl.H), dtype=torch.float32, device=dev)
    layer.debug_intermediates(a, y)
    torch.cuda.synchronize()
    return a.cpu().numpy().view(np.uint16), y.cpu().numpy()


def _check(wl, dev, *, intermediates=True, **layer_kw):
    """Layer output, intermediates and down rows against the oracle.  With
    scales over the whole e4m3 range one weight block can dominate a down
    row, so a one-step rounding difference of the bf16 intermediate (fp32 vs
    fp64 sums on either side of a boundary, itself within the intermediate's
    bound) moves that row by more than 1e-2 RMS: the down rows and the output
    are allowed that propagated difference on top (``flip_allowance``)."""
    layer = make_layer(wl, dev, **layer_kw)
    got = run_forward(layer, wl, dev)
    assert layer.device_error() == 0
    ref = oracle.moe_forward(wl, intermediates=intermediates, out_f64=True)
    extra_out = None
    if intermediates:
        a, y = _intermediates(layer, wl, dev)
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
    return got


SINGLE = [("decode-1", False, "full"), ("decode-1", True, "low"), ("decode-32", False, "low"),
          ("decode-32", True, "full")]


@pytest.mark.parametrize("name,gated,scales", SINGLE, ids=[f"{a}-{'gated' if b else 'relu2'}-{c}" for a, b, c in SINGLE])
def test_single_launch_full_contract(dev, name, gated, scales):
    wl = W.generate(name, gated=gated, scales=scales, globals_="distinct")
    _check(wl, dev)


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("scales", ["full", "low"])
@pytest.mark.parametrize("n,H,I,E,k,sigma,seed", [(120, 512, 384, 16, 2, 1.0, 60), (96, 2688, 1856, 6, 2, 1.0, 61)])
def test_multi_kernel_path_full_contract(dev, n, H, I, E, k, sigma, seed, scales, gated):
    """Grouped GEMMs for the experts above the threshold and the streaming
    kernel (external routing) for the rest, in the same forward."""
    wl = W.small_custom(n, H, I, E, k, seed, bias_sigma=sigma, gated=gated, scales=scales, globals_="distinct")
    counts = np.bincount(wl.topk_ids.ravel(), minlength=E)
    assert np.any(counts > 8) and np.any((counts > 0) & (counts <= 8)), "want both kinds of expert"
    _check(wl, dev, gemv_max_rows=8, single_max_tokens=-1)


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("scales", ["full", "low"])
def test_matvec_fallback_full_contract(dev, scales, gated):
    wl = W.small_custom(300, 256, 192, 5, 4, seed=62, gated=gated, scales=scales, globals_="distinct")
    assert wl.R > 1024
    _check(wl, dev, gemv_max_rows=1 << 30)


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("scales", ["full", "low"])
def test_shared_expert_full_contract(dev, scales, gated):
    import torch

    wl = W.small_custom(40, 512, 256, 1, 1, seed=63, gated=gated, scales=scales, globals_="distinct")
    wl.topk_ids[:] = 0
    wl.topk_weights[:] = 1.0
    wl.dst[:] = 0
    layer = make_layer(wl, dev)
    out = to_dev(np.full((wl.n, wl.H), 0x7FC0, np.uint16), dev)
    layer.shared_expert_forward(to_dev(wl.x, dev), out)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    layer.close()
    ok, err, rms = layer_tolerance_check(bf16_from_dev(out), oracle.moe_forward(wl, out_f64=True).out_f64)
    assert ok, (err, rms)


@pytest.mark.parametrize("scales", ["full", "low"])
@pytest.mark.parametrize("M,N,K,seed", [(300, 1856, 2688, 64), (77, 512, 1024, 65)])
def test_matmul_full_contract(dev, M, N, K, seed, scales):
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    rng = np.random.Generator(np.random.PCG64(seed))
    A = W.f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scales_b = W.draw_scales(rng, (N, K // 16), scales)
    g = float(W.draw_globals(rng, 1, W.global_base(scales))[0])
    for epi in (0, 1):
        ref = oracle.nvfp4_matmul(A, codes, scales_b, g, epi)
        out = torch.empty((M, N), dtype=torch.float32 if epi == 0 else torch.int16, device=dev)
        api.nvfp4_matmul(to_dev(A, dev), to_dev(codes, dev), to_dev(scales_b, dev), g, out, epilogue=epi)
        torch.cuda.synchronize()
        if epi == 0:
            ok, err, rms = fp_tolerance_check(out.cpu().numpy(), ref)
            assert ok, (err, rms)
        else:
            # relu^2 rows against the oracle's unrounded relu(h)^2
            h = oracle.nvfp4_matmul(A, codes, scales_b, g, 0)
            ok, err, rms = layer_tolerance_check(out.cpu().numpy().view(np.uint16), np.maximum(h, 0.0) ** 2)
            assert ok, (err, rms)


# ------------------------------------------------------- the bound has teeth
# (site in moe_oracle.c, replacement): each is a mistake a kernel could make
PLANTED = {
    "up_down_globals_swapped": [("      h *= (double)up_global[e];", "      h *= (double)dn_global[e];"),
                                ("y[q * H + c] = s * (double)dn_global[e];", "y[q * H + c] = s * (double)up_global[e];")],
    "global_of_next_expert": [("      h *= (double)up_global[e];", "      h *= (double)up_global[(e + 1) % E];")],
    "scale_mantissa_ignored": [("ldexp(1.0 + (double)m / 8.0, (int)e - 7)", "ldexp(1.0, (int)e - 7)")],
    "scale_sign_ignored": [("  *out = s ? -mag : mag;", "  *out = mag;")],
    "subnormal_scales_flushed": [("double mag = (e == 0) ? ldexp((double)m / 8.0, -6) :",
                                  "double mag = (e == 0) ? 0.0 :")],
    "gate_and_up_globals_swapped": [("      h *= (double)up_global[e];", "      h *= (double)gate_global[e];"),
                                    ("        gv *= (double)gate_global[e];", "        gv *= (double)up_global[e];")],
}


def _variant(name):
    src = oracle.source_text()
    for old, new in PLANTED[name]:
        assert src.count(old) == 1, f"planting site of {name} not found exactly once: {old!r}"
        src = src.replace(old, new)
    return oracle.build_variant(src, "contract_" + name)


SENSITIVITY = [
    # (workload, layer kwargs, mistakes its GPU output must fail against)
    ("decode-1-full", dict(), ["up_down_globals_swapped", "global_of_next_expert", "scale_mantissa_ignored",
                               "scale_sign_ignored"]),
    ("decode-1-low", dict(), ["subnormal_scales_flushed", "scale_mantissa_ignored"]),
    ("gemm-full", dict(gemv_max_rows=8, single_max_tokens=-1),
     ["up_down_globals_swapped", "global_of_next_expert", "scale_mantissa_ignored", "scale_sign_ignored"]),
    ("gemm-low", dict(gemv_max_rows=8, single_max_tokens=-1), ["subnormal_scales_flushed"]),
    ("gemm-gated-full", dict(gemv_max_rows=8, single_max_tokens=-1), ["gate_and_up_globals_swapped"]),
    ("decode-1-gated-full", dict(), ["gate_and_up_globals_swapped"]),
]


def _sens_workload(label):
    scales = "low" if label.endswith("low") else "full"
    gated = "gated" in label
    if label.startswith("decode-1"):
        wl = W.generate("decode-1", gated=gated, scales=scales, globals_="distinct")
    else:
        wl = W.small_custom(120, 512, 384, 16, 2, seed=66, bias_sigma=1.0, gated=gated, scales=scales,
                            globals_="distinct")
    if gated:
        # Where |g| >> 1 silu(g) is g or 0, so silu(g_gate G) g_up U and
        # silu(g_up G) g_gate U agree and a swap of the two globals is
        # invisible there; smaller gate globals put the gate pre-activations
        # at O(1), where the logistic bends.
        wl.gate_global = (wl.gate_global * np.float32(2.0 ** (-10 if scales == "full" else -5))).astype(np.float32)
    return wl


@pytest.mark.parametrize("label,kw,mistakes", SENSITIVITY, ids=[s[0] for s in SENSITIVITY])
def test_planted_oracle_mistakes_fail_the_bound(dev, label, kw, mistakes):
    wl = _sens_workload(label)
    layer = make_layer(wl, dev, **kw)
    got = run_forward(layer, wl, dev)
    a, _ = _intermediates(layer, wl, dev)
    layer.close()
    ok, err, rms = layer_tolerance_check(got, oracle.moe_forward(wl, out_f64=True).out_f64)
    assert ok, ("correct oracle", err, rms)
    for name in mistakes:
        path = _variant(name)
        try:
            with oracle.use_library(path):
                bad = oracle.moe_forward(wl, intermediates=True, out_f64=True)
        finally:
            os.remove(path)
        ok_out, err_out, rms_out = layer_tolerance_check(got, bad.out_f64)
        ok_a, _, _ = layer_tolerance_check(a, bad.a_f64)
        assert not (ok_out and ok_a), f"{label}: the GPU output also passes against an oracle with {name}"
