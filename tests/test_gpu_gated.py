"""GPU parity of the gated expert layer (a = bf16(silu(gate) * up)) against the oracle.

Every path a gated layer can take is covered: the single-launch streaming
kernel (whose up items are (gate tile, up tile) pairs), the multi-kernel path
with the grouped tensor-core GEMM (weight blocks of 16 gate rows then the 16
up rows of the same features, met by a lane shuffle in the epilogue) and the
streaming kernel in external-routing mode for the small experts, and the
allocation-free entry point (the GEMV kernel streaming both rows).  The layer
output must meet max|y - y_ref| <= 1e-2 RMS(y_ref); the intermediate rows are
compared too."""
import numpy as np
import pytest

import oracle
from nvfp4_quantized_moe_topk_gb300 import workload as W
from helpers import bf16_from_dev, fp_tolerance_check, layer_tolerance_check, make_layer, run_forward, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    return torch.device("cuda:0")


def _check(wl, dev, single_max_tokens=0, gemv_max_rows=0, sample=None, intermediates=True):
    import torch

    layer = make_layer(wl, dev, single_max_tokens=single_max_tokens, gemv_max_rows=gemv_max_rows)
    got = run_forward(layer, wl, dev)
    assert layer.device_error() == 0
    if sample is not None:
        for t0, t1 in sample:
            part = oracle.moe_forward(wl, tok_range=(t0, t1), out_f64=True)
            ok, err, rms = layer_tolerance_check(got[t0:t1], part.out_f64[t0:t1])
            assert ok, f"tokens {t0}:{t1}: max|err| {err} vs rms {rms}"
        layer.close()
        return got
    ref = oracle.moe_forward(wl, intermediates=intermediates, out_f64=True)
    ok, err, rms = layer_tolerance_check(got, ref.out_f64)
    assert ok, f"layer output: max|err| {err} vs rms {rms}"
    if intermediates:
        a = torch.empty((wl.R, wl.I), dtype=torch.int16, device=dev)
        y = torch.empty((wl.R, wl.H), dtype=torch.float32, device=dev)
        layer.debug_intermediates(a, y)
        torch.cuda.synchronize()
        a = a.cpu().numpy().view(np.uint16)
        oka, ea, ra_ = layer_tolerance_check(a, ref.a_f64)
        assert oka, f"silu*up rows: {ea} vs rms {ra_}"
        oky, ey, ry = fp_tolerance_check(y.cpu().numpy(), ref.y_rows)
        assert oky, f"down rows: {ey} vs rms {ry}"
    layer.close()
    return got


def test_gated_tiny(dev):
    _check(W.generate("tiny", gated=True), dev)


def test_gated_decode_1(dev):
    _check(W.generate("decode-1", gated=True), dev)


def test_gated_decode_32(dev):
    _check(W.generate("decode-32", gated=True), dev)


@pytest.mark.parametrize("n,H,I,E,k,seed", [(1, 64, 64, 1, 1, 60), (7, 128, 192, 5, 3, 61), (13, 320, 256, 9, 4, 62),
                                             (20, 128, 128, 3, 2, 63)])
def test_gated_small_shapes_single_launch(dev, n, H, I, E, k, seed):
    _check(W.small_custom(n, H, I, E, k, seed, gated=True), dev, gemv_max_rows=1 << 30)


def test_gated_one_expert_many_tokens(dev):
    # every pair on one expert: 40 rows, five 8-token passes per item
    wl = W.small_custom(20, 128, 128, 3, 2, seed=64, gated=True)
    wl.topk_ids[:] = 1
    _check(wl, dev, gemv_max_rows=1 << 30)


@pytest.mark.parametrize("n,H,I,E,k,T,seed", [(300, 256, 192, 8, 4, 8, 65), (129, 1024, 512, 16, 8, 8, 66),
                                               (600, 128, 64, 4, 2, 0, 67), (449, 128, 128, 1, 1, 1, 68)])
def test_gated_grouped_gemm_path(dev, n, H, I, E, k, T, seed):
    """Multi-kernel path: experts above T rows on the grouped GEMM (gated
    epilogue), the others on the streaming kernel in external-routing mode.
    449 rows on one expert: two full 224-row token tiles and a one-row tile."""
    wl = W.small_custom(n, H, I, E, k, seed, bias_sigma=1.0, gated=True)
    _check(wl, dev, single_max_tokens=-1, gemv_max_rows=T)


def test_gated_prefill_4314_sampled(dev):
    wl = W.generate("prefill-4314", gated=True)
    _check(wl, dev, sample=[(0, 24), (2150, 2166), (4300, 4314)])


def test_gated_deterministic(dev):
    wl = W.generate("decode-32", gated=True)
    layer = make_layer(wl, dev)
    a = run_forward(layer, wl, dev)
    b = run_forward(layer, wl, dev)
    assert np.array_equal(a, b)
    layer.close()


def test_gated_noalloc_matches_forward(dev):
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    wl = W.generate("decode-32", gated=True)
    layer = make_layer(wl, dev)
    weights = [to_dev(a, dev) for a in (wl.up_codes, wl.up_scales, wl.down_codes, wl.down_scales,
                                         wl.up_global, wl.down_global)]
    gate = [to_dev(a, dev) for a in (wl.gate_codes, wl.gate_scales, wl.gate_global)]
    x, ids, tw = to_dev(wl.x, dev), to_dev(wl.topk_ids, dev), to_dev(wl.topk_weights, dev)
    ref = to_dev(wl.dst, dev)
    layer.forward(x, ids, tw, ref)
    got = to_dev(wl.dst, dev)
    api.forward_noalloc(wl.H, wl.I, wl.E, wl.k, *weights, x, ids, tw, got, gate_codes=gate[0],
                        gate_scales=gate[1], gate_global=gate[2])
    torch.cuda.synchronize()
    res = oracle.moe_forward(wl, out_f64=True)
    for label, out in (("no-alloc", got), ("forward", ref)):
        ok, err, rms = layer_tolerance_check(bf16_from_dev(out), res.out_f64)
        assert ok, (label, err, rms)
    layer.close()
