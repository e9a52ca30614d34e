"""The allocation-free entry point against the handle-based forward.

Callers that cannot call cudaMalloc (a plugin whose host owns all device
memory, a fixed memory budget) use moe_nvfp4_forward_noalloc, which keeps its
intermediates in the library's fixed device array.  Its output must match the
existing forward's within the layer tolerance, on two calls in a row (the
array keeps the previous call's contents, so the second call checks that
nothing stale leaks through).  Collected last on purpose."""
import numpy as np
import pytest

import oracle
from nvfp4_quantized_moe_topk_gb300 import workload as W
from helpers import bf16_from_dev, layer_tolerance_check, make_layer, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,seeds", [("decode-32", (1002, 77)), ("decode-1", (1001, 78)), ("tiny", (1000, 79))])
def test_noalloc_matches_forward_twice(name, seeds):
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    dev = torch.device("cuda:0")
    wl = W.generate(name, seed=seeds[0])
    cfg = W.CONFIGS[name]
    layer = make_layer(wl, dev)
    weights = [to_dev(a, dev) for a in (wl.up_codes, wl.up_scales, wl.down_codes, wl.down_scales,
                                         wl.up_global, wl.down_global)]
    x = to_dev(wl.x, dev)
    # two different routings, one call each, back to back
    routings = [(wl.topk_ids, wl.topk_weights), W.make_routing(wl.n, wl.E, wl.k, cfg["bias_sigma"], seeds[1])]
    for ids_h, w_h in routings:
        ids, tw = to_dev(ids_h, dev), to_dev(w_h, dev)
        ref = to_dev(wl.dst, dev)
        layer.forward(x, ids, tw, ref)
        got = to_dev(wl.dst, dev)
        api.forward_noalloc(wl.H, wl.I, wl.E, wl.k, *weights, x, ids, tw, got)
        torch.cuda.synchronize()
        wl.topk_ids, wl.topk_weights = ids_h, w_h
        want = oracle.moe_forward(wl, out_f64=True).out_f64
        for label, out in (("no-alloc", got), ("forward", ref)):
            ok, err, rms = layer_tolerance_check(bf16_from_dev(out), want)
            assert ok, (name, label, err, rms)
    layer.close()


def test_noalloc_rejects_oversized_batches():
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    dev = torch.device("cuda:0")
    wl = W.generate("decode-1")
    weights = [to_dev(a, dev) for a in (wl.up_codes, wl.up_scales, wl.down_codes, wl.down_scales,
                                         wl.up_global, wl.down_global)]
    n = 200  # 1200 rows > the fixed array's capacity at these shapes
    x = torch.zeros((n, wl.H), dtype=torch.int16, device=dev)
    ids = torch.zeros((n, wl.k), dtype=torch.int32, device=dev)
    tw = torch.zeros((n, wl.k), dtype=torch.float32, device=dev)
    dst = torch.zeros((n, wl.H), dtype=torch.int16, device=dev)
    with pytest.raises(api.MoeError) as ei:
        api.forward_noalloc(wl.H, wl.I, wl.E, wl.k, *weights, x, ids, tw, dst)
    assert ei.value.status == 3


def test_noalloc_several_routing_slices():
    """5600 pairs at small shapes: the routing's slice histograms live in the
    fixed array too; checked against the oracle."""
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    dev = torch.device("cuda:0")
    wl = W.small_custom(700, 64, 64, 8, 8, seed=80)
    weights = [to_dev(a, dev) for a in (wl.up_codes, wl.up_scales, wl.down_codes, wl.down_scales,
                                         wl.up_global, wl.down_global)]
    got = to_dev(wl.dst, dev)
    api.forward_noalloc(wl.H, wl.I, wl.E, wl.k, *weights, to_dev(wl.x, dev), to_dev(wl.topk_ids, dev),
                        to_dev(wl.topk_weights, dev), got)
    torch.cuda.synchronize()
    ok, err, rms = layer_tolerance_check(bf16_from_dev(got), oracle.moe_forward(wl, out_f64=True).out_f64)
    assert ok, (err, rms)


def _weights(wl, dev):
    ws = [to_dev(a, dev) for a in (wl.up_codes, wl.up_scales, wl.down_codes, wl.down_scales, wl.up_global,
                                   wl.down_global)]
    gate = {}
    if wl.gated:
        gate = dict(gate_codes=to_dev(wl.gate_codes, dev), gate_scales=to_dev(wl.gate_scales, dev),
                    gate_global=to_dev(wl.gate_global, dev))
    return ws, gate


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("scales", ["full", "low"])
def test_noalloc_full_contract_weights(scales, gated):
    """Every finite e4m3 scale byte (or the subnormal-heavy low range) and a
    distinct global per (expert, matrix), two calls in a row, each against the
    oracle's unrounded output."""
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    dev = torch.device("cuda:0")
    wl = W.generate("decode-32", gated=gated, scales=scales, globals_="distinct")
    ws, gate = _weights(wl, dev)
    x = to_dev(wl.x, dev)
    for seed in (81, 82):
        ids_h, w_h = W.make_routing(wl.n, wl.E, wl.k, 0.0, seed)
        got = to_dev(wl.dst, dev)
        api.forward_noalloc(wl.H, wl.I, wl.E, wl.k, *ws, x, to_dev(ids_h, dev), to_dev(w_h, dev), got, **gate)
        torch.cuda.synchronize()
        wl.topk_ids, wl.topk_weights = ids_h, w_h
        ok, err, rms = layer_tolerance_check(bf16_from_dev(got), oracle.moe_forward(wl, out_f64=True).out_f64)
        assert ok, (seed, err, rms)


def test_noalloc_capacity_edge_at_decode_shapes():
    """At H 2688, I 1856, E 128, top-6 the fixed array holds 96 tokens (576
    rows): 96 runs and matches the oracle, 97 is MOE_ERR_CAPACITY and leaves
    dst untouched."""
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    dev = torch.device("cuda:0")
    wl = W.generate("decode-32", n=97, seed=1002)
    ws, _ = _weights(wl, dev)
    x, ids, tw = to_dev(wl.x, dev), to_dev(wl.topk_ids, dev), to_dev(wl.topk_weights, dev)
    dst = to_dev(wl.dst, dev)
    with pytest.raises(api.MoeError) as ei:
        api.forward_noalloc(wl.H, wl.I, wl.E, wl.k, *ws, x, ids, tw, dst)
    assert ei.value.status == 3
    torch.cuda.synchronize()
    assert np.array_equal(bf16_from_dev(dst), wl.dst)
    api.forward_noalloc(wl.H, wl.I, wl.E, wl.k, *ws, x, ids, tw, dst, n_tokens=96)
    torch.cuda.synchronize()
    out = bf16_from_dev(dst)
    ref = oracle.moe_forward(wl, tok_range=(0, 96), out_f64=True).out_f64
    ok, err, rms = layer_tolerance_check(out[:96], ref[:96])
    assert ok, (err, rms)
    assert np.array_equal(out[96], wl.dst[96])
