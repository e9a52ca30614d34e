"""The allocation-free entry point against the handle-based forward.

Callers that cannot call cudaMalloc (a plugin whose host owns all device
memory, a fixed memory budget) use moe_nvfp4_forward_noalloc, which keeps its
intermediates in the library's fixed device array.  Its output must match the
existing forward's within the layer tolerance, on two calls in a row (the
array keeps the previous call's contents, so the second call checks that
nothing stale leaks through).  Collected last on purpose."""
import numpy as np
import pytest

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
        ok, err, rms = layer_tolerance_check(bf16_from_dev(got), bf16_from_dev(ref))
        assert ok, (name, err, rms)
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

    import oracle
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
    ok, err, rms = layer_tolerance_check(bf16_from_dev(got), oracle.moe_forward(wl).dst)
    assert ok, (err, rms)
