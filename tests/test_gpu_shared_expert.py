"""The shared expert (the FFN every token passes through at weight 1, whose
output is the pre-filled dst the routed experts are added onto) and the two
layers captured in one CUDA graph, against the oracle.

The oracle's shared expert is its layer at E = 1, k = 1, weight 1, onto a
zero dst; the composition is the routed layer's oracle with that result as
its pre-filled dst."""
import numpy as np
import pytest

import oracle
from nvfp4_quantized_moe_topk_gb300 import workload as W
from helpers import bf16_from_dev, layer_tolerance_check, make_layer, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    return torch.device("cuda:0")


def _shared(n, H, I, seed, gated=False):
    wl = W.small_custom(n, H, I, 1, 1, seed, gated=gated)
    wl.topk_ids[:] = 0
    wl.topk_weights[:] = 1.0
    wl.dst[:] = 0
    return wl


def _run_shared(wl, dev):
    import torch

    layer = make_layer(wl, dev)
    out = to_dev(np.full((wl.n, wl.H), 0x7FC0, np.uint16), dev)  # NaN everywhere: every element must be written
    layer.shared_expert_forward(to_dev(wl.x, dev), out)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    layer.close()
    return bf16_from_dev(out)


@pytest.mark.parametrize("n,H,I,gated,seed", [(1, 2688, 1856, False, 90), (32, 2688, 1856, False, 91),
                                               (300, 1024, 512, False, 92), (17, 256, 192, True, 93),
                                               (700, 512, 256, True, 94)])
def test_shared_expert_matches_oracle(dev, n, H, I, gated, seed):
    wl = _shared(n, H, I, seed, gated)
    got = _run_shared(wl, dev)
    ref = oracle.moe_forward(wl, out_f64=True).out_f64
    ok, err, rms = layer_tolerance_check(got, ref)
    assert ok, (err, rms)


def test_shared_expert_prefill_4314_sampled(dev):
    base = W.generate("prefill-4314")
    wl = W.Workload("shared", base.n, base.H, base.I, 1, 1, base.x, np.zeros((base.n, 1), np.int32),
                    np.ones((base.n, 1), np.float32), base.up_codes[:1], base.up_scales[:1], base.down_codes[:1],
                    base.down_scales[:1], base.up_global[:1], base.down_global[:1],
                    np.zeros((base.n, base.H), np.uint16))
    got = _run_shared(wl, dev)
    for t0, t1 in [(0, 16), (2000, 2010), (4306, 4314)]:
        ref = oracle.moe_forward(wl, tok_range=(t0, t1), out_f64=True).out_f64
        ok, err, rms = layer_tolerance_check(got[t0:t1], ref[t0:t1])
        assert ok, (t0, err, rms)


@pytest.mark.parametrize("name", ["decode-32", "tiny"])
def test_shared_then_routed_in_one_graph(dev, name):
    """dst = shared(x), then dst += routed(x): both captured in one CUDA graph."""
    import torch

    routed = W.generate(name)
    sh = _shared(routed.n, routed.H, routed.I, seed=95)
    sh.x = routed.x
    shared_layer = make_layer(sh, dev)
    routed_layer = make_layer(routed, dev)
    x = to_dev(routed.x, dev)
    # the shared stage on its own first: against the oracle, and its bits
    # (deterministic, the same inside the graph) pre-fill the oracle's routed stage
    stage1 = to_dev(np.zeros((routed.n, routed.H), np.uint16), dev)
    shared_layer.shared_expert_forward(x, stage1)
    torch.cuda.synchronize()
    dst0 = bf16_from_dev(stage1)
    ok0, err0, rms0 = layer_tolerance_check(dst0, oracle.moe_forward(sh, out_f64=True).out_f64)
    assert ok0, ("shared stage", err0, rms0)
    comp = W.generate(name)
    comp.dst = dst0
    ref = oracle.moe_forward(comp, out_f64=True).out_f64

    ids, tw = to_dev(routed.topk_ids, dev), to_dev(routed.topk_weights, dev)
    dst = to_dev(np.zeros((routed.n, routed.H), np.uint16), dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):  # warm once outside the capture
        shared_layer.shared_expert_forward(x, dst, stream=stream)
        routed_layer.forward(x, ids, tw, dst, stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        shared_layer.shared_expert_forward(x, dst, stream=stream)
        routed_layer.forward(x, ids, tw, dst, stream=stream)
    dst.fill_(0x7FC0)
    g.replay()
    torch.cuda.synchronize()
    got = bf16_from_dev(dst)
    ok, err, rms = layer_tolerance_check(got, ref)
    assert ok, (err, rms)
    g.replay()  # replays give the same bits
    torch.cuda.synchronize()
    assert np.array_equal(bf16_from_dev(dst), got)
    shared_layer.close()
    routed_layer.close()


def test_shared_expert_needs_a_one_expert_top1_handle(dev):
    from nvfp4_quantized_moe_topk_gb300 import api

    wl = W.generate("tiny")
    layer = make_layer(wl, dev)
    with pytest.raises(api.MoeError) as ei:
        layer.shared_expert_forward(to_dev(wl.x, dev), to_dev(wl.dst, dev))
    assert ei.value.status == 2
    layer.close()
