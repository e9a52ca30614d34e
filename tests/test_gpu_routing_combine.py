"""GPU parity: routing permutation (bit-exact) and WeightedRowSum against the oracle."""
import json
import os

import numpy as np
import pytest

import oracle
from nvfp4_quantized_moe_topk_gb300 import workload as W
from helpers import bf16_from_dev, make_layer, to_dev

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def dev():
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    return torch.device("cuda:0")


def _gpu_routing(layer, wl, dev, ids):
    import torch

    n, k = ids.shape
    x = to_dev(np.zeros((n, wl.H), np.uint16), dev)
    dst = to_dev(np.zeros((n, wl.H), np.uint16), dev)
    layer.forward(x, to_dev(ids, dev), to_dev(np.zeros((n, k), np.float32), dev), dst)
    counts = torch.empty(wl.E, dtype=torch.int32, device=dev)
    offsets = torch.empty(wl.E + 1, dtype=torch.int32, device=dev)
    perm = torch.full((n * k,), -7, dtype=torch.int32, device=dev)
    inv = torch.empty(n * k, dtype=torch.int32, device=dev)
    layer.debug_routing(counts, offsets, perm, inv)
    torch.cuda.synchronize()
    return counts.cpu().numpy(), offsets.cpu().numpy(), perm.cpu().numpy(), inv.cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "decode-1", "decode-32", "prefill-4314", "prefill-16384"])
def test_routing_bit_exact(dev, name):
    wl = W.generate(name, weights=False)
    # weights are irrelevant to the routing; use a zero-weight layer of the same shape
    wz = W.Workload(name, wl.n, wl.H, 64, wl.E, wl.k, wl.x, wl.topk_ids, wl.topk_weights,
                    np.zeros((wl.E, 64, wl.H // 2), np.uint8), np.full((wl.E, 64, wl.H // 16), 0x38, np.uint8),
                    np.zeros((wl.E, wl.H, 32), np.uint8), np.full((wl.E, wl.H, 4), 0x38, np.uint8),
                    wl.up_global, wl.down_global, wl.dst)
    layer = make_layer(wz, dev, gemv_max_rows=1 << 30)
    c, o, p, i = _gpu_routing(layer, wz, dev, wl.topk_ids)
    rc, ro, rp, ri, dropped = oracle.routing(wl.topk_ids, wl.E)
    assert dropped == 0
    assert np.array_equal(c, rc) and np.array_equal(o, ro)
    assert np.array_equal(p, rp) and np.array_equal(i, ri)
    assert layer.device_error() == 0
    layer.close()


@pytest.mark.parametrize("n,k,E,seed", [(257, 3, 5, 1), (1000, 8, 1024, 2), (3, 32, 7, 3), (4099, 6, 128, 4)])
def test_routing_duplicates_and_ragged(dev, n, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(n, k)).astype(np.int32)
    wl = W.Workload("r", n, 64, 64, E, k, None, ids, None, np.zeros((E, 64, 32), np.uint8),
                    np.full((E, 64, 4), 0x38, np.uint8), np.zeros((E, 64, 32), np.uint8),
                    np.full((E, 64, 4), 0x38, np.uint8), np.ones(E, np.float32), np.ones(E, np.float32), None)
    layer = make_layer(wl, dev, gemv_max_rows=1 << 30)
    c, o, p, i = _gpu_routing(layer, wl, dev, ids)
    rc, ro, rp, ri, _ = oracle.routing(ids, E)
    assert np.array_equal(c, rc) and np.array_equal(o, ro) and np.array_equal(p, rp) and np.array_equal(i, ri)
    layer.close()


def test_routing_flags_and_drops_bad_ids(dev):
    ids = np.array([[3, 3], [0, 7], [3, -1]], np.int32)
    golden = json.load(open(os.path.join(GOLDEN, "routing_hand.json")))["cases"][1]
    E = golden["E"]
    wl = W.Workload("r", 3, 64, 64, E, 2, None, ids, None, np.zeros((E, 64, 32), np.uint8),
                    np.full((E, 64, 4), 0x38, np.uint8), np.zeros((E, 64, 32), np.uint8),
                    np.full((E, 64, 4), 0x38, np.uint8), np.ones(E, np.float32), np.ones(E, np.float32), None)
    layer = make_layer(wl, dev, gemv_max_rows=1 << 30)
    c, o, p, i = _gpu_routing(layer, wl, dev, ids)
    assert c.tolist() == golden["counts"] and o.tolist() == golden["offsets"]
    assert p[:4].tolist() == golden["perm_pair"] and i.tolist() == golden["inv"]
    from nvfp4_quantized_moe_topk_gb300 import api

    assert layer.device_error() & api.DEVFLAG_BAD_ROUTING
    assert layer.device_error() == 0  # reading clears
    layer.close()


@pytest.mark.parametrize("n,k,E,seed", [(1500, 6, 40, 5), (700, 8, 8, 6)])
def test_routing_slices_drop_and_flag_bad_ids(dev, n, k, E, seed):
    """Several 4096-pair slices (histogram kernel + per-slice scatter), with
    out-of-range ids scattered over all of them: bit-exact and flagged."""
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(n, k)).astype(np.int32)
    bad = rng.random((n, k)) < 0.01
    ids[bad] = rng.choice(np.array([-1, -5, E, E + 3], np.int32), size=int(bad.sum()))
    wl = W.Workload("r", n, 64, 64, E, k, None, ids, None, np.zeros((E, 64, 32), np.uint8),
                    np.full((E, 64, 4), 0x38, np.uint8), np.zeros((E, 64, 32), np.uint8),
                    np.full((E, 64, 4), 0x38, np.uint8), np.ones(E, np.float32), np.ones(E, np.float32), None)
    layer = make_layer(wl, dev, gemv_max_rows=1 << 30)
    c, o, p, i = _gpu_routing(layer, wl, dev, ids)
    rc, ro, rp, ri, dropped = oracle.routing(ids, E)
    assert dropped == int(bad.sum()) > 0
    kept = n * k - dropped
    assert np.array_equal(c, rc) and np.array_equal(o, ro)
    assert np.array_equal(p[:kept], rp) and np.array_equal(i, ri)
    from nvfp4_quantized_moe_topk_gb300 import api

    assert layer.device_error() & api.DEVFLAG_BAD_ROUTING
    layer.close()


def test_weighted_row_sum_hand_fixtures(dev):
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    for case in json.load(open(os.path.join(GOLDEN, "weighted_row_sum_hand.json")))["cases"]:
        dst = np.array(case["dst"], np.float32)
        src = np.array(case["src"], np.float32)
        cols = dst.shape[1]
        pad = (-cols) % 8  # the kernel works on 8-column vectors
        dstp = np.pad(dst, ((0, 0), (0, pad)))
        srcp = np.pad(src, ((0, 0), (0, pad)))
        d = to_dev(W.f32_to_bf16_bits(dstp), dev)
        api.weighted_row_sum(d, to_dev(srcp, dev), to_dev(np.array(case["rows"], np.int32), dev),
                             to_dev(np.array(case["w"], np.float32), dev))
        torch.cuda.synchronize()
        got = W.bf16_bits_to_f32(bf16_from_dev(d))[:, :cols]
        assert np.array_equal(got, np.array(case["expected"], np.float32)), case["name"]


@pytest.mark.parametrize("n,k,cols,src_rows,seed", [(1, 6, 2688, 6, 0), (33, 8, 4096, 300, 1), (5, 3, 8, 4, 2)])
def test_weighted_row_sum_random(dev, n, k, cols, src_rows, seed):
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    rng = np.random.default_rng(seed)
    dst = W.f32_to_bf16_bits(rng.standard_normal((n, cols), dtype=np.float32))
    src = (rng.standard_normal((src_rows, cols)) * 100).astype(np.float32)
    rows = rng.integers(-1, src_rows + 1, size=(n, k)).astype(np.int32)  # includes out-of-range rows
    w = rng.random((n, k), dtype=np.float32)
    d = to_dev(dst, dev)
    api.weighted_row_sum(d, to_dev(src, dev), to_dev(rows, dev), to_dev(w, dev))
    torch.cuda.synchronize()
    ref, _ = oracle.weighted_row_sum(dst, src.astype(np.float64), rows, w)
    got = bf16_from_dev(d)
    g = W.bf16_bits_to_f32(got).astype(np.float64)
    r = W.bf16_bits_to_f32(ref).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(r), 1e-30))) - 7)
    assert np.all(np.abs(g - r) <= ulp)  # fp32 fma chain vs fp64: at most one final rounding apart
    assert np.mean(got == ref) > 0.99
