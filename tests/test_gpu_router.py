"""GPU parity of the router kernel (moe_router_topk) against the oracle's router.

ids and counts must match bit for bit (both sides compare the same fp32 biased
logits); weights within 1e-6 relative (expf and fp32 division against fp64)."""
import json
import os

import numpy as np
import pytest

import oracle
from helpers import to_dev

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def dev():
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    return torch.device("cuda:0")


def _route(dev, logits, bias, k, with_counts=True):
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    n, E = logits.shape
    ids = torch.full((n, k), -7, dtype=torch.int32, device=dev)
    w = torch.zeros((n, k), dtype=torch.float32, device=dev)
    counts = torch.full((E,), 99, dtype=torch.int32, device=dev) if with_counts else None
    api.router_topk(to_dev(logits, dev), None if bias is None else to_dev(bias, dev), ids, w, counts)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), None if counts is None else counts.cpu().numpy()


# shapes of the layer's workloads (decode, 4314- and 16384-token prefill) and edge shapes
@pytest.mark.parametrize("n,E,k,sigma,seed", [(1, 128, 6, 0.0, 1), (32, 128, 6, 0.0, 2), (4314, 128, 6, 1.5, 3),
                                              (16384, 128, 8, 2.0, 4), (100, 1024, 32, 1.0, 5), (33, 8, 8, 0.0, 6),
                                              (7, 40, 1, 0.5, 7)])
def test_router_matches_oracle(dev, n, E, k, sigma, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    logits = rng.standard_normal((n, E), dtype=np.float32)
    bias = (rng.standard_normal(E, dtype=np.float32) * np.float32(sigma)) if sigma > 0 else None
    ids, w, counts = _route(dev, logits, bias, k)
    rids, rw, rcounts = oracle.router_topk(logits, bias, k)
    assert np.array_equal(ids, rids)
    assert np.array_equal(counts, rcounts)
    assert np.allclose(w, rw, rtol=1e-6, atol=1e-7)
    ids2, w2, _ = _route(dev, logits, bias, k)
    assert np.array_equal(ids2, ids) and np.array_equal(w2, w)  # run-to-run identical


def test_router_ties_hand_fixture(dev):
    g = json.load(open(os.path.join(GOLDEN, "router_hand.json")))
    ids, w, counts = _route(dev, np.array(g["logits"], np.float32), np.array(g["bias"], np.float32), g["k"])
    assert ids.tolist() == g["ids"] and counts.tolist() == g["counts"]
    assert np.allclose(w, np.array(g["weights"]), rtol=1e-6, atol=0)


def test_router_quantised_logits_with_many_ties(dev):
    # logits on a coarse grid: most rows have several equal values among the top-k
    rng = np.random.Generator(np.random.PCG64(11))
    logits = (rng.integers(-3, 4, size=(500, 64)) * 0.5).astype(np.float32)
    ids, w, counts = _route(dev, logits, None, 8)
    rids, rw, rcounts = oracle.router_topk(logits, None, 8)
    assert np.array_equal(ids, rids) and np.array_equal(counts, rcounts)
    assert np.allclose(w, rw, rtol=1e-6, atol=1e-7)


def test_router_without_counts_and_empty(dev):
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    rng = np.random.Generator(np.random.PCG64(12))
    logits = rng.standard_normal((10, 16), dtype=np.float32)
    ids, w, _ = _route(dev, logits, None, 4, with_counts=False)
    rids, rw, _ = oracle.router_topk(logits, None, 4)
    assert np.array_equal(ids, rids)
    empty = torch.zeros((0, 16), dtype=torch.float32, device=dev)
    api.router_topk(empty, None, torch.zeros((0, 4), dtype=torch.int32, device=dev),
                    torch.zeros((0, 4), dtype=torch.float32, device=dev))
    with pytest.raises(api.MoeError):
        api.router_topk(to_dev(logits, dev), None, torch.zeros((10, 17), dtype=torch.int32, device=dev),
                        torch.zeros((10, 17), dtype=torch.float32, device=dev))


@pytest.mark.parametrize("n", [1, 8, 9, 200])
def test_router_counts_overwrite_stale_values(dev, n):
    """Up to 8 tokens run as one block that writes the histogram itself, more
    as several blocks adding into a zeroed one: either way whatever the
    counts buffer held before is gone."""
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    rng = np.random.Generator(np.random.PCG64(20 + n))
    logits = rng.standard_normal((n, 96), dtype=np.float32)
    ids = torch.empty((n, 6), dtype=torch.int32, device=dev)
    w = torch.empty((n, 6), dtype=torch.float32, device=dev)
    counts = torch.full((96,), 7, dtype=torch.int32, device=dev)
    api.router_topk(to_dev(logits, dev), None, ids, w, counts)
    torch.cuda.synchronize()
    _, _, rcounts = oracle.router_topk(logits, None, 6)
    assert np.array_equal(counts.cpu().numpy(), rcounts)
