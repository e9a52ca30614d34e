"""Edge cases of the layer against the oracle: the largest supported hidden and
intermediate sizes (4096) on both paths, relu^2 and gated, and the two sides
of the single-launch bound (n <= 64 tokens and n*k <= 1024 pairs)."""
import numpy as np
import pytest

import oracle
from nvfp4_quantized_moe_topk_gb300 import workload as W
from helpers import layer_tolerance_check, make_layer, run_forward

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    return torch.device("cuda:0")


def _check(wl, dev, sample=None, **kw):
    layer = make_layer(wl, dev, **kw)
    got = run_forward(layer, wl, dev)
    assert layer.device_error() == 0
    layer.close()
    ranges = sample if sample is not None else [(0, wl.n)]
    for t0, t1 in ranges:
        ref = oracle.moe_forward(wl, tok_range=(t0, t1), out_f64=True).out_f64
        ok, err, rms = layer_tolerance_check(got[t0:t1], ref[t0:t1])
        assert ok, (t0, t1, err, rms)


@pytest.mark.parametrize("gated", [False, True])
def test_max_sizes_single_launch(dev, gated):
    _check(W.small_custom(16, 4096, 4096, 4, 2, seed=110, gated=gated), dev)


@pytest.mark.parametrize("gated", [False, True])
def test_max_sizes_grouped_gemm(dev, gated):
    wl = W.small_custom(600, 4096, 4096, 4, 2, seed=111, bias_sigma=1.0, gated=gated)
    _check(wl, dev, sample=[(0, 6), (297, 303), (594, 600)], gemv_max_rows=8)


@pytest.mark.parametrize("n,k", [(64, 16), (65, 16), (64, 1), (128, 8), (129, 8)])
def test_single_launch_bound(dev, n, k):
    """n = 64, n*k = 1024 runs as one launch; 65 tokens or 1032 pairs do not."""
    _check(W.small_custom(n, 256, 192, 32, k, seed=112 + n + k), dev)
