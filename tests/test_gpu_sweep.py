"""A seeded sweep of small random layer shapes on every path, relu^2 and
gated, against the oracle: H and I multiples of 64 up to 512, 1-40 experts,
top-1 to top-8, 1-300 tokens, routing skewed or not, the GEMV threshold at 4,
8 or off (everything on the streaming kernel), with single launches allowed
or forced off."""
import numpy as np
import pytest

import oracle
from nvfp4_quantized_moe_topk_gb300 import workload as W
from helpers import layer_tolerance_check, make_layer, run_forward

pytestmark = pytest.mark.gpu


def _cases(count=24, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        E = int(rng.integers(1, 41))
        k = int(rng.integers(1, min(E, 8) + 1))
        out.append(dict(n=int(rng.integers(1, 301)), H=64 * int(rng.integers(1, 9)), I=64 * int(rng.integers(1, 9)),
                        E=E, k=k, sigma=float(rng.choice([0.0, 1.5])), T=int(rng.choice([4, 8, 1 << 30])),
                        single=int(rng.choice([0, -1])), gated=bool(rng.integers(0, 2)), seed=3000 + i))
    return out


@pytest.mark.parametrize("c", _cases(), ids=lambda c: "n{n}_H{H}_I{I}_E{E}_k{k}_T{T}_s{single}_g{gated:d}".format(**c))
def test_random_shapes(c):
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    dev = torch.device("cuda:0")
    wl = W.small_custom(c["n"], c["H"], c["I"], c["E"], c["k"], c["seed"], bias_sigma=c["sigma"], gated=c["gated"])
    layer = make_layer(wl, dev, gemv_max_rows=c["T"], single_max_tokens=c["single"])
    got = run_forward(layer, wl, dev)
    assert layer.device_error() == 0
    layer.close()
    ok, err, rms = layer_tolerance_check(got, oracle.moe_forward(wl, out_f64=True).out_f64)
    assert ok, (err, rms)
