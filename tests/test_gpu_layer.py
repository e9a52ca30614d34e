"""GPU parity of the whole layer (routing -> up -> relu^2 -> down -> combine) against the oracle.

Full-size configs are compared in full where the oracle finishes in seconds
(tiny, decode-1, decode-32) and on sampled tokens otherwise (each token's
output depends only on its own row and routing), with the same launch
configuration the benchmark times.  Intermediates (relu^2 rows, down rows)
are compared too.  Batches with at most 1024 pairs and no expert above the
GEMV threshold run as the single-launch small-batch kernel; larger ones take
the multi-kernel path (routing, GEMV, combine), covered by its own cases."""
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


def _intermediates(layer, wl, dev):
    import torch

    a = torch.empty((wl.R, wl.I), dtype=torch.int16, device=dev)
    y = torch.empty((wl.R, wl.H), dtype=torch.float32, device=dev)
    layer.debug_intermediates(a, y)
    torch.cuda.synchronize()
    return a.cpu().numpy().view(np.uint16), y.cpu().numpy()


def _check_layer(wl, dev, gemv_max_rows=0, sample=None, check_intermediates=True):
    layer = make_layer(wl, dev, gemv_max_rows=gemv_max_rows)
    got = run_forward(layer, wl, dev)
    assert layer.device_error() == 0
    if sample is None:
        ref = oracle.moe_forward(wl, intermediates=check_intermediates, out_f64=True)
        rows = None
    else:
        rows = sample
        ref = None
    if rows is None:
        ok, err, rms = layer_tolerance_check(got, ref.out_f64)
        assert ok, f"layer output: max|err| {err} vs rms {rms}"
        if check_intermediates:
            a, y = _intermediates(layer, wl, dev)
            okr, e2, r2 = layer_tolerance_check(a, ref.a_f64)
            assert okr, f"relu^2 rows: {e2} vs rms {r2}"
            oky, e3, r3 = fp_tolerance_check(y, ref.y_rows)
            assert oky, f"down rows: {e3} vs rms {r3}"
    else:
        for (t0, t1) in rows:
            part = oracle.moe_forward(wl, tok_range=(t0, t1), out_f64=True)
            ok, err, rms = layer_tolerance_check(got[t0:t1], part.out_f64[t0:t1])
            assert ok, f"tokens {t0}:{t1}: max|err| {err} vs rms {rms}"
    layer.close()
    return got


def test_tiny_single_launch(dev):
    _check_layer(W.generate("tiny"), dev, gemv_max_rows=1 << 30)


def test_tiny_default_threshold(dev):
    _check_layer(W.generate("tiny"), dev)


def test_decode_1(dev):
    _check_layer(W.generate("decode-1"), dev)


def test_decode_32(dev):
    _check_layer(W.generate("decode-32"), dev)


@pytest.mark.parametrize("n,H,I,E,k,seed", [(1, 64, 64, 1, 1, 10), (7, 128, 192, 5, 3, 11), (13, 320, 256, 9, 4, 12),
                                             (2, 4096, 2048, 4, 2, 13)])
def test_small_shapes_single_launch(dev, n, H, I, E, k, seed):
    _check_layer(W.small_custom(n, H, I, E, k, seed), dev, gemv_max_rows=1 << 30)


@pytest.mark.parametrize("n,H,I,E,k,seed", [(40, 64, 64, 32, 32, 34), (300, 128, 192, 5, 4, 35),
                                             (129, 1024, 512, 16, 8, 36)])
def test_pairs_above_single_launch_limit_use_general_path(dev, n, H, I, E, k, seed):
    # more than 1024 pairs: routing kernel, GEMV up / down, combine
    wl = W.small_custom(n, H, I, E, k, seed)
    assert wl.R > 1024
    _check_layer(wl, dev, gemv_max_rows=1 << 30, check_intermediates=wl.R * (H + I) < 1 << 22)


def test_decode_duplicates_force_multiple_token_passes(dev):
    # every pair on one expert: 40 rows of expert 1, five 8-token passes per tile
    wl = W.small_custom(20, 128, 128, 3, 2, seed=30)
    wl.topk_ids[:] = 1
    _check_layer(wl, dev, gemv_max_rows=1 << 30)


def test_decode_max_pairs_and_many_experts(dev):
    wl = W.small_custom(32, 64, 64, 1024, 32, seed=31)
    assert wl.R == 1024
    _check_layer(wl, dev, gemv_max_rows=1 << 30, check_intermediates=False)


def test_decode_bad_ids_dropped_and_flagged(dev):
    from nvfp4_quantized_moe_topk_gb300 import api

    wl = W.small_custom(8, 128, 64, 4, 2, seed=32)
    wl.topk_ids[1] = [7, -1]
    wl.topk_ids[3, 0] = 4
    layer = make_layer(wl, dev, gemv_max_rows=1 << 30)
    got = run_forward(layer, wl, dev)
    assert layer.device_error() & api.DEVFLAG_BAD_ROUTING
    ref = oracle.moe_forward(wl, out_f64=True)
    ok, err, rms = layer_tolerance_check(got, ref.out_f64)
    assert ok, (err, rms)
    assert np.array_equal(got[1], wl.dst[1])  # both of token 1's pairs dropped: dst row untouched
    layer.close()


def test_decode_all_ids_invalid_leaves_dst(dev):
    from nvfp4_quantized_moe_topk_gb300 import api

    wl = W.small_custom(4, 64, 64, 2, 2, seed=33)
    wl.topk_ids[:] = 2
    layer = make_layer(wl, dev, gemv_max_rows=1 << 30)
    got = run_forward(layer, wl, dev)
    assert np.array_equal(got, wl.dst)
    assert layer.device_error() & api.DEVFLAG_BAD_ROUTING
    layer.close()


def test_decode_repeated_calls_are_identical(dev):
    wl = W.generate("decode-1")
    layer = make_layer(wl, dev)
    first = run_forward(layer, wl, dev)
    for _ in range(4):
        assert np.array_equal(run_forward(layer, wl, dev), first)
    assert layer.device_error() == 0
    layer.close()


def test_duplicate_expert_ids(dev):
    wl = W.small_custom(6, 128, 64, 4, 3, seed=14)
    wl.topk_ids[2] = [1, 1, 1]
    wl.topk_ids[4] = [0, 3, 0]
    _check_layer(wl, dev)


def test_zero_and_negative_weights(dev):
    wl = W.small_custom(5, 128, 64, 4, 2, seed=15)
    wl.topk_weights[0] = 0
    wl.topk_weights[1] = -wl.topk_weights[1]
    _check_layer(wl, dev)


@pytest.mark.parametrize("name,pinned", [("decode-32", True), ("decode-1", True), ("tiny", True),
                                         ("decode-1", False), ("decode-32", False)])
def test_deterministic_and_forward_host_matches(dev, name, pinned):
    """Host-buffer calls give the device forward's bits: small ones (inputs
    <= 64 KB: decode-1, tiny) go through one packed pinned copy each way,
    larger ones copy each array."""
    import torch

    wl = W.generate(name)
    layer = make_layer(wl, dev)
    a = run_forward(layer, wl, dev)
    b = run_forward(layer, wl, dev)
    assert np.array_equal(a, b)
    host = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    xh = host(torch.from_numpy(wl.x.view(np.int16)))
    ih = host(torch.from_numpy(wl.topk_ids))
    wh = host(torch.from_numpy(wl.topk_weights))
    dh = host(torch.from_numpy(wl.dst.view(np.int16).copy()))
    layer.forward_host(xh, ih, wh, dh)
    assert np.array_equal(dh.numpy().view(np.uint16), a)
    layer.close()


@pytest.mark.parametrize("pinned", [True, False])
def test_forward_host_multi_kernel_path(dev, pinned):
    """A batch on the multi-kernel path through host buffers: dst goes in on
    the side stream and comes back in four combine ranges; same bits as the
    device forward."""
    import torch

    wl = W.small_custom(301, 256, 192, 8, 4, seed=21, bias_sigma=1.0)
    layer = make_layer(wl, dev)
    a = run_forward(layer, wl, dev)
    host = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    xh = host(torch.from_numpy(wl.x.view(np.int16)))
    ih = host(torch.from_numpy(wl.topk_ids))
    wh = host(torch.from_numpy(wl.topk_weights))
    dh = host(torch.from_numpy(wl.dst.view(np.int16).copy()))
    layer.forward_host(xh, ih, wh, dh)
    assert np.array_equal(dh.numpy().view(np.uint16), a)
    assert layer.device_error() == 0
    layer.close()


def test_n_zero_and_capacity(dev):
    from nvfp4_quantized_moe_topk_gb300 import api

    wl = W.small_custom(4, 64, 64, 2, 1, seed=16)
    layer = make_layer(wl, dev)
    x = to_dev(wl.x, dev)
    dst = to_dev(wl.dst, dev)
    layer.forward(x, to_dev(wl.topk_ids, dev), to_dev(wl.topk_weights, dev), dst, n_tokens=0)
    assert np.array_equal(bf16_from_dev(dst), wl.dst)
    with pytest.raises(api.MoeError) as ei:
        layer.forward(x, to_dev(wl.topk_ids, dev), to_dev(wl.topk_weights, dev), dst, n_tokens=5)
    assert ei.value.status == 3
    layer.close()


@pytest.mark.parametrize("name,single", [("decode-32", 0), ("tiny", -1)])
def test_concurrent_streams_match_serial(dev, name, single):
    """Two handles on two streams, enqueued back to back so they can overlap,
    give the same bits as the same calls made one after the other."""
    import torch

    wl = W.generate(name)
    routing2 = W.make_routing(wl.n, wl.E, wl.k, W.CONFIGS[name]["bias_sigma"], seed=4242)
    layers = [make_layer(wl, dev, single_max_tokens=single) for _ in range(2)]
    x = to_dev(wl.x, dev)
    ids = [to_dev(wl.topk_ids, dev), to_dev(routing2[0], dev)]
    tw = [to_dev(wl.topk_weights, dev), to_dev(routing2[1], dev)]
    serial = []
    for i in range(2):
        d = to_dev(wl.dst, dev)
        layers[i].forward(x, ids[i], tw[i], d)
        torch.cuda.synchronize()
        serial.append(bf16_from_dev(d))
    streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
    dsts = [to_dev(wl.dst, dev) for _ in range(2)]
    torch.cuda.synchronize()
    for i in range(2):
        layers[i].forward(x, ids[i], tw[i], dsts[i], stream=streams[i])
    torch.cuda.synchronize()
    for i in range(2):
        assert np.array_equal(bf16_from_dev(dsts[i]), serial[i]), f"handle {i}"
        assert layers[i].device_error() == 0
        layers[i].close()


@pytest.mark.parametrize("case", ["twelve_tokens", "all_ids_invalid", "packed_multi_kernel"])
def test_forward_host_packed_cases(dev, case):
    """Small host calls (one packed pinned copy in): the single launch writes
    the result straight into the mapped staging copy of dst -- with more than 8
    tokens through the second-barrier combine, and with no valid pair at all
    (nothing written: the staged pre-filled values are the result); a batch
    forced onto the multi-kernel path copies dst back instead.  Same bits as
    the device forward."""
    import torch

    wl = W.small_custom(12 if case == "twelve_tokens" else 5, 128, 64, 6, 2, seed=23)
    if case == "all_ids_invalid":
        wl.topk_ids[:] = -1
    kw = dict(single_max_tokens=-1) if case == "packed_multi_kernel" else {}
    layer = make_layer(wl, dev, **kw)
    a = run_forward(layer, wl, dev)
    if case == "all_ids_invalid":
        assert np.array_equal(a, wl.dst)
    dh = torch.from_numpy(wl.dst.view(np.int16).copy()).pin_memory()
    layer.forward_host(torch.from_numpy(wl.x.view(np.int16)).pin_memory(),
                       torch.from_numpy(wl.topk_ids).pin_memory(),
                       torch.from_numpy(wl.topk_weights).pin_memory(), dh)
    assert np.array_equal(dh.numpy().view(np.uint16), a)
    flags = layer.device_error()
    layer.close()
    assert flags == 0 or (case == "all_ids_invalid" and flags == 1)  # 1: out-of-range ids reported
