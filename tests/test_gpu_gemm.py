"""GPU parity of the tcgen05 NVFP4 GEMM (standalone nvfp4_matmul and the layer's grouped path)."""
import json
import os

import numpy as np
import pytest

import oracle
from nvfp4_quantized_moe_topk_gb300 import workload as W
from helpers import bf16_from_dev, fp_tolerance_check, layer_tolerance_check, make_layer, run_forward, to_dev

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def dev():
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    return torch.device("cuda:0")


def _matmul(dev, A, codes, scales, g, epilogue):
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    M, N = A.shape[0], codes.shape[0]
    C = torch.empty((M, N), dtype=torch.float32 if epilogue == 0 else torch.int16, device=dev)
    api.nvfp4_matmul(to_dev(A, dev), to_dev(codes, dev), to_dev(scales, dev), g, C, epilogue)
    torch.cuda.synchronize()
    out = C.cpu().numpy()
    return out if epilogue == 0 else out.view(np.uint16)


def test_hand_fixture_on_tensor_cores(dev):
    g = json.load(open(os.path.join(GOLDEN, "nvfp4_matmul_hand.json")))
    K = 64  # the fixture's 32 columns, zero-padded to one 64-wide k-block
    codes = np.zeros((16, K // 2), np.uint8)
    scales = np.full((16, K // 16), 0x38, np.uint8)
    codes[0, :16] = np.frombuffer(bytes.fromhex(g["codes_row0_hex"]), np.uint8)
    scales[0, :2] = np.frombuffer(bytes.fromhex(g["scales_row0_hex"]), np.uint8)
    x = np.zeros((1, K), np.float32)
    for i, v in g["x"].items():
        x[0, int(i)] = v
    A = W.f32_to_bf16_bits(x)
    out0 = _matmul(dev, A, codes, scales, g["global"], 0)
    assert out0[0, 0] == np.float32(g["expected_fp32"])
    out1 = _matmul(dev, A, codes, scales, g["global"], 1)
    assert int(out1[0, 0]) == int(g["expected_relu2_bf16_bits"], 16)


@pytest.mark.parametrize("M,N,K,seed", [(1, 16, 64, 0), (200, 272, 128, 1), (129, 1856, 192, 2), (385, 512, 2688, 3)])
def test_dyadic_bit_exact(dev, M, N, K, seed):
    """Dyadic inputs make every partial sum exact in fp32: the tensor-core result
    must equal the oracle bit for bit, so a lossy unpack, a wrong swizzle or a
    missing / doubled global fails (pull request #91, "Testing")."""
    rng = np.random.default_rng(seed)
    x = rng.choice(np.array([0, 1, -1, 2, -2], np.float32) / 4, size=(M, K))
    A = W.f32_to_bf16_bits(x)
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scales = W.e4m3_byte_of_pow2(rng.integers(-1, 2, (N, K // 16)))
    ref = oracle.nvfp4_matmul(A, codes, scales, 2.0 ** -4, 0)
    got = _matmul(dev, A, codes, scales, 2.0 ** -4, 0)
    assert np.array_equal(got.astype(np.float64), ref)
    ref1 = oracle.nvfp4_matmul(A, codes, scales, 2.0 ** -4, 1)
    got1 = _matmul(dev, A, codes, scales, 2.0 ** -4, 1)
    assert np.array_equal(got1, ref1)


@pytest.mark.parametrize("M,N,K,seed", [(300, 1856, 2688, 4), (77, 2688, 1856, 5), (513, 256, 4096, 6)])
def test_random_within_tolerance(dev, M, N, K, seed):
    rng = np.random.default_rng(seed)
    A = W.f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, (N, K // 16)).astype(np.uint8)
    ref = oracle.nvfp4_matmul(A, codes, scales, 0.0625, 0)
    got = _matmul(dev, A, codes, scales, 0.0625, 0)
    ok, err, rms = fp_tolerance_check(got, ref)
    assert ok, (err, rms)
    assert np.max(np.abs(got - ref)) <= 1e-5 * np.max(np.abs(ref))


def _layer_vs_oracle(wl, dev, T, sample=None):
    layer = make_layer(wl, dev, gemv_max_rows=T, single_max_tokens=-1)
    got = run_forward(layer, wl, dev)
    assert layer.device_error() == 0
    if sample is None:
        ref = oracle.moe_forward(wl, out_f64=True)
        ok, err, rms = layer_tolerance_check(got, ref.out_f64)
        assert ok, (err, rms)
    else:
        for t0, t1 in sample:
            ref = oracle.moe_forward(wl, tok_range=(t0, t1), out_f64=True)
            ok, err, rms = layer_tolerance_check(got[t0:t1], ref.out_f64[t0:t1])
            assert ok, (t0, t1, err, rms)
    again = run_forward(layer, wl, dev)
    assert np.array_equal(got, again)
    layer.close()
    return got


@pytest.mark.parametrize("T", [1, 4, 8])
def test_tiny_layer_through_grouped_gemm(dev, T):
    _layer_vs_oracle(W.generate("tiny"), dev, T)


@pytest.mark.parametrize("n,H,I,E,k,T,seed", [(70, 128, 192, 3, 2, 1, 20), (300, 256, 128, 6, 3, 16, 21),
                                               (40, 2688, 1856, 4, 2, 2, 22)])
def test_custom_layers_through_grouped_gemm(dev, n, H, I, E, k, T, seed):
    _layer_vs_oracle(W.small_custom(n, H, I, E, k, seed, bias_sigma=1.5), dev, T)


def test_prefill_4314_sampled(dev):
    wl = W.generate("prefill-4314")
    _layer_vs_oracle(wl, dev, 0, sample=[(0, 12), (2150, 2162), (4302, 4314)])


def test_prefill_16384_sampled(dev):
    wl = W.generate("prefill-16384")
    _layer_vs_oracle(wl, dev, 0, sample=[(0, 4), (9000, 9004), (16380, 16384)])


@pytest.mark.parametrize("n,H,I,E,k,T,seed", [(500, 256, 320, 3, 2, 1, 23), (250, 384, 192, 2, 1, 16, 24),
                                               (449, 128, 128, 1, 1, 1, 25), (448, 192, 256, 1, 1, 1, 26)])
def test_grouped_gemm_token_tiles_and_ragged_features(dev, n, H, I, E, k, T, seed):
    """Experts of a few hundred rows span several 224-row token tiles (the last
    one ragged; 449 rows leave a one-row tile, 448 fill two exactly), and
    I = 320 / H = 384 leave a partial 128-feature block; the
    relu^2 rows and fp32 down rows must match the oracle as well as dst."""
    import torch

    wl = W.small_custom(n, H, I, E, k, seed)
    layer = make_layer(wl, dev, gemv_max_rows=T, single_max_tokens=-1)
    got = run_forward(layer, wl, dev)
    assert layer.device_error() == 0
    ref = oracle.moe_forward(wl, intermediates=True, out_f64=True)
    ok, err, rms = layer_tolerance_check(got, ref.out_f64)
    assert ok, (err, rms)
    a = torch.empty((wl.R, wl.I), dtype=torch.int16, device=dev)
    y = torch.empty((wl.R, wl.H), dtype=torch.float32, device=dev)
    layer.debug_intermediates(a, y)
    torch.cuda.synchronize()
    ok_a, ea, ra = layer_tolerance_check(a.cpu().numpy().view(np.uint16), ref.a_f64)
    assert ok_a, ("relu^2 rows", ea, ra)
    ok_y, ey, ry = fp_tolerance_check(y.cpu().numpy(), ref.y_rows)
    assert ok_y, ("down rows", ey, ry)
    layer.close()
