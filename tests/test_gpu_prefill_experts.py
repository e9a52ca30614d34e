"""Whole experts of the prefill workloads, row by row, against fp64 references.

The sampled-token layer checks reach only a few dozen tokens of a prefill
batch; a wrong token tile or feature tile of the grouped GEMM (its later
waves, a ragged last tile) could fall between them.  Here, in the launch
configuration the benchmark times (the multi-kernel path at the default
threshold), the packed per-row intermediates of whole experts are compared:

  * relu^2 rows: Ap[r] against relu(g_up * (x[t] . W_up^T))^2 in fp64
    before rounding (bound: 1e-2 * RMS + half a bf16 ulp per element);
  * down rows: Yp[r] (fp32) against g_down * (a_ref[r] . W_down^T) in fp64,
    a_ref the reference relu^2 rows rounded to bf16 (bound: 1e-3 * the
    expert's RMS per element -- fp32 accumulation of exact bf16 products is
    far tighter than that -- plus, where the GPU's bf16 relu^2 value lies one
    rounding step from the reference's, that step carried through |W_down|).

Weights are decoded by the oracle (``oracle.dequant``, exact fp64), the
relu^2 rows rounded by the oracle package's bf16 rounding, and the
products are numpy fp64 matrix products (the library matmul serves as the
step; the pages' GEMM is a plain matrix product with the global as alpha,
gllm pull request #91, "What changes", bf16 NVFP4 GEMM).

prefill-4314: every expert above the threshold (every grouped-GEMM tile),
and a second routing in which one expert holds 224*m + 1 rows, so its last
token tile has one row.  prefill-16384: the three largest experts (the most
tiles, the latest waves) and the smallest expert above the threshold."""
import numpy as np
import pytest

import oracle
from oracle import numpy_ref
from nvfp4_quantized_moe_topk_gb300 import workload as W
from helpers import layer_tolerance_check, make_layer, to_dev

pytestmark = pytest.mark.gpu

TILE_ROWS = 224  # packed rows per grouped-GEMM token tile
T = 8  # the default threshold: experts with more rows take the grouped GEMM


@pytest.fixture(scope="module")
def dev():
    import torch

    from nvfp4_quantized_moe_topk_gb300 import api

    api.load(build_if_missing=True)
    return torch.device("cuda:0")


def _forward_rows(layer, wl, dev, experts, offsets, counts):
    """Run the layer and copy out the packed Ap / Yp rows of the given experts."""
    import torch

    x, ids, tw = to_dev(wl.x, dev), to_dev(wl.topk_ids, dev), to_dev(wl.topk_weights, dev)
    dst = to_dev(wl.dst, dev)
    layer.forward(x, ids, tw, dst)
    a = torch.empty((wl.R, wl.I), dtype=torch.int16, device=dev)
    y = torch.empty((wl.R, wl.H), dtype=torch.float32, device=dev)
    layer.debug_intermediates(a, y)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    rows = {}
    for e in experts:
        o, c = int(offsets[e]), int(counts[e])
        rows[e] = (a[o:o + c].cpu().numpy().view(np.uint16), y[o:o + c].cpu().numpy())
    return rows


def _check_expert(wl, e, perm, offsets, counts, a_gpu, y_gpu):
    o, c = int(offsets[e]), int(counts[e])
    toks = perm[o:o + c] // wl.k
    X = W.bf16_bits_to_f32(wl.x[toks]).astype(np.float64)  # the gathered rows, exactly
    Wu = oracle.dequant(wl.up_codes[e], wl.up_scales[e], wl.I, wl.H)
    Wd = oracle.dequant(wl.down_codes[e], wl.down_scales[e], wl.H, wl.I)
    h = (X @ Wu.T) * float(wl.up_global[e])
    a_raw = np.maximum(h, 0.0) ** 2
    ok_a, ea, ra = layer_tolerance_check(a_gpu, a_raw)
    assert ok_a, f"expert {e} ({c} rows): relu^2 rows max|err| {ea:.4g} vs rms {ra:.4g}"
    a_ref = numpy_ref.bf16_round(a_raw)
    gd = float(wl.down_global[e])
    yr = (a_ref @ Wd.T) * gd
    flip = np.abs(W.bf16_bits_to_f32(a_gpu).astype(np.float64) - a_ref)
    allow = abs(gd) * (flip @ np.abs(Wd).T) if flip.any() else 0.0
    rms = float(np.sqrt(np.mean(yr * yr)))
    err = np.abs(y_gpu.astype(np.float64) - yr)
    assert np.all(err <= 1e-3 * rms + allow), \
        f"expert {e} ({c} rows): down rows max|err| {err.max():.4g} vs rms {rms:.4g}"


def _run(wl, dev, experts):
    counts, offsets, perm, _, dropped = oracle.routing(wl.topk_ids, wl.E)
    assert dropped == 0
    layer = make_layer(wl, dev, gemv_max_rows=T)
    rows = _forward_rows(layer, wl, dev, experts, offsets, counts)
    layer.close()
    for e in experts:
        _check_expert(wl, e, perm, offsets, counts, *rows[e])
    return counts


def test_prefill_4314_every_grouped_gemm_expert(dev):
    wl = W.generate("prefill-4314")
    counts = np.bincount(wl.topk_ids.ravel(), minlength=wl.E)
    experts = [int(e) for e in np.nonzero(counts > T)[0]]
    assert sum(int(counts[e]) for e in experts) > 20000  # nearly all of the 25,884 rows
    _run(wl, dev, experts)


def _one_row_last_tile(wl, rng):
    """Move pairs into the largest expert until it holds 224 * m + 1 rows
    (pairs taken from other experts, never giving a token the expert twice)."""
    ids = wl.topk_ids
    counts = np.bincount(ids.ravel(), minlength=wl.E)
    e = int(np.argmax(counts))
    need = (1 - counts[e]) % TILE_ROWS  # rows to add so that count = 1 (mod 224)
    cand = [t for t in rng.permutation(wl.n) if e not in ids[t]]
    for t in cand[:need]:
        ids[t, wl.k - 1] = e
    counts = np.bincount(ids.ravel(), minlength=wl.E)
    assert counts[e] % TILE_ROWS == 1 and counts[e] > TILE_ROWS
    return e


def test_prefill_4314_expert_with_a_one_row_last_tile(dev):
    wl = W.generate("prefill-4314")
    e = _one_row_last_tile(wl, np.random.Generator(np.random.PCG64(67)))
    counts = np.bincount(wl.topk_ids.ravel(), minlength=wl.E)
    small = [int(s) for s in np.nonzero(counts > T)[0] if s != e][:2]
    _run(wl, dev, [e] + small)


def test_prefill_16384_largest_experts(dev):
    wl = W.generate("prefill-16384")
    counts = np.bincount(wl.topk_ids.ravel(), minlength=wl.E)
    order = np.argsort(-counts, kind="stable")
    above = [int(e) for e in order if counts[e] > T]
    experts = above[:3] + [above[-1]]
    assert counts[experts[0]] > 10 * TILE_ROWS
    _run(wl, dev, experts)
