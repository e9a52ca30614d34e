"""Host logic of bench.py that the reported numbers rest on (CPU only): the
per-kernel work model behind `roofline.achieved`, and the lookup of the
committed ncu traffic, which must go null once a kernel's sources change."""
import hashlib
import json
import os
import types

import numpy as np

import bench


def _wl(n, H, I, E, k, gated=False):
    return types.SimpleNamespace(n=n, H=H, I=I, E=E, k=k, gated=gated)


def test_work_model_hand_case():
    # 70 tokens, top-2: expert 0 holds 100 pairs, expert 1 35, expert 2 5; with
    # T = 8 experts 0 and 1 run on the grouped GEMMs, expert 2 on the streaming kernel
    n, H, I, E, k, T = 70, 256, 128, 3, 2, 8
    ids = np.array([0] * 100 + [1] * 35 + [2] * 5, np.int32).reshape(n, k)
    w = bench.algorithmic_work(_wl(n, H, I, E, k), [ids], T)
    mat = H * I // 2 + H * I // 16  # codes + e4m3 block scales of one matrix
    assert w["gemm_up"][1] == 2.0 * 135 * I * H
    assert w["gemm_down"][1] == 2.0 * 135 * H * I
    assert w["gather"][0] == n * H * 2 + n * k * H * 2  # x once per token, one row per pair
    assert w["combine"][0] == n * H * 4 + n * k * H * 4 + n * k * 8
    assert w["small_experts"][0] == (mat + 5 * (H * 2 + I * 2)) + (mat + 5 * (I * 2 + H * 4))
    assert w["routing"][0] == n * k * 16


def test_work_model_gated_up_reads_two_matrices():
    n, H, I, E, k, T = 70, 256, 128, 3, 2, 8
    ids = np.array([0] * 100 + [1] * 35 + [2] * 5, np.int32).reshape(n, k)
    plain = bench.algorithmic_work(_wl(n, H, I, E, k), [ids], T)
    gated = bench.algorithmic_work(_wl(n, H, I, E, k, gated=True), [ids], T)
    assert gated["gemm_up"][1] == 2 * plain["gemm_up"][1]
    assert gated["gemm_down"][1] == plain["gemm_down"][1]
    mat = H * I // 2 + H * I // 16
    assert gated["small_experts"][0] == plain["small_experts"][0] + mat


def test_work_model_single_launch_counts_only_the_layer_bytes():
    """A batch run as one launch: the touched experts' weights once, x read,
    dst read and written, 8 B of ids and weights per pair -- no intermediates."""
    n, H, I, E, k, T = 2, 256, 128, 8, 3, 8
    ids = np.array([[0, 3, 5], [3, 6, 1]], np.int32)  # five experts touched
    mat = H * I // 2 + H * I // 16
    w = bench.algorithmic_work(_wl(n, H, I, E, k), [ids], T)
    assert set(w) == {"decode"}
    assert w["decode"][0] == 5 * 2 * mat + 3 * n * H * 2 + 8 * n * k
    g = bench.algorithmic_work(_wl(n, H, I, E, k, gated=True), [ids], T)
    assert g["decode"][0] == 5 * 3 * mat + 3 * n * H * 2 + 8 * n * k


def _fake_tree(tmp_path, text):
    csrc = tmp_path / "nvfp4_quantized_moe_topk_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("gemm2.cu", "common.cuh", "kernels.h"):
        (csrc / f).write_text(text + f)
    h = hashlib.sha256()
    for f in ("gemm2.cu", "common.cuh", "kernels.h"):
        h.update((csrc / f).read_bytes())
    return csrc, h.hexdigest()[:16]


def test_traffic_lookup_by_workload_and_kernel(tmp_path, monkeypatch):
    csrc, sha = _fake_tree(tmp_path, "v1 ")
    (tmp_path / "profiles").mkdir()
    rec = lambda kern, b: {"kernel": kern, "source": "gemm2.cu", "bytes_per_launch": b, "source_sha": sha}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"w": rec("gemm_up", 100), "w:gemm_down": rec("gemm_down", 200)}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("w", "gemm_up") == 100.0
    assert bench.profiled_traffic("w", "gemm_down") == 200.0
    assert bench.profiled_traffic("w", "decode") is None  # no capture of that kernel
    assert bench.profiled_traffic("other", "gemm_up") is None
    (csrc / "kernels.h").write_text("changed")  # sources differ from the captured ones
    assert bench.profiled_traffic("w", "gemm_up") is None
    assert bench.profiled_traffic("w", "gemm_down") is None
