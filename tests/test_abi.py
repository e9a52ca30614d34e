"""The C ABI library builds for sm_103a, loads, and exports every declared entry point.

Host-only checks: argument validation paths that return before any CUDA call.
No compute runs here (there may be no GPU)."""
import ctypes
import os
import re

import pytest

from nvfp4_quantized_moe_topk_gb300 import api
from nvfp4_quantized_moe_topk_gb300 import build as B

HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:MOE_API\s+)?(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, re.M):
            names.append(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    B.build()
    return api.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert set(api.ENTRY_POINTS) <= set(names)


def test_status_strings(lib):
    for s in range(8):
        assert api.status_string(s)
    assert api.status_string(3).startswith("n_tokens")


def test_null_handle_and_bad_sizes_rejected_before_any_cuda_call(lib):
    vp = ctypes.c_void_p
    assert lib.moe_nvfp4_forward(None, None, None, None, None, 1, None) == 1
    assert lib.moe_nvfp4_forward_host(None, None, None, None, None, 1, None) == 1
    assert lib.moe_nvfp4_destroy(None) == 0
    flags = ctypes.c_int32()
    assert lib.moe_nvfp4_get_device_error(None, ctypes.byref(flags)) == 1
    # nvfp4_matmul: K not a multiple of 64 / N not a multiple of 16 / bad epilogue / M = 0
    assert lib.nvfp4_matmul(vp(16), vp(16), vp(16), ctypes.c_float(1.0), vp(16), 4, 32, 96, 0, None) == 2
    assert lib.nvfp4_matmul(vp(16), vp(16), vp(16), ctypes.c_float(1.0), vp(16), 4, 24, 128, 0, None) == 2
    assert lib.nvfp4_matmul(vp(16), vp(16), vp(16), ctypes.c_float(1.0), vp(16), 4, 32, 128, 7, None) == 1
    assert lib.nvfp4_matmul(None, None, None, ctypes.c_float(1.0), None, 0, 32, 128, 0, None) == 0
    # weighted_row_sum: cols not a multiple of 8, n < 0, n = 0
    assert lib.weighted_row_sum(vp(16), vp(16), vp(16), vp(16), 2, 2, 12, 4, None) == 2
    assert lib.weighted_row_sum(vp(16), vp(16), vp(16), vp(16), -1, 2, 16, 4, None) == 1
    assert lib.weighted_row_sum(None, None, None, None, 0, 2, 16, 4, None) == 0


def test_create_validates_shapes_first(lib):
    w = api.Weights(16, 16, 16, 16, 16, 16)
    h = ctypes.c_void_p(123)
    for cfg, want in [((96, 128, 8, 2, 32, 0), 2),      # H not a multiple of 64
                      ((256, 128, 2000, 2, 32, 0), 2),  # too many experts
                      ((256, 128, 8, 0, 32, 0), 1),     # k = 0
                      ((256, 128, 8, 2, -1, 0), 1)]:    # negative capacity
        c = api.Config(*cfg)
        assert lib.moe_nvfp4_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h)) == want
        assert h.value is None
    c = api.Config(256, 128, 8, 2, 32, 0)
    assert lib.moe_nvfp4_create(ctypes.byref(c), None, None, ctypes.byref(h)) == 1
    # activation: not one of the MOE_ACT_ values / gated without gate weights
    c = api.Config(256, 128, 8, 2, 32, 0, 0, 7)
    assert lib.moe_nvfp4_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h)) == 1
    c = api.Config(256, 128, 8, 2, 32, 0, 0, api.ACT_SWIGLU)
    assert lib.moe_nvfp4_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h)) == 1
    assert h.value is None
    wg = api.Weights(16, 16, 16, 16, 16, 16, 16, None, 16)
    assert lib.moe_nvfp4_create(ctypes.byref(c), ctypes.byref(wg), None, ctypes.byref(h)) == 1
    vp = ctypes.c_void_p
    assert lib.moe_nvfp4_shared_expert_forward(None, vp(16), vp(16), 4, None) == 1
    assert lib.moe_nvfp4_debug_offset_grid_barrier(None, 1) == 1
    assert lib.moe_nvfp4_forward_noalloc(ctypes.byref(c), ctypes.byref(w), vp(16), vp(16), vp(16), vp(16), 4,
                                         None) == 1


def test_noalloc_rejects_misaligned_pointers_before_any_cuda_call(lib):
    """Codes, x and dst need 16-byte alignment, scales 2, globals / ids /
    weights 4: anything else is MOE_ERR_INVALID_ARG, with nothing enqueued
    (these fake addresses are never dereferenced)."""
    vp = ctypes.c_void_p
    c = api.Config(256, 128, 8, 2, 32, 0)
    good = dict(up_codes=256, up_scales=256, down_codes=256, down_scales=256, up_global=256, down_global=256)
    fields = [f for f, _ in api.Weights._fields_]
    for name, bad in [("up_scales", 257), ("down_scales", 259), ("up_global", 258), ("down_global", 262),
                      ("up_codes", 264), ("down_codes", 260)]:
        w = api.Weights(*[dict(good, **{name: bad}).get(f) for f in fields])
        assert lib.moe_nvfp4_forward_noalloc(ctypes.byref(c), ctypes.byref(w), vp(256), vp(256), vp(256),
                                             vp(256), 4, None) == 1, name
    w = api.Weights(*[good.get(f) for f in fields])
    for args in [(vp(256), vp(258), vp(256), vp(256)),   # ids not 4-byte aligned
                 (vp(256), vp(256), vp(254), vp(256)),   # weights not 4-byte aligned
                 (vp(264), vp(256), vp(256), vp(256)),   # x not 16-byte aligned
                 (vp(256), vp(256), vp(256), vp(248))]:  # dst not 16-byte aligned
        assert lib.moe_nvfp4_forward_noalloc(ctypes.byref(c), ctypes.byref(w), *args, 4, None) == 1
    cg = api.Config(256, 128, 8, 2, 32, 0, 0, api.ACT_SWIGLU)
    wg = api.Weights(*[dict(good, gate_codes=256, gate_scales=257, gate_global=256).get(f) for f in fields])
    assert lib.moe_nvfp4_forward_noalloc(ctypes.byref(cg), ctypes.byref(wg), vp(256), vp(256), vp(256), vp(256),
                                         4, None) == 1


def test_library_is_built_for_sm103a_only():
    assert "arch=compute_103a,code=sm_103a" in " ".join(B.ARCH)
    assert os.path.exists(B.LIB)


def test_header_is_plain_c(tmp_path):
    """The boundary header compiles as strict C99 (no C++ or CUDA types in the signatures)."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = tmp_path / "use_header.c"
    src.write_text('#include "moe_nvfp4.h"\nint main(void) { return MOE_OK; }\n')
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", f"-I{inc}", "-fsyntax-only",
                        str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
