"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/nvfp4_ggemm.h declares, and rejects bad arguments with the
documented status before touching a device."""
import ctypes
import os
import re

import pytest

from block_scaled_fp4_grouped_gb300 import binding as nb
from block_scaled_fp4_grouped_gb300 import build as nbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    nbuild.build()
    return nb.lib()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"NVFP4_API\s+[\w\s\*]*?\b(nvfp4_\w+)\s*\(", text)
    return names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"
    assert set(names) == set(nb.EXPORTED)


def test_device_check_build_loads_and_exports_the_same_symbols(L):
    """The -DNVFP4_DEBUG build (built by the same script) is a drop-in
    replacement: same exports, same option checks."""
    path = nbuild.build(debug=True)
    D = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(D, n), f"{n} not exported by the device-check build"
    D.nvfp4_ggemm_version.restype = ctypes.c_int
    assert D.nvfp4_ggemm_version() == nb.nvfp4_ggemm_version()


def test_version_and_strings(L):
    assert nb.nvfp4_ggemm_version() >= 10000
    for st in range(0, 9):
        s = nb.nvfp4_status_string(st)
        assert s and "unknown" not in s
    assert "unknown" in nb.nvfp4_status_string(99)


def test_default_options(L):
    opt = nb.nvfp4_ggemm_default_options()
    assert opt.struct_size == ctypes.sizeof(nb.nvfp4_ggemm_options_t)
    assert opt.sf_layout == nb.NVFP4_SF_RAW and opt.sf_path == nb.NVFP4_SF_FUSED
    assert opt.wait_timeout_ns == 2_000_000_000 and opt.tile_n == 0 and opt.debug_skip_load == 0
    assert (opt.b_stages, opt.a_stages) == (0, 0)


@pytest.mark.parametrize("M,N,K,want", [
    ([], 256, 256, nb.NVFP4_ERR_INVALID_ARG),                    # no groups
    ([64] * 1025, 256, 256, nb.NVFP4_ERR_INVALID_ARG),           # too many groups
    ([-1, 64], 256, 256, nb.NVFP4_ERR_INVALID_ARG),              # negative M
    ([(1 << 20) + 1], 256, 256, nb.NVFP4_ERR_INVALID_ARG),       # M too large
    ([64], 260, 256, nb.NVFP4_ERR_UNSUPPORTED_SHAPE),            # N % 8
    ([64], 0, 256, nb.NVFP4_ERR_UNSUPPORTED_SHAPE),              # N too small
    ([64], 256, 352, nb.NVFP4_ERR_UNSUPPORTED_SHAPE),            # K % 64
    ([64], 256, 32, nb.NVFP4_ERR_UNSUPPORTED_SHAPE),             # K too small
    ([64], 256, 1 << 19, nb.NVFP4_ERR_UNSUPPORTED_SHAPE),        # K too large
])
def test_plan_rejects_bad_shapes(L, M, N, K, want):
    st, h = nb.nvfp4_ggemm_plan(0, M, N, K)
    assert st == want and h is None


def test_plan_rejects_bad_options(L):
    for field, val in [("sf_layout", 2), ("sf_path", 5), ("cache_b_scales", 3), ("tile_n", 80),
                       ("tile_n", 288), ("max_ctas", -1), ("debug_skip_load", -2), ("struct_size", 8),
                       ("b_stages", 3), ("a_stages", 9), ("debug_check_fail", 0x20), ("debug_check_fail", 0x27),
                       ("debug_check_fail", -1), ("b_static", 3), ("b_static", -1), ("row_units", 3),
                       ("row_units", -1)]:
        opt = nb.nvfp4_ggemm_default_options()
        setattr(opt, field, val)
        st, h = nb.nvfp4_ggemm_plan(0, [64], 256, 256, opt)
        assert st == nb.NVFP4_ERR_INVALID_ARG, field


def test_plan_rejects_bad_device_index(L):
    st, h = nb.nvfp4_ggemm_plan(-1, [64], 256, 256)
    assert st == nb.NVFP4_ERR_INVALID_ARG


def test_null_plan_calls(L):
    assert nb.nvfp4_ggemm_run(None, [], [], [], [], []) == nb.NVFP4_ERR_INVALID_ARG
    assert nb.nvfp4_ggemm_run_host(None, [], [], [], [], []) == nb.NVFP4_ERR_INVALID_ARG
    assert nb.nvfp4_ggemm_prepare_b_scales(None, []) == nb.NVFP4_ERR_INVALID_ARG
    assert nb.nvfp4_ggemm_sync_status(None)[0] == nb.NVFP4_ERR_INVALID_ARG
    assert nb.nvfp4_ggemm_destroy(None) == nb.NVFP4_OK
    assert L.nvfp4_ggemm_plan(None, 0, 1, None, 256, 256, None) == nb.NVFP4_ERR_INVALID_ARG


def test_relayout_argument_checks(L):
    assert nb.nvfp4_sf_relayout(0, 0, 128, 256) == nb.NVFP4_ERR_INVALID_ARG
    assert nb.nvfp4_sf_relayout(16, 32, 0, 256) == nb.NVFP4_ERR_INVALID_ARG
    assert nb.nvfp4_sf_relayout(16, 32, 128, 352) == nb.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert nb.nvfp4_sf_relayout(16, 32, 128, 0) == nb.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert nb.nvfp4_sf_relayout(17, 32, 128, 256) == nb.NVFP4_ERR_ALIGNMENT
    assert nb.nvfp4_sf_relayout(16, 40, 128, 256) == nb.NVFP4_ERR_ALIGNMENT


def test_atom_bytes(L):
    assert nb.nvfp4_sf_atom_bytes(1, 256) == 4 * 512
    assert nb.nvfp4_sf_atom_bytes(128, 256) == 4 * 512
    assert nb.nvfp4_sf_atom_bytes(129, 7168) == 2 * 112 * 512
    assert nb.nvfp4_sf_atom_bytes(4096, 7168) == 32 * 112 * 512
    assert nb.nvfp4_sf_atom_bytes(5, 100) == 0
    # K % 256 != 0: the atoms of the pages' layout, K/64 per 128-row block, unpadded
    assert nb.nvfp4_sf_atom_bytes(130, 320) == 2 * 5 * 512
    assert nb.nvfp4_sf_atom_bytes(1, 64) == 512


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.mark.skipif(_has_gpu(), reason="checks the no-device path")
def test_plan_without_device_reports_unsupported_device(L):
    st, h = nb.nvfp4_ggemm_plan(0, [64, 128], 256, 256)
    assert st == nb.NVFP4_ERR_UNSUPPORTED_DEVICE and h is None


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(nb, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(nb, "_lib", None)
    with pytest.raises(nb.NativeLibraryMissing):
        nb.lib()


def test_batched_plan_and_run_argument_checks(L):
    # batch < 1, groups x batch past the group limit, null arrays: before any device work
    for G, batch in [(1, 0), (2, -1), (512, 3), (0, 2)]:
        st, h = nb.nvfp4_ggemm_plan_batched(0, [64] * G, 256, 256, batch)
        assert st == nb.NVFP4_ERR_INVALID_ARG and h is None, (G, batch)
    assert L.nvfp4_ggemm_plan_batched(None, 0, 1, 2, None, None, None, None) == nb.NVFP4_ERR_INVALID_ARG
    assert nb.nvfp4_ggemm_run_batched(None, [], [], [], [], [], [0] * 5) == nb.NVFP4_ERR_INVALID_ARG


def test_noalloc_needs_k_multiple_of_64(L):
    # whole 64-k MMA slices, as plan/run; checked before any device work
    for K in (96, 32, 200, 0, -64):
        st, _ = nb.nvfp4_ggemm_run_noalloc([64], 256, K, [16], [16], [16], [16], [16])
        assert st == nb.NVFP4_ERR_UNSUPPORTED_SHAPE, K
