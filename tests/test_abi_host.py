"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every entry point that include/*.h declares, and
reject bad arguments on the host -- before any CUDA call -- with the documented
status codes.
"""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names += re.findall(r"TW_API\s+[\w\s\*]+?\b(tw_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def tw():
    import ternary_weight_quant_b300 as tw
    return tw


def test_header_declares_entry_points():
    names = _declared_symbols()
    for expected in ["tw_pack_ternary", "tw_quant_act", "tw_rmsnorm_quant_act", "tw_ternary_gemv",
                     "tw_ternary_gemm", "tw_ternary_matmul", "tw_quant_gemv", "tw_status_string",
                     "tw_pack_workspace_bytes", "tw_device_status", "tw_gemm_workspace_bytes"]:
        assert expected in names


def test_library_exports_every_declared_symbol(tw):
    lib = ctypes.CDLL(tw.LIB_PATH)
    for name in _declared_symbols():
        assert hasattr(lib, name), name


def test_internal_launchers_are_hidden(tw):
    lib = ctypes.CDLL(tw.LIB_PATH)
    for internal in ["tw_launch_gemv", "tw_launch_pack", "tw_pack_ws_size", "tw_launch_fused_gemv"]:
        assert not hasattr(lib, internal)


def test_status_strings(tw):
    lib = tw.lib()
    for code in range(9):
        s = lib.tw_status_string(code).decode()
        assert s.startswith("TW_")
    assert lib.tw_status_string(99).decode() == "unknown tw_status"
    assert lib.tw_version() >= 100


def test_workspace_bytes(tw):
    assert tw.tw_pack_workspace_bytes(256, 256) >= 256 * 8 + 4
    assert tw.tw_pack_workspace_bytes(0, 256) == 0
    assert tw.tw_pack_workspace_bytes(4, 6) == 0
    assert tw.tw_pack_workspace_bytes(1 << 30, 1 << 12) == 0  # N*K >= 2^40


FAKE = 0x10000  # a 64 KiB-aligned non-null address; never dereferenced: these calls fail on the host


def test_null_pointers_rejected(tw):
    lib = tw.lib()
    assert lib.tw_pack_ternary(None, 4, 4, FAKE, FAKE, FAKE, 4096, None) == tw.TW_ERR_NULL
    assert lib.tw_quant_act(FAKE, 1, 16, None, FAKE, None, None) == tw.TW_ERR_NULL
    assert lib.tw_rmsnorm_quant_act(FAKE, None, 1e-6, 1, 16, FAKE, FAKE, None, None) == tw.TW_ERR_NULL
    assert lib.tw_ternary_gemv(FAKE, FAKE, None, FAKE, None, 1, 4, 16, FAKE, None, None) == tw.TW_ERR_NULL
    assert lib.tw_ternary_gemv(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 16, None, None, None) == tw.TW_ERR_NULL
    for fn in (lib.tw_ternary_gemm, lib.tw_ternary_matmul):
        assert fn(FAKE, FAKE, None, FAKE, None, 1, 4, 16, FAKE, None, None, 0, None) == tw.TW_ERR_NULL
        assert fn(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 16, None, None, None, 0, None) == tw.TW_ERR_NULL
    assert lib.tw_quant_gemv(None, None, 1e-6, FAKE, FAKE, 1, 4, 64, FAKE, None, None, None, None,
                             None) == tw.TW_ERR_NULL
    assert lib.tw_device_status(None) == tw.TW_ERR_NULL


@pytest.mark.parametrize("M,N,K", [(0, 4, 16), (1, 0, 16), (1, 4, 0), (1, 4, 6), (1, 4, 65536),
                                   (-1, 4, 16), (1, 1 << 31, 16)])
def test_bad_shapes_rejected(tw, M, N, K):
    lib = tw.lib()
    assert lib.tw_ternary_gemv(FAKE, FAKE, FAKE, FAKE, None, M, N, K, FAKE, None, None) == tw.TW_ERR_SHAPE
    for fn in (lib.tw_ternary_gemm, lib.tw_ternary_matmul):
        assert fn(FAKE, FAKE, FAKE, FAKE, None, M, N, K, FAKE, None, None, 0, None) == tw.TW_ERR_SHAPE


def test_gemv_rejects_large_m(tw):
    lib = tw.lib()
    assert lib.tw_ternary_gemv(FAKE, FAKE, FAKE, FAKE, None, 17, 4, 16, FAKE, None, None) == tw.TW_ERR_SHAPE


def test_quant_gemv_shape_checks(tw):
    lib = tw.lib()
    args = lambda M, K: (FAKE, None, 1e-6, FAKE, FAKE, M, 8, K, FAKE, None, None, None, None, None)
    assert lib.tw_quant_gemv(*args(5, 64)) == tw.TW_ERR_SHAPE     # M > 4
    assert lib.tw_quant_gemv(*args(1, 80)) == tw.TW_ERR_SHAPE     # K % 64 != 0
    assert lib.tw_quant_gemv(*args(1, 0)) == tw.TW_ERR_SHAPE
    bad = (FAKE + 4, None, 1e-6, FAKE, FAKE, 1, 8, 64, FAKE, None, None, None, None, None)
    assert lib.tw_quant_gemv(*bad) == tw.TW_ERR_ALIGN


def test_gemm_requires_k_multiple_of_16(tw):
    lib = tw.lib()
    assert lib.tw_ternary_gemm(FAKE, FAKE, FAKE, FAKE, None, 64, 4, 20, FAKE, None, None, 0, None) == tw.TW_ERR_SHAPE


def test_gemm_workspace_checks(tw):
    lib = tw.lib()
    need = tw.tw_gemm_workspace_bytes(64, 256)
    assert need == 64 * 256 * 2
    assert tw.tw_gemm_workspace_bytes(0, 256) == 0 and tw.tw_gemm_workspace_bytes(4, 6) == 0
    args = (FAKE, FAKE, FAKE, FAKE, None, 64, 4, 256, FAKE, None)
    assert lib.tw_ternary_gemm(*args, FAKE, need - 1, None) == tw.TW_ERR_WORKSPACE
    assert lib.tw_ternary_gemm(*args, FAKE + 16, need, None) == tw.TW_ERR_ALIGN


def test_pack_checks(tw):
    lib = tw.lib()
    ws = tw.tw_pack_workspace_bytes(4, 16)
    assert lib.tw_pack_ternary(FAKE, 4, 18, FAKE, FAKE, FAKE, ws, None) == tw.TW_ERR_SHAPE
    assert lib.tw_pack_ternary(FAKE, 4, 16, FAKE, FAKE, None, ws, None) == tw.TW_ERR_WORKSPACE
    assert lib.tw_pack_ternary(FAKE, 4, 16, FAKE, FAKE, FAKE, ws - 1, None) == tw.TW_ERR_WORKSPACE
    assert lib.tw_pack_ternary(FAKE + 4, 4, 16, FAKE, FAKE, FAKE, ws, None) == tw.TW_ERR_ALIGN
    assert lib.tw_pack_ternary(FAKE, 4, 16, FAKE + 1, FAKE, FAKE, ws, None) == tw.TW_ERR_ALIGN


def test_alignment_checks(tw):
    lib = tw.lib()
    assert lib.tw_quant_act(FAKE + 8, 1, 16, FAKE, FAKE, None, None) == tw.TW_ERR_ALIGN
    assert lib.tw_quant_act(FAKE, 1, 16, FAKE + 2, FAKE, None, None) == tw.TW_ERR_ALIGN
    assert lib.tw_rmsnorm_quant_act(FAKE, FAKE + 4, 1e-6, 1, 16, FAKE, FAKE, None, None) == tw.TW_ERR_ALIGN
    assert lib.tw_ternary_gemv(FAKE, FAKE + 1, FAKE, FAKE, None, 1, 4, 16, FAKE, None, None) == tw.TW_ERR_ALIGN
    assert lib.tw_ternary_gemv(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 16, FAKE + 2, None, None) == tw.TW_ERR_ALIGN
    assert lib.tw_ternary_gemm(FAKE, FAKE, FAKE + 4, FAKE, None, 64, 4, 16, FAKE, None, None, 0,
                               None) == tw.TW_ERR_ALIGN


def test_import_fails_loudly_without_the_library(tmp_path):
    """A copy of the package without libtw.so must refuse to import: there is no CPU path."""
    import shutil
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = tmp_path / "ternary_weight_quant_b300"
    pkg.mkdir()
    shutil.copy(os.path.join(root, "ternary_weight_quant_b300", "__init__.py"), pkg / "__init__.py")
    r = subprocess.run([sys.executable, "-c", "import ternary_weight_quant_b300"], cwd=str(tmp_path),
                       capture_output=True, text=True, env={**os.environ, "PYTHONPATH": str(tmp_path)})
    assert r.returncode != 0 and "libtw.so not built" in r.stderr


def test_t5_row_bytes_and_checks(tw):
    lib = tw.lib()
    assert [tw.tw_t5_row_bytes(K) for K in (4, 80, 84, 2560, 6912)] == [16, 16, 32, 512, 1392]
    assert tw.tw_t5_row_bytes(0) == 0 and tw.tw_t5_row_bytes(6) == 0 and tw.tw_t5_row_bytes(65536) == 0
    # pack: NULL, shape, workspace, alignment (packed5 must be 16-byte aligned)
    assert lib.tw_pack_ternary_t5(None, 4, 16, FAKE, FAKE, FAKE, 4096, None) == tw.TW_ERR_NULL
    assert lib.tw_pack_ternary_t5(FAKE, 4, 6, FAKE, FAKE, FAKE, 4096, None) == tw.TW_ERR_SHAPE
    assert lib.tw_pack_ternary_t5(FAKE, 4, 16, FAKE, FAKE, FAKE, 8, None) == tw.TW_ERR_WORKSPACE
    assert lib.tw_pack_ternary_t5(FAKE, 4, 16, FAKE + 4, FAKE, FAKE, 4096, None) == tw.TW_ERR_ALIGN
    # GEMV: 1 or 2 tokens, K % 16 == 0, K <= 40960, 16-byte aligned packed5 and x_q
    g = lambda M, K, p5=FAKE, xq=FAKE: lib.tw_ternary_gemv_t5(p5, FAKE, xq, FAKE, M, 8, K, FAKE, None, None)
    assert lib.tw_ternary_gemv_t5(FAKE, FAKE, None, FAKE, 1, 8, 64, FAKE, None, None) == tw.TW_ERR_NULL
    assert g(3, 64) == tw.TW_ERR_SHAPE
    assert g(1, 68) == tw.TW_ERR_SHAPE
    assert g(1, 40976) == tw.TW_ERR_SHAPE
    assert g(1, 64, p5=FAKE + 4) == tw.TW_ERR_ALIGN
    assert g(2, 64, xq=FAKE + 8) == tw.TW_ERR_ALIGN
