"""The C-ABI library loads, exports every symbol the header declares, and its
host-side validation returns the documented status without launching
anything (these calls never reach a kernel, so they run without a GPU)."""
import ctypes
import os
import re

import pytest

import weight_only_int4_gemm_gb300 as w
from weight_only_int4_gemm_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("w4a16.h", "w8a8_fp8.h")]

OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_UNSUP, ERR_WS = 0, 1, 2, 3, 4, 5
FAKE = 0x10000  # an aligned, never-dereferenced address


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b((?:w4a16|w8a8_fp8)_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    _lib.load()
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "w4a16_gemm" in names and "w4a16_pack" in names and "w4a16_dequant_ref" in names
    assert "w8a8_fp8_gemm" in names and "w8a8_fp8_quantize_act" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.SIGNATURES), "binding signatures out of sync with header"


def test_packed_bytes():
    tag = 16  # the layout tag at the end of every blob
    assert w.w4a16_packed_bytes(4096, 4096, False) == 4096 * 4096 // 2 + tag
    assert w.w4a16_packed_bytes(4096, 4096, True) == 4096 * 4096 // 2 + 32 * 512 * 4 + tag
    # zero-point rows are padded to a multiple of 4 words (16 bytes)
    assert w.w4a16_packed_bytes(128, 8, True) == 128 * 8 // 2 + 1 * 4 * 4 + tag
    assert w.w4a16_packed_bytes(256, 4104, True) == 256 * 4104 // 2 + 2 * 516 * 4 + tag
    lib = _lib.load()
    assert lib.w4a16_packed_bytes(100, 4096, 128, 0) == 0
    assert lib.w4a16_packed_bytes(128, 12, 128, 0) == 0
    assert lib.w4a16_packed_bytes(128, 8, 64, 0) == 0


def test_workspace_bytes_invalid_shapes(lib):
    bad = ctypes.c_size_t(-1).value
    assert lib.w4a16_workspace_bytes(0, 128, 8, 128) == bad
    assert lib.w4a16_workspace_bytes(1, 130, 8, 128) == bad
    assert lib.w4a16_workspace_bytes(1, 128, 9, 128) == bad
    assert lib.w4a16_workspace_bytes(1, 128, 8, 32) == bad


def _gemm(lib, x=FAKE, packed=FAKE, scales=FAKE, y=FAKE, B=1, K=128, N=8, group=128,
          ws=None, ws_bytes=0, path=-1):
    return lib.w4a16_gemm_path(x, packed, scales, 0, y, B, K, N, group, ws, ws_bytes, path, None)


def test_gemm_validation(lib):
    assert _gemm(lib, group=64) == ERR_UNSUP
    assert _gemm(lib, K=100) == ERR_SHAPE
    assert _gemm(lib, K=0) == ERR_SHAPE
    assert _gemm(lib, N=12) == ERR_SHAPE
    assert _gemm(lib, B=0) == ERR_SHAPE
    assert _gemm(lib, B=-3) == ERR_SHAPE
    assert _gemm(lib, x=None) == ERR_NULL
    assert _gemm(lib, y=None) == ERR_NULL
    assert _gemm(lib, x=FAKE + 8) == ERR_ALIGN
    assert _gemm(lib, scales=FAKE + 2) == ERR_ALIGN
    assert _gemm(lib, path=7) == ERR_UNSUP
    # a shape that splits K needs workspace: missing / too small / misaligned
    B, K, N = 1, 4096, 4096
    need = lib.w4a16_workspace_bytes(B, K, N, 128)
    assert need > 0
    assert _gemm(lib, B=B, K=K, N=N, path=0) == ERR_NULL
    assert _gemm(lib, B=B, K=K, N=N, ws=FAKE, ws_bytes=need - 1, path=0) == ERR_WS
    assert _gemm(lib, B=B, K=K, N=N, ws=FAKE + 4, ws_bytes=need, path=0) == ERR_ALIGN
    # without a tensor-core device the forced tensor-core path is refused
    assert _gemm(lib, B=64, K=4096, N=4096, path=1) == ERR_UNSUP
    assert lib.w4a16_debug_forced_timeout(FAKE, FAKE, FAKE, 0, FAKE, 64, 4096, 4096, 128,
                                          None, 0, 0, None) == ERR_UNSUP


def test_pack_and_dequant_validation(lib):
    assert lib.w4a16_pack(FAKE, None, 128, 8, 64, FAKE, None) == ERR_UNSUP
    assert lib.w4a16_pack(FAKE, None, 120, 8, 128, FAKE, None) == ERR_SHAPE
    assert lib.w4a16_pack(None, None, 128, 8, 128, FAKE, None) == ERR_NULL
    assert lib.w4a16_pack(FAKE, FAKE + 4, 128, 8, 128, FAKE, None) == ERR_ALIGN
    assert lib.w4a16_dequant_ref(FAKE, FAKE, 0, None, 128, 8, 128, None) == ERR_NULL
    assert lib.w4a16_dequant_ref(FAKE, FAKE, 0, FAKE, 128, 7, 128, None) == ERR_SHAPE
    assert lib.w4a16_dequant_ref(FAKE + 1, FAKE, 0, FAKE, 128, 8, 128, None) == ERR_ALIGN


def test_quantize_validation(lib):
    assert lib.w4a16_quantize_rtn(FAKE, 128, 8, 64, FAKE, FAKE, None) == ERR_UNSUP
    assert lib.w4a16_quantize_rtn(FAKE, 100, 8, 128, FAKE, FAKE, None) == ERR_SHAPE
    assert lib.w4a16_quantize_rtn(FAKE, 128, 12, 128, FAKE, FAKE, None) == ERR_SHAPE
    assert lib.w4a16_quantize_rtn(None, 128, 8, 128, FAKE, FAKE, None) == ERR_NULL
    assert lib.w4a16_quantize_rtn(FAKE, 128, 8, 128, FAKE + 4, FAKE, None) == ERR_ALIGN


def _grouped(lib, x=FAKE, offsets=FAKE, E=8, T=64, y=FAKE, max_rows=16, K=2048, N=1536,
             group=128, ws=FAKE, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.w4a16_grouped_workspace_bytes(T, E, max_rows, K, N, 128)
    return lib.w4a16_gemm_grouped(x, offsets, E, T, FAKE, FAKE, 0, y, max_rows, K, N, group,
                                  ws, ws_bytes, None)


def test_grouped_validation(lib):
    bad = ctypes.c_size_t(-1).value
    need = lib.w4a16_grouped_workspace_bytes(64, 8, 16, 2048, 1536, 128)
    assert 0 < need < bad
    assert lib.w4a16_grouped_workspace_bytes(64, 0, 16, 2048, 1536, 128) == bad
    assert lib.w4a16_grouped_workspace_bytes(64, 257, 16, 2048, 1536, 128) == bad
    assert lib.w4a16_grouped_workspace_bytes(0, 8, 16, 2048, 1536, 128) == bad
    assert lib.w4a16_grouped_workspace_bytes(64, 8, 16, 2048, 1536, 64) == bad
    assert _grouped(lib, group=64) == ERR_UNSUP
    assert _grouped(lib, K=100) == ERR_SHAPE
    assert _grouped(lib, N=12) == ERR_SHAPE
    assert _grouped(lib, T=0, ws_bytes=need) == ERR_SHAPE
    assert _grouped(lib, E=0, ws_bytes=need) == ERR_SHAPE
    assert _grouped(lib, E=257, ws_bytes=need) == ERR_SHAPE
    assert _grouped(lib, max_rows=0, ws_bytes=need) == ERR_SHAPE
    assert _grouped(lib, x=None) == ERR_NULL
    assert _grouped(lib, offsets=None) == ERR_NULL
    assert _grouped(lib, y=None) == ERR_NULL
    assert _grouped(lib, ws=None) == ERR_NULL
    assert _grouped(lib, x=FAKE + 8) == ERR_ALIGN
    assert _grouped(lib, offsets=FAKE + 2) == ERR_ALIGN
    assert _grouped(lib, ws=FAKE + 4) == ERR_ALIGN
    assert _grouped(lib, ws_bytes=need - 1) == ERR_WS


def test_fused_validation(lib):
    def fused(bias=FAKE, epi=1, y=FAKE, B=1, K=128, N=8, group=128):
        return lib.w4a16_gemm_fused(FAKE, FAKE, FAKE, 0, bias, epi, y, B, K, N, group, None, 0,
                                    None)
    assert fused(epi=4) == ERR_UNSUP
    assert fused(epi=-1) == ERR_UNSUP
    assert fused(bias=None) == ERR_NULL
    assert fused(bias=FAKE + 2) == ERR_ALIGN
    assert fused(epi=2, bias=None, K=100) == ERR_SHAPE   # bias not needed without the flag
    assert fused(group=64) == ERR_UNSUP
    assert fused(y=None) == ERR_NULL


def test_fp8_validation(lib):
    bad = ctypes.c_size_t(-1).value
    assert lib.w8a8_fp8_workspace_bytes(1, 4096, 4096) > 0  # small batch splits K
    assert lib.w8a8_fp8_workspace_bytes(0, 4096, 4096) == bad
    assert lib.w8a8_fp8_workspace_bytes(1, 100, 4096) == bad
    assert lib.w8a8_fp8_quantize_act(FAKE, 4, 100, FAKE, FAKE, None) == ERR_SHAPE
    assert lib.w8a8_fp8_quantize_act(FAKE, 0, 128, FAKE, FAKE, None) == ERR_SHAPE
    assert lib.w8a8_fp8_quantize_act(None, 4, 128, FAKE, FAKE, None) == ERR_NULL
    assert lib.w8a8_fp8_quantize_act(FAKE, 4, 128, FAKE + 8, FAKE, None) == ERR_ALIGN
    assert lib.w8a8_fp8_quantize_act(FAKE, 4, 128, FAKE, FAKE + 2, None) == ERR_ALIGN
    assert lib.w8a8_fp8_quantize_weight(FAKE, 128, 12, FAKE, FAKE, None) == ERR_SHAPE
    assert lib.w8a8_fp8_quantize_weight(FAKE, 128, 8, None, FAKE, None) == ERR_NULL
    assert lib.w8a8_fp8_quantize_weight(FAKE + 4, 128, 8, FAKE, FAKE, None) == ERR_ALIGN

    assert lib.w8a8_fp8_packed_bytes(256, 264) == 3 * 128 * 256
    assert lib.w8a8_fp8_packed_bytes(100, 8) == 0
    assert lib.w8a8_fp8_pack_weight(FAKE, 128, 12, FAKE, None) == ERR_SHAPE
    assert lib.w8a8_fp8_pack_weight(None, 128, 8, FAKE, None) == ERR_NULL
    assert lib.w8a8_fp8_pack_weight(FAKE, 128, 8, FAKE + 8, None) == ERR_ALIGN

    def gemm(xq=FAKE, sx=FAKE, wq=FAKE, sw=FAKE, y=FAKE, B=1, K=4096, N=4096, ws=FAKE,
             ws_bytes=None):
        if ws_bytes is None:
            ws_bytes = lib.w8a8_fp8_workspace_bytes(B, K, N)
        return lib.w8a8_fp8_gemm(xq, sx, wq, sw, y, B, K, N, ws, ws_bytes, None)

    assert gemm(K=96, ws_bytes=0) == ERR_SHAPE
    assert gemm(N=4, ws_bytes=0) == ERR_SHAPE
    assert gemm(B=0, ws_bytes=0) == ERR_SHAPE
    assert gemm(sw=None) == ERR_NULL
    assert gemm(y=None) == ERR_NULL
    assert gemm(xq=FAKE + 8) == ERR_ALIGN
    assert gemm(sx=FAKE + 1) == ERR_ALIGN
    assert gemm(ws=None) == ERR_NULL
    assert gemm(ws=FAKE + 4) == ERR_ALIGN
    need = lib.w8a8_fp8_workspace_bytes(1, 4096, 4096)
    assert gemm(ws_bytes=need - 1) == ERR_WS
    # valid arguments without tcgen05 tensor cores: refused, nothing launched
    assert gemm() == ERR_UNSUP


def test_status_strings(lib):
    for s in range(8):
        assert lib.w4a16_status_string(s)
    assert lib.w4a16_status_string(99) == b"unknown status"


def test_select_path(lib):
    assert lib.w4a16_select_path(1, 4096, 4096) == w.PATH_SKINNY
    assert lib.w4a16_select_path(0, 4096, 4096) == -1
    assert lib.w4a16_select_path(16, 100, 4096) == -1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load()


def test_packed_check_validation(lib):
    """Argument errors of the blob-tag check are reported before any copy."""
    assert lib.w4a16_packed_check(FAKE, 256, 8, 64, 0, None) == ERR_UNSUP
    assert lib.w4a16_packed_check(FAKE, 100, 8, 128, 0, None) == ERR_SHAPE
    assert lib.w4a16_packed_check(None, 256, 8, 128, 0, None) == ERR_NULL
    assert lib.w4a16_packed_check(FAKE + 4, 256, 8, 128, 0, None) == ERR_ALIGN
