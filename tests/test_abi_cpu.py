"""Host-side checks of the C ABI (no GPU needed, no compute calls).

The library must build for sm_103a, load, and export every function the header
declares; host validation must reject bad arguments before touching the device.
"""
import ctypes
import os

import pytest

import w4a8_quantized_gemm_gb300 as eg
from w4a8_quantized_gemm_gb300 import builder


@pytest.fixture(scope="module")
def lib():
    builder.build()
    return eg.load()


def test_library_exports_every_header_function(lib):
    names = eg.header_functions()
    assert len(names) >= 16
    raw = ctypes.CDLL(eg.LIB_PATH)
    missing = [n for n in names if not hasattr(raw, n)]
    assert not missing, missing
    assert lib.egopq_version() >= 10000


def test_packed_size_and_shape_gate(lib):
    assert lib.egopq_packed_w4_bytes(3584, 3584, 128) == 3584 * 3584 // 2 + 28 * 3584 * 5 // 2
    assert lib.egopq_packed_w4_bytes(152064, 3584, 128) == 152064 * 3584 // 2 + 28 * 152064 * 5 // 2
    assert lib.egopq_packed_w4_bytes(80, 3584, 128) == 0       # N does not tile 128 rows
    assert lib.egopq_packed_w4_bytes(128, 200, 128) == 0
    assert lib.egopq_packed_w4_bytes(128, 256, 64) == 0


def test_host_validation_rejects_before_launch(lib):
    A = 0x10000  # aligned fake device address: never dereferenced on these paths
    s = None
    # NULL and misaligned pointers
    assert lib.egopq_pack_w4(None, A, A, 128, 128, 128, A, s) == -1
    assert lib.egopq_pack_w4(A + 4, A, A, 128, 128, 128, A, s) == -3
    # shape gate
    assert lib.egopq_pack_w4(A, A, A, 100, 128, 128, A, s) == -2
    assert lib.egopq_quant_act_i8(A, 4, 200, 128, A, A, A, None, s) == -2
    # the codes may be left out only when the operand form is written
    assert lib.egopq_quant_act_i8(A, 4, 256, 128, None, A, A, None, s) == -1
    assert b"a_q and a_tc" in lib.egopq_last_error_string()
    assert lib.egopq_w4a8_gemm_ex(A, A, A, A, A, 4, 256, 512, 32, A, 0, s) == -2
    assert lib.egopq_w4a8_gemm_ex(A, A, A, A, A, -1, 256, 512, 128, A, 0, s) == -1
    # unknown path is refused on the host
    assert lib.egopq_w4a8_gemm_ex(A, A, A, A, A, 4, 256, 512, 128, A, 7, s) == -1
    assert b"path" in lib.egopq_last_error_string()
    # empty batch: accepted as a no-op without touching any pointer
    assert lib.egopq_w4a8_gemm_ex(None, None, None, None, None, 0, 256, 512, 128, None, 0, s) == 0
    assert lib.egopq_quant_act_i8(None, 0, 512, 128, None, None, None, None, s) == 0
    assert lib.egopq_selftest_timeout(0, s) == -1


def test_auto_path_and_operand_queries(lib):
    """The AUTO choice and the tensor-core operand form come from the library
    (host-only queries, no device touched)."""
    GEMV, TC = eg.PATH_GEMV, eg.PATH_TC
    assert [lib.egopq_auto_path(m, eg.VARIANT_W4A8) for m in (1, 4, 5, 16, 4096)] == \
        [GEMV, GEMV, TC, TC, TC]
    assert [lib.egopq_auto_path(m, eg.VARIANT_W8A8) for m in (1, 64, 65)] == [GEMV, GEMV, TC]
    assert [lib.egopq_auto_path(m, eg.VARIANT_W4A16) for m in (1, 4, 5)] == [GEMV, GEMV, TC]
    assert [lib.egopq_auto_path(m, eg.VARIANT_W8A16) for m in (1, 4, 5)] == [GEMV, GEMV, TC]
    assert lib.egopq_auto_path(1, 9) == -1
    assert lib.egopq_auto_path(-1, eg.VARIANT_W4A8) == -1
    assert lib.egopq_tc_operand_bytes(16, 3584, 128) == 2 * 16 * 3584
    assert lib.egopq_tc_operand_bytes(16, 3500, 128) == 0
    assert lib.egopq_tc_operand_bytes(0, 3584, 128) == 0
    assert lib.egopq_tc_operand_form(64) == eg.TC_FORM_E4M3_PLANES
    assert lib.egopq_tc_operand_form(65) == eg.TC_FORM_F16
    assert lib.egopq_tc_operand_form(0) == -1
    # token tile of the tensor-core path: by M up to 64, then a wide tile
    # (192 or 128 tokens, from the grid on the device's SMs) or 128
    W4A8, W8A16, W8A8 = eg.VARIANT_W4A8, eg.VARIANT_W8A16, eg.VARIANT_W8A8
    assert [lib.egopq_tc_token_tile(m, 3584, 3584, W4A8) for m in (1, 16, 17, 64)] == \
        [16, 16, 32, 64]
    assert lib.egopq_tc_token_tile(256, 256, 512, W4A8) == 128     # same tiles at either width
    assert lib.egopq_tc_token_tile(4096, 152064, 3584, W4A8) == 192
    # the down projection at 2048 tokens: 192-token tiles leave a short last
    # round, which a split second launch takes (cheaper than 128-token tiles)
    assert lib.egopq_tc_token_tile(2048, 3584, 18944, W4A8) == 192
    assert lib.egopq_tc_token_tile(4096, 12288, 3072, W8A16) == 192
    assert lib.egopq_tc_token_tile(64, 3584, 3584, W8A8) == -2      # GEMV only up to 64
    assert lib.egopq_tc_token_tile(65, 3584, 3584, W8A8) == 128      # one m-tile at either width
    assert lib.egopq_tc_token_tile(4096, 12288, 3072, W8A8) == 192
    assert lib.egopq_tc_token_tile(0, 3584, 3584, W4A8) == -1
    assert lib.egopq_tc_token_tile(16, 3500, 3584, W4A8) == -2
    assert lib.egopq_tc_token_tile(16, 3584, 3584, 9) == -1
    # launches of the tensor-core GEMM: a split second launch for the short
    # last round of a long-K persistent grid, one launch otherwise
    assert lib.egopq_tc_launches(2048, 3584, 18944, W4A8) == 2
    assert lib.egopq_tc_launches(4096, 152064, 3584, W4A8) == 1
    assert lib.egopq_tc_launches(16, 3584, 18944, W4A8) == 1
    assert lib.egopq_tc_launches(4096, 3584, 18944, W8A16) == 1
    assert lib.egopq_tc_launches(0, 3584, 3584, W4A8) == -1
    assert lib.egopq_tc_launches(64, 3584, 3584, W8A8) == -2


def test_sizes_beyond_the_limit_are_unsupported_shapes(lib):
    A, s = 0x10000, None
    big = 1 << 31
    assert lib.egopq_w4a8_gemm_ex(A, A, A, A, A, 4, big, 512, 128, A, 0, s) == -2
    assert lib.egopq_w4a8_linear(A, A, 4, big, 512, 128, A, A, 1 << 20, 0, s) == -2
    assert lib.egopq_w4a8_linear_noalloc(A, A, 4, big, 512, 128, A, 0, s) == -2
    assert lib.egopq_w4a8_linear_noalloc(A, A, big, 256, 512, 128, A, 0, s) == -2
    assert b"2^31" in lib.egopq_last_error_string()
    assert lib.egopq_quant_act_i8(A, big, 512, 128, A, A, A, None, s) == -2


def test_release_build_has_no_debug_hooks(lib):
    assert lib.egopq_debug_build() == 0
    assert lib.egopq_debug_set_record_limit(4096) == -1
    assert b"debug build" in lib.egopq_last_error_string()


def test_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(eg, "LIB_PATH", os.path.join(os.path.dirname(eg.LIB_PATH), "nope.so"))
    monkeypatch.setattr(eg, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        eg.load()


def test_header_names_follow_the_pages_operations():
    names = set(eg.header_functions())
    for required in ["egopq_pack_w4", "egopq_quant_act_i8", "egopq_w4a8_gemm",
                     "egopq_w4a16_gemm", "egopq_w8a16_gemm"]:
        assert required in names
