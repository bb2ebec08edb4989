"""The C-ABI library builds, loads and exports every declared entry point, and
host-side argument validation answers without touching a GPU."""
import ctypes
import os
import re

import pytest

import int8_rotated_quantized_gb300 as cr
from int8_rotated_quantized_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "convrot.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return cr.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CONVROT_API\s+[\w\s\*]+?\b(convrot_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for must in ["convrot_quantize_weight", "convrot_linear_fwd", "convrot_linear_bwd_x", "convrot_embedding_lookup",
                 "convrot_prepare_bwd_weight", "convrot_gemm_s32", "convrot_get_error", "convrot_status_string",
                 "convrot_linear_fwd_noalloc", "convrot_selftest_wait_timeout", "convrot_dequant_weight_t",
                 "convrot_gemm_bf16", "convrot_linear_bwd_x_bf16", "convrot_bwd_x_bf16_workspace_bytes",
                 "convrot_linear_workspace_bytes", "convrot_widen_codes", "convrot_gemm_dequant_w16",
                 "convrot_linear_fwd_lora", "convrot_linear_lora_workspace_bytes", "convrot_linear_bwd_x_r2",
                 "convrot_bwd_x_r2_workspace_bytes", "convrot_selftest_gemm_fault",
                 "convrot_probe_mma_s8_rate", "convrot_selftest_bounds_flag"]:
        assert must in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name


def test_checked_variant_exports_every_declared_symbol(L):
    """The bounds-checked build (-DCONVROT_CHECKED) is a drop-in replacement."""
    assert os.path.exists(cr.library_path("checked"))
    C = ctypes.CDLL(cr.library_path("checked"))
    for name in declared_symbols():
        assert hasattr(C, name), name
    C.convrot_status_string.restype = ctypes.c_char_p
    assert C.convrot_status_string(6) == b"CONVROT_ERR_BOUNDS"


def test_status_strings_and_version(L):
    assert cr.status_string(0) == "CONVROT_OK"
    assert cr.status_string(1) == "CONVROT_ERR_INVALID_ARG"
    assert cr.status_string(4) == "CONVROT_ERR_TIMEOUT"
    assert cr.status_string(5) == "CONVROT_ERR_INDEX"
    assert cr.status_string(6) == "CONVROT_ERR_BOUNDS"
    assert cr.status_string(99) == "CONVROT_ERR_UNKNOWN"
    assert L.convrot_version() >= 100


def test_workspace_sizes(L):
    assert L.convrot_act_workspace_bytes(4096, 4096) == 4096 * 4096 * 2 + 4096 * 4
    assert L.convrot_act_workspace_bytes(3, 16) % 256 == 0
    assert L.convrot_act_workspace_bytes(3, 16) >= 3 * 16 * 2 + 3 * 4
    # two words per column of the backward weight, 256-aligned
    assert L.convrot_bwd_weight_workspace_bytes(16384, 4096) == 2 * 4096 * 4
    assert L.convrot_gemm_s32_workspace_bytes(64, 256) == 64 * 256 * 2
    assert L.convrot_act_workspace_bytes(-1, 4) == 0


FAKE = ctypes.c_void_p(1 << 20)  # an aligned non-null address; never dereferenced on invalid input


@pytest.mark.parametrize("block", [0, 3, 12, 512, 1024])
def test_bad_block_is_rejected(L, block):
    rc = L.convrot_quantize_weight(FAKE, 4, 256, 256, block, None, None, 0, 1.0, 1.0, FAKE, FAKE, None)
    assert rc == cr.ERR_INVALID_ARG


def test_bad_shapes_are_rejected(L):
    # K not a multiple of the block, K not a multiple of 16, ldw < K, row too long
    assert L.convrot_quantize_weight(FAKE, 4, 96, 96, 64, None, None, 0, 1.0, 1.0, FAKE, FAKE, None) == 1
    assert L.convrot_quantize_weight(FAKE, 4, 40, 40, 8, None, None, 0, 1.0, 1.0, FAKE, FAKE, None) == 1
    assert L.convrot_quantize_weight(FAKE, 4, 256, 128, 32, None, None, 0, 1.0, 1.0, FAKE, FAKE, None) == 1
    assert L.convrot_quantize_weight(FAKE, 4, 65536, 65536, 128, None, None, 0, 1.0, 1.0, FAKE, FAKE, None) == 1
    # LoRA pair incomplete, rank out of range
    assert L.convrot_quantize_weight(FAKE, 4, 256, 256, 32, FAKE, None, 4, 1.0, 1.0, FAKE, FAKE, None) == 1
    assert L.convrot_quantize_weight(FAKE, 4, 256, 256, 32, FAKE, FAKE, 0, 1.0, 1.0, FAKE, FAKE, None) == 1
    # GEMM: N not a multiple of 16, K not a multiple of 16
    assert L.convrot_gemm_dequant(FAKE, FAKE, 8, 256, FAKE, FAKE, 24, None, FAKE, None) == 1
    assert L.convrot_gemm_dequant(FAKE, FAKE, 8, 200, FAKE, FAKE, 32, None, FAKE, None) == 1
    # forward: workspace too small or misaligned
    need = L.convrot_act_workspace_bytes(8, 256)
    assert L.convrot_linear_fwd(FAKE, 8, 256, FAKE, FAKE, 32, 32, None, FAKE, FAKE, need - 1, None) == 1
    assert L.convrot_linear_fwd(FAKE, 8, 256, FAKE, FAKE, 32, 32, None, FAKE, ctypes.c_void_p((1 << 20) + 16),
                                need, None) == 1
    # integer GEMM entries: K beyond the int32-safe limit (127 * 127 * K < 2^31 for K <= 2^17)
    assert L.convrot_gemm_s32(FAKE, FAKE, 1, 16, 1 << 18, FAKE, FAKE, 1 << 30, None) == 1
    assert L.convrot_gemm_s32(FAKE, FAKE, 1, 16, (1 << 17) + 16, FAKE, FAKE, 1 << 30, None) == 1
    assert L.convrot_gemm_dequant(FAKE, FAKE, 8, (1 << 17) + 16, FAKE, FAKE, 32, None, FAKE, None) == 1
    assert L.convrot_gemm_dequant_w16(FAKE, FAKE, 8, (1 << 17) + 16, FAKE, FAKE, 32, None, FAKE, None) == 1
    # bf16 backward: N not a multiple of 16, K not a multiple of the block, workspace too small
    assert L.convrot_dequant_weight_t(FAKE, FAKE, 24, 256, 32, FAKE, None) == 1
    assert L.convrot_dequant_weight_t(FAKE, FAKE, 32, 80, 32, FAKE, None) == 1
    assert L.convrot_gemm_bf16(FAKE, 8, 24, FAKE, 32, FAKE, None) == 1
    assert L.convrot_gemm_bf16(FAKE, 8, 32, FAKE, 24, FAKE, None) == 1
    # LoRA bypass: rank out of range, K not a multiple of 32, workspace too small
    need_l = L.convrot_linear_lora_workspace_bytes(8, 256, 32)
    # + the bf16 parts of the down-projection (8 rows) and of B (32 rows), 128 bytes per row, each 256-aligned
    assert need_l == L.convrot_linear_workspace_bytes(8, 256, 32) + 1024 + 4096
    assert L.convrot_linear_fwd_lora(FAKE, 8, 256, FAKE, FAKE, 32, 32, None, FAKE, FAKE, 17, 1.0, 1.0, FAKE, FAKE,
                                     need_l, None) == 1
    assert L.convrot_linear_fwd_lora(FAKE, 8, 48, FAKE, FAKE, 32, 16, None, FAKE, FAKE, 4, 1.0, 1.0, FAKE, FAKE,
                                     1 << 30, None) == 1
    assert L.convrot_linear_fwd_lora(FAKE, 8, 256, FAKE, FAKE, 32, 32, None, FAKE, FAKE, 4, 1.0, 1.0, FAKE, FAKE,
                                     need_l - 1, None) == 1
    assert L.convrot_widen_codes(FAKE, 24, FAKE, None) == 1
    # second reading of the int8 backward: N not a multiple of 32, workspace too small
    need_r2 = L.convrot_bwd_x_r2_workspace_bytes(8, 512, 256)
    assert L.convrot_linear_bwd_x_r2(FAKE, 8, 48, FAKE, FAKE, 256, 32, FAKE, FAKE, 1 << 30, None) == 1
    assert L.convrot_linear_bwd_x_r2(FAKE, 8, 512, FAKE, FAKE, 256, 32, FAKE, FAKE, need_r2 - 1, None) == 1
    need = L.convrot_bwd_x_bf16_workspace_bytes(64, 256)
    assert need == 64 * 256 * 2
    assert L.convrot_linear_bwd_x_bf16(FAKE, 8, 64, FAKE, FAKE, 256, 32, FAKE, FAKE, need - 1, None) == 1


def test_null_and_misaligned_pointers_are_rejected(L):
    assert L.convrot_quantize_activation(None, 4, 256, 256, 32, FAKE, FAKE, None) == 1
    assert L.convrot_quantize_activation(ctypes.c_void_p((1 << 20) + 2), 4, 256, 256, 32, FAKE, FAKE, None) == 1
    assert L.convrot_embedding_lookup(None, 4, FAKE, FAKE, 10, 256, 128, FAKE, None) == 1
    assert L.convrot_prepare_bwd_weight(FAKE, FAKE, 256, 256, 32, FAKE, FAKE, None, 1 << 30, None) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(cr, "_libs", {})
    monkeypatch.setattr(cr, "library_path", lambda variant="release": str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        cr.lib()
