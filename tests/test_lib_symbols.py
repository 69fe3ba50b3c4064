"""The C-ABI library builds, loads without a GPU and exports every function
the public header declares (no compute call is made)."""
import ctypes

import pytest

from grouped_gemm_glu_gb300 import build as B
from grouped_gemm_glu_gb300 import lib as L


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def test_header_declares_the_hot_path(lib):
    names = L.header_symbols()
    for n in ("moe_route_permute", "moe_grouped_fc1_glu_quant_fwd", "moe_grouped_fc2_fwd",
              "moe_grouped_dglu_quant_bwd", "moe_unpermute_combine", "moe_grouped_wgrad", "moe_quantize_mxfp8",
              "moe_nvfp4_cast", "moe_repack_fc1", "moe_combine_bwd", "moe_permute_bwd"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(L.LIB_PATH)
    missing = [n for n in L.header_symbols() if not hasattr(raw, n)]
    assert not missing, missing
    assert set(L.header_symbols()) == set(L._SIGS), "binding signatures out of sync with the header"


def test_workspace_size_is_host_only(lib):
    # pure host arithmetic: callable without a device
    assert lib.moe_route_workspace_size(8192, 8, 32) >= 4 * 32 * (8192 * 8 // 2048)


def test_argument_validation_needs_no_device(lib):
    # a null pointer is rejected on the host before anything is launched
    assert lib.moe_unpermute_combine(None, None, None, 1, 8, 1, None, None, None) == L.MOE_ERR_ARG
    assert lib.moe_quantize_mxfp8_dual(None, 1, 32, 32, None, None, None, None, None, None) == L.MOE_ERR_ARG
    assert lib.moe_combine_bwd(None, None, None, None, None, None, 1, 8, 1, 1, 128, None, None, None,
                               None, None, None) == L.MOE_ERR_ARG
    assert lib.moe_permute_bwd(None, None, 1, 8, 1, None, None, None) == L.MOE_ERR_ARG
    prm = L.glu_params("swiglu")
    out = L.ActOut()
    assert lib.moe_grouped_fc1_glu_quant_fwd(None, None, None, None, None, None, 4, 256, 512, 1152,
                                             ctypes.byref(prm), 1, ctypes.byref(out), None, 0, 0, None,
                                             None) == L.MOE_ERR_ARG
    assert lib.moe_wait_selftest(0, None, None, None) == L.MOE_ERR_ARG
    assert lib.moe_quantize_mxfp8(None, 1, 32, 32, 0, None, None, 0, None, None, None, None) == L.MOE_ERR_ARG
    assert lib.moe_grouped_fc2_fwd(None, None, None, None, 4, 512, 256, 1152, 0, None, None, 0, 0, None,
                                   None) == L.MOE_ERR_ARG
    # mixed operand types (one bf16, one MXFP8) are rejected: one type per MMA
    a_bf, w_mx = L.in_operand(0x10000), L.in_operand(0x10000, 0x20000)
    assert lib.moe_grouped_fc2_fwd(ctypes.byref(a_bf), ctypes.byref(w_mx), 0x10000, 0x10000, 4, 512, 256, 1152, 0,
                                   ctypes.byref(out), None, 0, 0, None, None) == L.MOE_ERR_ARG
    assert lib.moe_grouped_wgrad(None, None, None, None, None, None, 4, 512, 256, 1152, None, 0, None, 0, 0, None,
                                 None) == L.MOE_ERR_ARG
    # shape and alignment rules are host checks too (these addresses are never dereferenced)
    a16, a8 = 0x10000, 0x10008
    assert lib.moe_glu_act(a16, a16, a16, 1, 48, 64, ctypes.byref(prm), a16, None) == L.MOE_ERR_ARG  # F % 32
    assert lib.moe_glu_act(a16, a16, a16, 1, 64, 64, ctypes.byref(prm), a8, None) == L.MOE_ERR_ARG  # y unaligned
    assert lib.moe_glu_act(a8, a16, a16, 1, 64, 64, ctypes.byref(prm), a16, None) == L.MOE_ERR_ARG  # pre unaligned
    assert lib.moe_dglu_act(a8, a16, a16, a16, 1, 64, 64, ctypes.byref(prm), a16, None) == L.MOE_ERR_ARG
    assert lib.moe_nvfp4_cast(a16, a16, a16, a16, 1, 40, 64, a16, a16, a16, None) == L.MOE_ERR_ARG  # N % 16
    assert lib.moe_repack_fc1(a16, a16, 1, 32, 64, 0, None) == L.MOE_ERR_ARG  # in place
