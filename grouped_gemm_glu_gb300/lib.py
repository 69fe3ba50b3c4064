"""ctypes binding of libmoeglu.so (the C ABI declared in include/moeglu.h).

Argument marshalling only: every step runs in the library's CUDA kernels.
``load()`` raises if the shared library has not been built; there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import math
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoeglu.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "moeglu.h")

MOE_OK, MOE_ERR_ARG, MOE_ERR_CUDA, MOE_ERR_CAPACITY, MOE_ERR_TIMEOUT, MOE_ERR_UNSUPPORTED = 0, 1, 2, 4, 8, 16
ACT = {"swiglu": 0, "geglu": 1, "geglu_tanh": 2, "srelu": 3, "sreglu": 4, "none": 5}
OUT_BF16, OUT_MXFP8, OUT_NVFP4 = 0, 1, 2


class GluParams(C.Structure):
    _fields_ = [("act", C.c_int32), ("alpha", C.c_float), ("up_offset", C.c_float),
                ("gate_lo", C.c_float), ("gate_hi", C.c_float), ("up_lo", C.c_float), ("up_hi", C.c_float)]


class ActOut(C.Structure):
    _fields_ = [("q_row", C.c_void_p), ("s_row", C.c_void_p), ("q_col", C.c_void_p), ("s_col", C.c_void_p),
                ("y", C.c_void_p), ("amax", C.c_void_p), ("pre", C.c_void_p), ("row_dot", C.c_void_p),
                ("rht_amax", C.c_void_p), ("rht_signs", C.c_uint32)]


IN_BF16, IN_MXFP8, IN_NVFP4, IN_MXFP8_TILED, IN_NVFP4_TILED = 0, 1, 2, 3, 4


class InT(C.Structure):
    _fields_ = [("dtype", C.c_int32), ("data", C.c_void_p), ("scale", C.c_void_p), ("global_scale", C.c_void_p)]


def in_operand(data_ptr: int, scale_ptr: int | None = None, global_scale_ptr: int | None = None,
               tiled: bool = False) -> InT:
    """A GEMM operand: bf16 when scale_ptr is None, MXFP8 codes + scales
    (tiled: scales already in the tensor-core order, a weight cast with
    col = 2), or NVFP4 codes + block scales + per-tensor scale when
    global_scale_ptr is set (tiled: a weight from moe_nvfp4_cast_cols_tiled)."""
    if scale_ptr is None:
        return InT(IN_BF16, data_ptr, None, None)
    if global_scale_ptr is None:
        return InT(IN_MXFP8_TILED if tiled else IN_MXFP8, data_ptr, scale_ptr, None)
    return InT(IN_NVFP4_TILED if tiled else IN_NVFP4, data_ptr, scale_ptr, global_scale_ptr)


def glu_params(act: str = "swiglu", alpha: float = 1.0, up_offset: float = 0.0,
               gate_lo: float = -math.inf, gate_hi: float = math.inf,
               up_lo: float = -math.inf, up_hi: float = math.inf) -> GluParams:
    return GluParams(ACT[act], alpha, up_offset, gate_lo, gate_hi, up_lo, up_hi)


P, I, U64, SZ, F32 = C.c_void_p, C.c_int, C.c_uint64, C.c_size_t, C.c_float

_SIGS = {
    "moe_repack_fc1": [P, P, I, I, I, I, P],
    "moe_route_workspace_size": ([I, I, I], SZ),
    "moe_route_permute": [P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, SZ, P, P],
    "moe_grouped_fc1_glu_quant_fwd": [P, P, P, P, P, P, I, I, I, I, C.POINTER(GluParams), I, C.POINTER(ActOut), P,
                                      SZ, I, P, P],
    "moe_grouped_fc1_workspace_size": ([I, I, I], SZ),
    "moe_grouped_dglu_quant_bwd": [P, P, P, P, P, P, I, I, I, I, C.POINTER(GluParams), I, C.POINTER(ActOut), P, P, SZ,
                                   I, P, P],
    "moe_grouped_dglu_workspace_size": ([I, I], SZ),
    "moe_quantize_mxfp8": [P, I, I, I, I, P, P, I, P, P, P, P],
    "moe_quantize_mxfp8_dual": [P, I, I, I, P, P, P, P, P, P],
    "moe_mxfp8_tiled_scale_bytes": ([I, I, I], SZ),
    "moe_grouped_fc1_glu_quant_fwd_mxfp8": [P, P, P, P, P, P, P, P, I, I, I, I, C.POINTER(GluParams), I,
                                            C.POINTER(ActOut), P, SZ, I, P, P],
    "moe_grouped_fc2_workspace_size": ([I, I, I, I], SZ),
    "moe_grouped_fc2_fwd": [C.POINTER(InT), C.POINTER(InT), P, P, I, I, I, I, I, C.POINTER(ActOut), P, SZ, I, P, P],
    "moe_grouped_wgrad_workspace_size": ([I, I, I, I], SZ),
    "moe_grouped_wgrad": [P, P, P, P, P, P, I, I, I, I, P, I, P, SZ, I, P, P],
    "moe_unpermute_combine": [P, P, P, I, I, I, P, P, P],
    "moe_combine_bwd": [P, P, P, P, P, P, I, I, I, I, I, P, P, P, P, P, P],
    "moe_permute_bwd": [P, P, I, I, I, P, P, P],
    "moe_dglu_row_dot_parts": ([I], I),
    "moe_feature_scale_grad": [P, I, P, I, I, P, P],
    "moe_nvfp4_cast": [P, P, P, P, I, I, I, P, P, P, P],
    "moe_glu_act": [P, P, P, I, I, I, C.POINTER(GluParams), P, P],
    "moe_amax_bf16": [P, SZ, P, P],
    "moe_rht_amax_cols": [P, I, I, P, I, C.c_uint32, P, P, P],
    "moe_nvfp4_rht_cast_cols": [P, I, I, P, I, P, C.c_uint32, P, P, P, P, P],
    "moe_grouped_wgrad_nvfp4": [P, P, P, P, P, P, P, P, I, I, I, I, P, I, P, SZ, I, P, P],
    "moe_nvfp4_cast_cols": [P, I, I, I, P, P, P, P, P, P],
    "moe_nvfp4_cast_cols_tiled": [P, I, I, I, P, P, P, P, P, P],
    "moe_nvfp4_tiled_scale_bytes": ([I, I, I], SZ),
    "moe_dglu_act": [P, P, P, P, I, I, I, C.POINTER(GluParams), P, P],
    "moe_route_permute_noalloc": [P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P],
    "moe_route_noalloc_max_scratch_bytes": ([], SZ),
    "moe_get_status": [P, P, P],
    "moe_set_wait_limit_ns": ([U64], None),
    "moe_wait_selftest": [I, P, P, P],
    "moe_set_cta_pairs": ([I], None),
    "moe_set_tail_swap": [I],
    "moe_launch_count": ([], U64),
}

_lib = None


def header_symbols(path: str = HEADER) -> list[str]:
    """Function names declared in the public header."""
    txt = open(path).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", txt, flags=re.M)))


def load():
    """Loads the library (once) and declares the signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with grouped_gemm_glu_gb300.build.build() "
                           "(the CUDA library is the only implementation)")
    lib = C.CDLL(LIB_PATH)
    for name, sig in _SIGS.items():
        fn = getattr(lib, name)
        if isinstance(sig, tuple):
            fn.argtypes, fn.restype = sig
        else:
            fn.argtypes, fn.restype = sig, C.c_int
    _lib = lib
    return lib


class MoeError(RuntimeError):
    pass


def check(rc: int, what: str):
    if rc != MOE_OK:
        raise MoeError(f"{what} failed with status {rc}")
