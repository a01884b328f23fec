"""ctypes loader for libdg.so (argument marshalling only).

The library is built in-tree by ``moe_grouped_gemm_fp8_gb300.build``; if it
is missing this module raises instead of falling back to anything else.  With
``DG_DEBUG_LIBRARY=1`` in the environment when the library is first loaded,
the build with device-side checks (``libdg_debug.so``) is loaded instead.
"""
import ctypes as C
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
DEBUG = os.environ.get("DG_DEBUG_LIBRARY", "0") not in ("", "0")
LIB_PATH = os.path.join(HERE, "libdg_debug.so" if DEBUG else "libdg.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "dg.h")

_LIB = None

DG_OK = 0
STATUS_NAMES = {
    0: "DG_OK", 1: "DG_ERR_INVALID_ARG", 2: "DG_ERR_ALIGNMENT", 3: "DG_ERR_UNSUPPORTED_ARCH",
    4: "DG_ERR_CUDA", 5: "DG_ERR_DEVICE_TIMEOUT", 6: "DG_ERR_DEVICE_BAD_INDEX",
    7: "DG_ERR_TOO_LARGE", 8: "DG_ERR_DEVICE_BAD_SCALE", 9: "DG_ERR_DEVICE_CHECK",
}
DG_SF_FP32 = 0
DG_SF_UE8M0_PACKED = 1

_p = C.c_void_p
_i64 = C.c_int64
_i32 = C.c_int32
_st = C.c_int

SIGNATURES = {
    "dg_fp8_gemm_nt": (_st, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _p]),
    "dg_fp8_gemm_nt_ws": (_st, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _p,
                                C.c_uint64, _p]),
    "dg_fp8_gemm_nt_static_ws": (_st, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _p]),
    "dg_fp8_gemm_nt_workspace_size": (_st, [_i64, _i64, _i64, _i32, _i32, C.POINTER(C.c_uint64)]),
    "dg_plan_fp8_gemm_nt_ws": (_st, [_i64, _i64, _i64, _i32, _i32, _p, _p, _p, _p, _p, _p, _p]),
    "dg_fp8_gemm_nt_fp32_sf": (_st, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _p]),
    "dg_fp8_gemm_nn": (_st, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _p]),
    "dg_fp8_gemm_tn": (_st, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _p]),
    "dg_fp8_gemm_tt": (_st, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _p]),
    "dg_m_grouped_fp8_gemm_nt_contiguous": (_st, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _p]),
    "dg_m_grouped_fp8_gemm_nt_masked": (_st, [_p, _p, _p, _p, _p, _p, _i32, _i64, _i64, _i64, _i64, _p]),
    "dg_k_grouped_fp8_gemm_tn_contiguous": (_st, [_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _p]),
    "dg_quantize_fp8": (_st, [_p, _p, _p, _i64, _i64, _i64, _i32, _i32, _p]),
    "dg_quantize_fp8_cols": (_st, [_p, _p, _p, _i64, _i64, _i32, _p]),
    "dg_transform_sf": (_st, [_p, _p, _i64, _i64, _i64, _i32, _p]),
    "dg_get_tma_aligned_size": (_i64, [_i64, _i32]),
    "dg_get_mk_alignment_for_contiguous_layout": (_i32, []),
    "dg_set_mk_alignment_for_contiguous_layout": (_st, [_i32]),
    "dg_plan_fp8_gemm_nt": (_st, [_i64, _i64, _i64, _i32, _i32, _p, _p, _p, _p]),
    "dg_plan_m_grouped_fp8_gemm_nt_contiguous": (_st, [_i64, _i64, _i64, _i32, _i32, _p, _p]),
    "dg_plan_m_grouped_fp8_gemm_nt_masked": (_st, [_i32, _i64, _i64, _i64, _i64, _i32, _p, _p, _p]),
    "dg_set_num_sms": (_st, [_i32]),
    "dg_get_num_sms": (_i32, []),
    "dg_set_pdl": (_st, [_i32]),
    "dg_get_pdl": (_i32, []),
    "dg_set_wait_timeout_ns": (_st, [C.c_uint64]),
    "dg_get_device_error": (_st, [_p, C.POINTER(C.c_uint64)]),
    "dg_debug_set_drop_load": (_st, [_i32]),
    "dg_debug_plant_check": (_st, [_i32]),
    "dg_status_string": (C.c_char_p, [_st]),
    "dg_version": (_i32, []),
}


def header_functions():
    """Names of the functions include/dg.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_[a-z0-9_]+)\s*\(", text)))


def lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "%s is not built; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def status_name(code: int) -> str:
    return STATUS_NAMES.get(int(code), "status %d" % int(code))
