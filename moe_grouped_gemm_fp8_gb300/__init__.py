"""FP8 GEMM with fine-grained scaling for NVIDIA GB300 (sm_103a).

D = C + A @ B.T with E4M3 operands, 1x128 / 128x128 power-of-two scales,
FP32 accumulation and BF16 output, in the dense NT form and the two
M-grouped MoE layouts (contiguous, masked); and the K-grouped layout of MoE
weight gradients (FP32 output).  The kernels live in libdg.so
(C ABI: include/dg.h); this package is a thin torch binding over it.
"""
from .api import (  # noqa: F401
    DGError,
    debug_plant_check,
    debug_set_drop_load,
    fp8_gemm_nn,
    fp8_gemm_nt,
    fp8_gemm_nt_fp32_sf,
    fp8_gemm_nt_workspace_size,
    fp8_gemm_tn,
    fp8_gemm_tt,
    get_device_error,
    get_mk_alignment_for_contiguous_layout,
    set_mk_alignment_for_contiguous_layout,
    get_num_sms,
    get_pdl,
    get_tma_aligned_size,
    k_grouped_fp8_gemm_tn_contiguous,
    m_grouped_fp8_gemm_nt_contiguous,
    m_grouped_fp8_gemm_nt_masked,
    plan_fp8_gemm_nt,
    plan_fp8_gemm_nt_ws,
    plan_m_grouped_fp8_gemm_nt_contiguous,
    plan_m_grouped_fp8_gemm_nt_masked,
    quantize_fp8,
    quantize_fp8_cols,
    set_num_sms,
    set_pdl,
    set_wait_timeout_ns,
    sf_packed_shape,
    transform_sf_into_required_layout,
)

__version__ = "0.1.0"
