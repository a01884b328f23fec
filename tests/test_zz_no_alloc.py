"""dg_fp8_gemm_nt_static_ws, the GEMM for callers that cannot allocate device
memory (a runtime that reserves everything at start-up, a plugin whose host
gives it no scratch buffer, code where cudaMalloc would synchronise or is not
allowed): its stream-K workspace is an array inside the library.

Called through the C ABI and compared with dg_fp8_gemm_nt, the entry point
that needs no scratch, within the tolerance of the other parity tests, on two
calls in a row (the second finds the first call's contents in the array).
Kept in a file of its own so that it runs after every other test; it also
passes alone in a fresh process."""
import ctypes as C
import os

import pytest
import torch

import moe_grouped_gemm_fp8_gb300 as dg
from moe_grouped_gemm_fp8_gb300 import _lib, workloads
import _parity as P

pytestmark = pytest.mark.gpu

DG_ERR_TOO_LARGE = 7


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _call(fn, qa, sfa, qb, sfb, d):
    m, k = qa.shape
    n = qb.shape[0]
    return int(fn(_ptr(qa), _ptr(sfa), _ptr(qb), _ptr(sfb), None, _ptr(d), m, n, k, k, k, 0, n,
                  C.c_void_p(torch.cuda.current_stream().cuda_stream)))


def test_static_workspace_matches_the_entry_point_without_scratch():
    L = _lib.lib()
    m, n, k = 4096, 2112, 7168  # 176 tiles of 256 x 192: one wave and 24 tiles, split by stream-K
    w = workloads.dense(m, n, k, seed=1)
    qa, sfa = dg.quantize_fp8(w.a.cuda(), 1)
    qb, sfb = dg.quantize_fp8(w.b.cuda(), 128)
    keep = {v: os.environ.get(v) for v in ("DG_STREAM_K", "DG_BLOCK_N", "DG_BLOCK_M")}
    os.environ["DG_STREAM_K"] = "1"
    os.environ["DG_BLOCK_N"] = "192"
    os.environ.pop("DG_BLOCK_M", None)
    try:
        sms = dg.get_num_sms()
        need = dg.fp8_gemm_nt_workspace_size(m, n, k, False, sms)
        assert 0 < need <= 32 << 20, need  # stream-K, within the library's array
        ref = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
        assert _call(L.dg_fp8_gemm_nt, qa, sfa, qb, sfb, ref) == 0
        for _ in range(2):
            d = P.sentinel_like((m, n))
            assert _call(L.dg_fp8_gemm_nt_static_ws, qa, sfa, qb, sfb, d) == 0
            assert dg.get_device_error()[0] == 0
            P.assert_close(P.bf16_to_f64(d), P.bf16_to_f64(ref), "static workspace vs no scratch")
        if sms > 145:  # 224-column tiles need more than the array holds here: refused up front
            os.environ["DG_BLOCK_N"] = "224"
            d = P.sentinel_like((m, n))
            assert _call(L.dg_fp8_gemm_nt_static_ws, qa, sfa, qb, sfb, d) == DG_ERR_TOO_LARGE
            torch.cuda.synchronize()
            assert bool((d.view(torch.int16) == P.SENTINEL_BITS).all())  # nothing was enqueued
    finally:
        for v, old in keep.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
