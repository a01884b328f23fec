"""CPU-only checks of libdg.so: it loads, exports every function include/dg.h
declares, and rejects bad arguments on the host before touching the device."""
import ctypes as C

import pytest

from moe_grouped_gemm_fp8_gb300 import _lib

DG_OK, INVALID, ALIGN, TOO_LARGE = 0, 1, 2, 7


@pytest.fixture(scope="module")
def L():
    from moe_grouped_gemm_fp8_gb300 import build
    build.build()
    return _lib.lib()


def test_exports_every_declared_function(L):
    names = _lib.header_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(L, n), n
        assert n in _lib.SIGNATURES, "binding lacks a signature for %s" % n


def test_exports_nothing_the_header_does_not_declare(L):
    """Every dg_* symbol libdg.so exports is declared in include/dg.h (the
    library's own exported names, read with nm)."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = sorted({line.split()[-1] for line in out.splitlines()
                       if line.split() and line.split()[-1].startswith("dg_")})
    assert exported == _lib.header_functions()


def test_pure_host_utilities(L):
    assert L.dg_get_tma_aligned_size(4097, 4) == 4100
    assert L.dg_get_tma_aligned_size(4096, 4) == 4096
    assert L.dg_get_tma_aligned_size(1, 1) == 16
    assert L.dg_get_tma_aligned_size(5, 2) == 8
    assert L.dg_get_tma_aligned_size(5, 3) == -1
    assert L.dg_get_mk_alignment_for_contiguous_layout() == 128
    assert L.dg_version() >= 100
    for s in range(9):
        assert L.dg_status_string(s)
    assert L.dg_set_num_sms(-1) == INVALID
    assert L.dg_set_wait_timeout_ns(0) == INVALID


P = C.c_void_p(0x1000)  # a 16-byte aligned fake pointer: never dereferenced on these paths


def gemm(L, **kw):
    a = dict(a=P, sfa=P, b=P, sfb=P, c=None, d=P, m=128, n=256, k=512, lda=512, ldb=512,
             ldc=0, ldd=256, stream=None)
    a.update(kw)
    return L.dg_fp8_gemm_nt(a["a"], a["sfa"], a["b"], a["sfb"], a["c"], a["d"], a["m"], a["n"],
                            a["k"], a["lda"], a["ldb"], a["ldc"], a["ldd"], a["stream"])


def test_dense_host_checks(L):
    assert gemm(L, k=100, lda=112, ldb=112) == ALIGN          # K % 128
    assert gemm(L, n=260, ldd=260) == ALIGN                   # N % 8
    assert gemm(L, k=0) == INVALID
    assert gemm(L, m=-1) == INVALID
    assert gemm(L, m=0) == DG_OK                              # empty problem: no-op
    assert gemm(L, n=0, ldd=0) == DG_OK
    assert gemm(L, a=None) == INVALID
    assert gemm(L, d=None) == INVALID
    assert gemm(L, lda=256) == INVALID                        # lda < K
    assert gemm(L, lda=520) == ALIGN                          # lda % 16
    assert gemm(L, a=C.c_void_p(0x1008)) == ALIGN             # 16-byte pointer alignment
    assert gemm(L, c=P, ldc=100) == INVALID                   # ldc < N
    assert gemm(L, m=1 << 31) == TOO_LARGE


def test_workspace_entry_points_host_checks(L):
    """dg_fp8_gemm_nt_ws: the same checks, plus a 16-byte aligned workspace;
    the size and plan queries are pure host arithmetic."""
    def gemm_ws(ws, nbytes, **kw):
        a = dict(a=P, sfa=P, b=P, sfb=P, c=None, d=P, m=128, n=256, k=512, lda=512, ldb=512,
                 ldc=0, ldd=256)
        a.update(kw)
        return L.dg_fp8_gemm_nt_ws(a["a"], a["sfa"], a["b"], a["sfb"], a["c"], a["d"], a["m"], a["n"],
                                   a["k"], a["lda"], a["ldb"], a["ldc"], a["ldd"], ws, nbytes, None)
    assert gemm_ws(C.c_void_p(0x1008), 1 << 20) == ALIGN     # unaligned workspace
    assert gemm_ws(P, 1 << 20, k=100, lda=112, ldb=112) == ALIGN
    assert gemm_ws(P, 1 << 20, m=0) == DG_OK
    out = C.c_uint64(7)
    assert L.dg_fp8_gemm_nt_workspace_size(128, 256, 100, 0, 152, C.byref(out)) == ALIGN
    assert L.dg_fp8_gemm_nt_workspace_size(128, 256, 512, 0, 0, C.byref(out)) == INVALID
    assert L.dg_fp8_gemm_nt_workspace_size(128, 256, 512, 0, 152, None) == INVALID
    assert L.dg_fp8_gemm_nt_workspace_size(0, 256, 512, 0, 152, C.byref(out)) == DG_OK and out.value == 0


def test_grouped_host_checks(L):
    cont = L.dg_m_grouped_fp8_gemm_nt_contiguous
    assert cont(P, P, P, P, P, P, 130, 256, 512, 4, None) == ALIGN      # m_sum % 128
    assert cont(P, P, P, P, P, None, 128, 256, 512, 4, None) == INVALID  # m_indices
    assert cont(P, P, P, P, P, P, 0, 256, 512, 4, None) == DG_OK
    assert cont(P, P, P, P, P, P, 128, 256, 512, 0, None) == DG_OK
    assert cont(P, P, P, P, P, P, 128, 256, 500, 4, None) == ALIGN
    masked = L.dg_m_grouped_fp8_gemm_nt_masked
    assert masked(P, P, P, P, P, P, 513, 256, 256, 512, 0, None) == TOO_LARGE
    assert masked(P, P, P, P, P, None, 4, 256, 256, 512, 0, None) == INVALID
    assert masked(P, P, P, P, P, P, 4, 0, 256, 512, 0, None) == DG_OK
    assert masked(P, P, P, P, P, P, 4, 256, 250, 512, 0, None) == ALIGN
    assert masked(P, P, P, P, P, P, 4, 256, 256, 512, -1, None) == INVALID


def test_quantize_and_transform_host_checks(L):
    q = L.dg_quantize_fp8
    assert q(P, P, P, 1, 10, 130, 1, 1, None) == ALIGN
    assert q(P, P, P, 1, 10, 128, 2, 1, None) == INVALID
    assert q(P, P, P, 1, 10, 128, 1, 7, None) == INVALID
    assert q(P, P, P, 0, 10, 128, 1, 1, None) == DG_OK
    assert q(None, P, P, 1, 10, 128, 1, 1, None) == INVALID
    t = L.dg_transform_sf
    assert t(P, P, 1, 10, 128, 3, None) == INVALID
    assert t(P, None, 1, 10, 128, 1, None) == INVALID
    assert t(P, C.c_void_p(0x1004), 1, 10, 128, 1, None) == ALIGN
    assert t(P, P, 0, 10, 128, 1, None) == DG_OK


def test_k_grouped_host_checks(L):
    kg = L.dg_k_grouped_fp8_gemm_tn_contiguous
    # a, sfa, b, sfb, c, d, ks, m, n, sum_k, groups, stream
    assert kg(P, P, P, P, None, P, P, 130, 256, 512, 4, None) == ALIGN     # m % 16
    assert kg(P, P, P, P, None, P, P, 128, 250, 512, 4, None) == ALIGN     # n % 16
    assert kg(P, P, P, P, None, P, P, 128, 256, 500, 4, None) == ALIGN     # sum_k % 128
    assert kg(P, P, P, P, None, P, P, 0, 256, 512, 4, None) == DG_OK       # empty output
    assert kg(P, P, P, P, None, P, P, 128, 256, 512, 0, None) == DG_OK
    assert kg(P, P, P, P, None, P, P, 128, 256, 512, 513, None) == TOO_LARGE
    assert kg(P, P, P, P, None, None, P, 128, 256, 512, 4, None) == INVALID  # d
    assert kg(P, P, P, P, None, P, None, 128, 256, 512, 4, None) == INVALID  # ks
    assert kg(None, P, P, P, None, P, P, 128, 256, 512, 4, None) == INVALID  # a with sum_k > 0
    assert kg(P, P, P, P, None, C.c_void_p(0x1008), P, 128, 256, 512, 4, None) == ALIGN
    assert kg(P, P, P, P, None, P, P, -16, 256, 512, 4, None) == INVALID


def test_quantize_cols_host_checks(L):
    qc = L.dg_quantize_fp8_cols
    assert qc(P, P, P, 100, 16, 1, None) == ALIGN      # rows % 128
    assert qc(P, P, P, 128, 18, 1, None) == ALIGN      # cols % 4
    assert qc(P, P, P, 128, 16, 7, None) == INVALID    # format
    assert qc(P, P, P, 0, 16, 1, None) == DG_OK
    assert qc(None, P, P, 128, 16, 1, None) == INVALID
    assert qc(P, C.c_void_p(0x1004), P, 128, 16, 1, None) == ALIGN


def test_layout_host_checks(L):
    for name, a_t, b_t in (("nn", False, False), ("tn", True, False), ("tt", True, True)):
        fn = getattr(L, "dg_fp8_gemm_" + name)
        # m=128, n=256, k=512: lda must cover M when A is stored [K, M], else K
        lda_ok = 128 if a_t else 512
        ldb_ok = 512 if b_t else 256
        assert fn(P, P, P, P, None, P, 128, 256, 512, lda_ok - 16, ldb_ok, 0, 256, None) == INVALID
        assert fn(P, P, P, P, None, P, 128, 256, 512, lda_ok, ldb_ok - 16, 0, 256, None) == INVALID
        assert fn(P, P, P, P, None, P, 128, 256, 500, lda_ok, ldb_ok + 16, 0, 256, None) == ALIGN
        assert fn(P, P, P, P, None, P, 0, 256, 512, lda_ok, ldb_ok, 0, 256, None) == DG_OK
        assert fn(None, P, P, P, None, P, 128, 256, 512, lda_ok, ldb_ok, 0, 256, None) == INVALID


def test_pdl_switch(L):
    assert L.dg_get_pdl() == 0
    assert L.dg_set_pdl(2) == INVALID
    assert L.dg_set_pdl(1) == DG_OK and L.dg_get_pdl() == 1
    assert L.dg_set_pdl(0) == DG_OK and L.dg_get_pdl() == 0


def test_fp32_scale_gemm_host_checks(L):
    fn = L.dg_fp8_gemm_nt_fp32_sf
    assert fn(P, P, P, P, None, P, 128, 256, 100, 112, 112, 0, 256, None) == ALIGN   # K % 128
    assert fn(P, P, P, P, None, P, 0, 256, 512, 512, 512, 0, 256, None) == DG_OK
    assert fn(P, None, P, P, None, P, 128, 256, 512, 512, 512, 0, 256, None) == INVALID
    assert fn(P, C.c_void_p(0x1002), P, P, None, P, 128, 256, 512, 512, 512, 0, 256, None) == ALIGN
    assert fn(P, P, P, P, None, P, 128, 256, 512, 256, 512, 0, 256, None) == INVALID  # lda < K


def test_tensors_must_be_on_the_current_device(monkeypatch):
    """The binding refuses tensors of another CUDA device than the current one
    (the library launches on the current device)."""
    import torch
    from moe_grouped_gemm_fp8_gb300 import api

    class On:
        def __init__(self, i):
            self.device = torch.device("cuda", i)

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 1)
    api._on_current_device(None, On(1), None, On(1))           # all on cuda:1: accepted
    with pytest.raises(ValueError, match="current CUDA device is cuda:1"):
        api._on_current_device(None, On(1), On(0))


def test_debug_library_exports_the_same_abi(L):
    """libdg_debug.so (the same sources with device-side checks) exports the
    same functions; its check hook is accepted, the release library's
    refuses to be switched on (it has no checks to plant into)."""
    import shutil
    import subprocess
    from moe_grouped_gemm_fp8_gb300 import build
    path = build.build(debug=True)
    D = C.CDLL(path)
    for n in _lib.header_functions():
        assert hasattr(D, n), n
    nm = shutil.which("nm")
    if nm is not None:
        out = subprocess.run([nm, "-D", "--defined-only", path], capture_output=True, text=True,
                             check=True).stdout
        exported = sorted({line.split()[-1] for line in out.splitlines()
                           if line.split() and line.split()[-1].startswith("dg_")})
        assert exported == _lib.header_functions()
    D.dg_debug_plant_check.argtypes = [C.c_int32]
    assert D.dg_debug_plant_check(1) == DG_OK and D.dg_debug_plant_check(0) == DG_OK
    assert L.dg_debug_plant_check(1) == INVALID and L.dg_debug_plant_check(0) == DG_OK


def test_mk_alignment_setter(L):
    """set_mk_alignment_for_contiguous_layout: positive multiples of 128 up to
    4096; anything else is refused and leaves the value unchanged."""
    assert L.dg_get_mk_alignment_for_contiguous_layout() == 128
    try:
        assert L.dg_set_mk_alignment_for_contiguous_layout(256) == DG_OK
        assert L.dg_get_mk_alignment_for_contiguous_layout() == 256
        for bad in (0, -128, 64, 100, 192, 4096 + 128):
            assert L.dg_set_mk_alignment_for_contiguous_layout(bad) == INVALID, bad
            assert L.dg_get_mk_alignment_for_contiguous_layout() == 256
        assert L.dg_set_mk_alignment_for_contiguous_layout(4096) == DG_OK
    finally:
        assert L.dg_set_mk_alignment_for_contiguous_layout(128) == DG_OK
    assert L.dg_get_mk_alignment_for_contiguous_layout() == 128


def test_floor_library_is_separate_and_checks_its_arguments():
    """libdg_floor.so (the benchmark's streaming-read floor) exports its one
    function and nothing of the GEMM library; it refuses a null or unaligned
    buffer and an empty grid before launching anything."""
    import shutil
    import subprocess
    from moe_grouped_gemm_fp8_gb300 import build
    path = build.build_floor()
    F = C.CDLL(path)
    F.dg_hbm_read_floor.argtypes = [C.c_void_p, C.c_size_t, C.c_void_p, C.c_int, C.c_void_p]
    F.dg_hbm_read_floor.restype = C.c_int
    nm = shutil.which("nm")
    if nm is not None:
        out = subprocess.run([nm, "-D", "--defined-only", path], capture_output=True, text=True,
                             check=True).stdout
        exported = sorted({line.split()[-1] for line in out.splitlines()
                           if line.split() and line.split()[-1].startswith("dg_")})
        assert exported == ["dg_hbm_read_floor"]
    cuda_error_invalid_value = 1
    assert F.dg_hbm_read_floor(None, 1024, None, 4, None) == cuda_error_invalid_value
    assert F.dg_hbm_read_floor(0x1008, 1024, None, 4, None) == cuda_error_invalid_value
    assert F.dg_hbm_read_floor(0x1000, 1024, None, 0, None) == cuda_error_invalid_value


def test_header_lists_exactly_the_environment_variables_the_library_reads():
    """dg.h's list of DG_* environment variables matches the names host.cu
    reads, so the documentation cannot drift from the code."""
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    header = open(os.path.join(root, "include", "dg.h")).read()
    block = header[header.index("Environment variables read by the library"):]
    block = block[:block.index("*/")]
    documented = set(re.findall(r"\b(DG_[A-Z0-9_]+)=", block))
    host = open(os.path.join(root, "moe_grouped_gemm_fp8_gb300", "csrc", "host.cu")).read()
    read = set(re.findall(r'env_(?:int|flag)\("(DG_[A-Z0-9_]+)"', host))
    assert read and documented == read, (sorted(documented ^ read))
