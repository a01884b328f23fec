"""Programmatic dependent launch: with PDL on, a kernel may start while the
previous one finishes, so every read of another kernel's output must come
after its grid-dependency wait.  These chains make each kernel consume the
previous kernel's output immediately (quantise -> GEMM -> GEMM accumulating
into the first GEMM's result), eagerly and inside a CUDA graph, and require
results bit-identical to the same chain without PDL."""
import pytest
import torch

import moe_grouped_gemm_fp8_gb300 as dg
from moe_grouped_gemm_fp8_gb300 import workloads

pytestmark = pytest.mark.gpu


def _no_device_error():
    st, word = dg.get_device_error()
    assert st == 0, "device error word 0x%x" % word


def _chain(a, b, b2, out):
    qa, sfa, qb, sfb, qb2, sfb2, d1, d2, qm, sfm = out
    dg.quantize_fp8(a, 1, out=(qa, sfa))
    dg.fp8_gemm_nt(qa, sfa, qb, sfb, d=d1)
    # d2 = d1 + A @ B2^T: reads d1 as C right after the kernel that wrote it
    dg.fp8_gemm_nt(qa, sfa, qb2, sfb2, d=d2, c=d1)
    # masked form reading the freshly quantised A
    dg.m_grouped_fp8_gemm_nt_masked(qm, sfm, qb.unsqueeze(0), sfb.unsqueeze(0),
                                    torch.full((1,), 77, dtype=torch.int32, device="cuda"), 77,
                                    d=d1.unsqueeze(0)[:, :128])


def _buffers(m, n, k, seed):
    w = workloads.dense(m, n, k, seed)
    w2 = workloads.dense(m, n, k, seed + 1)
    a = w.a.cuda()
    qb, sfb = dg.quantize_fp8(w.b.cuda(), 128)
    qb2, sfb2 = dg.quantize_fp8(w2.b.cuda(), 128)
    qa = torch.empty(m, k, dtype=torch.float8_e4m3fn, device="cuda")
    sfa = torch.empty(dg.sf_packed_shape(m, k), dtype=torch.int32, device="cuda")
    d1 = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    d2 = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    qm, sfm = dg.quantize_fp8(w.a[:128].unsqueeze(0).contiguous().cuda(), 1)
    return a, qb, sfb, qb2, sfb2, (qa, sfa, qb, sfb, qb2, sfb2, d1, d2, qm, sfm)


@pytest.mark.parametrize("graph", [False, True])
def test_pdl_chain_matches_serial(graph):
    m, n, k = 512, 2048, 2048
    a, qb, sfb, qb2, sfb2, out = _buffers(m, n, k, 101)
    dg.set_pdl(False)
    _chain(a, qb, qb2, out)
    torch.cuda.synchronize()
    ref = [t.clone() for t in out[6:8]]
    try:
        dg.set_pdl(True)
        for _ in range(3):
            for t in out[6:8]:
                t.zero_()
            out[0].view(torch.uint8).zero_()
            if graph:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    _chain(a, qb, qb2, out)
                g.replay()
            else:
                _chain(a, qb, qb2, out)
            torch.cuda.synchronize()
            _no_device_error()
            for got, want in zip(out[6:8], ref):
                assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    finally:
        dg.set_pdl(False)
