"""The masked GEMM under CUDA-graph capture: the per-expert counts live on
the device only, so one captured graph serves any counts written into the
same tensor before a replay ("GEMM denso e grouped": masked grouped GEMM for
decoding with CUDA graphs, where the CPU does not know the token counts)."""
import numpy as np
import pytest
import torch

import oracle
import moe_grouped_gemm_fp8_gb300 as dg
from moe_grouped_gemm_fp8_gb300 import workloads
import _parity as P

pytestmark = pytest.mark.gpu


def test_masked_gemm_replays_with_new_counts():
    G, cap, N, K = 6, 256, 512, 512
    w = workloads.masked(G, cap, N, K, seed=61, masked_m=[0] * G)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    dev = (P.dev_codes(qa), P.dev_packed_sf(sa, cap, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    mm_dev = torch.zeros(G, dtype=torch.int32, device="cuda")
    d = P.sentinel_like((G, cap, N))
    # first call outside the capture: per-device set-up happens here
    dg.m_grouped_fp8_gemm_nt_masked(*dev, mm_dev, expected_m=128, d=d)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dg.m_grouped_fp8_gemm_nt_masked(*dev, mm_dev, expected_m=128, d=d)
    for counts in ([256, 0, 17, 128, 129, 200], [1, 255, 0, 64, 256, 3]):
        d.copy_(P.sentinel_like((G, cap, N)))
        mm_dev.copy_(torch.tensor(counts, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        mm = np.array(counts, np.int32)
        o, written = oracle.gemm_masked(qa, sa, qb, sb, mm)
        bits = P.bf16_bits(d)
        wr = written.astype(bool)
        assert (bits[~wr] == P.SENTINEL_BITS).all(), counts
        P.assert_close(P.bf16_to_f64(d)[wr], o[wr], "graph replay %s" % counts)
    st, word = dg.get_device_error()
    assert st == 0, hex(word)


def _replay_matches_eager(fn, outs):
    """fn() writes into the tensors `outs`; capture it once, zero the outputs,
    replay, and require the results bit-identical to an eager call."""
    fn()
    torch.cuda.synchronize()
    ref = [o.clone() for o in outs]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    for _ in range(2):
        for o in outs:
            o.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for o, r in zip(outs, ref):
            assert torch.equal(o.view(torch.uint8), r.view(torch.uint8))
    st, word = dg.get_device_error()
    assert st == 0, hex(word)


@pytest.mark.parametrize("split_k", ["1", "2"])
def test_dense_quantise_and_gemm_capture(split_k, monkeypatch):
    """Quantise + dense GEMM (single CTA, and the split-K cluster path) in one graph."""
    monkeypatch.setenv("DG_SPLIT_K", split_k)
    w = workloads.dense(64 if split_k == "2" else 512, 1024, 2048, seed=67)
    a = w.a.cuda()
    qb, sfb = dg.quantize_fp8(w.b.cuda(), 128)
    qa = torch.empty(a.shape, dtype=torch.float8_e4m3fn, device="cuda")
    sfa = torch.empty(dg.sf_packed_shape(a.shape[0], a.shape[1]), dtype=torch.int32, device="cuda")
    d = torch.empty(a.shape[0], 1024, dtype=torch.bfloat16, device="cuda")

    def fn():
        dg.quantize_fp8(a, 1, out=(qa, sfa))
        dg.fp8_gemm_nt(qa, sfa, qb, sfb, d=d)
    _replay_matches_eager(fn, [d])


def test_contiguous_and_k_grouped_capture():
    cw = workloads.contiguous(3, 256, 512, seed=71, counts=[100, 0, 300])
    qa, sfa = dg.quantize_fp8(cw.a.cuda(), 1)
    qb, sfb = dg.quantize_fp8(cw.b.cuda(), 128)
    mi = cw.m_indices.cuda()
    d = torch.zeros(cw.a.shape[0], 256, dtype=torch.bfloat16, device="cuda")
    kw = workloads.k_grouped(3, 128, 256, seed=73, counts=[200, 0, 64])
    ka, ksa = dg.quantize_fp8_cols(kw.a.cuda())
    kb, ksb = dg.quantize_fp8_cols(kw.b.cuda())
    ks = kw.ks.cuda()
    dk = torch.zeros(3, 128, 256, dtype=torch.float32, device="cuda")

    def fn():
        dg.m_grouped_fp8_gemm_nt_contiguous(qa, sfa, qb, sfb, mi, d=d)
        dg.k_grouped_fp8_gemm_tn_contiguous(ka, ksa, kb, ksb, ks, d=dk)
    _replay_matches_eager(fn, [d, dk])


@pytest.mark.parametrize("bn", ["192", "224"])
def test_256_row_tiles_capture(bn, monkeypatch):
    """Dense (with C) and contiguous GEMMs on 256-row tiles, captured in one
    graph: the contiguous pair table is rebuilt from m_indices at every replay."""
    monkeypatch.setenv("DG_BLOCK_M", "256")
    monkeypatch.setenv("DG_BLOCK_N", bn)
    w = workloads.dense(600, 520, 1024, seed=69, with_c=True)
    qa, sfa = dg.quantize_fp8(w.a.cuda(), 1)
    qb, sfb = dg.quantize_fp8(w.b.cuda(), 128)
    c = w.c.cuda()
    d = torch.empty(600, 520, dtype=torch.bfloat16, device="cuda")
    cw = workloads.contiguous(4, 264, 512, seed=72, counts=[300, 0, 129, 520])
    cqa, csfa = dg.quantize_fp8(cw.a.cuda(), 1)
    cqb, csfb = dg.quantize_fp8(cw.b.cuda(), 128)
    mi = cw.m_indices.cuda()
    dc = torch.zeros(cw.a.shape[0], 264, dtype=torch.bfloat16, device="cuda")

    def fn():
        dg.fp8_gemm_nt(qa, sfa, qb, sfb, d=d, c=c)
        dg.m_grouped_fp8_gemm_nt_contiguous(cqa, csfa, cqb, csfb, mi, d=dc)
    _replay_matches_eager(fn, [d, dc])
