"""GPU parity at the full workload sizes, in the launch configuration the
bench uses: dense prefill-like (M=4096, five (N, K) pairs, with and without
C), dense decode-like (M in {64, 128}), contiguous MoE (8 experts, N=4096,
K=7168) and masked MoE (16 experts x 256 rows, N=7168, K=2048).

Which rows are written is checked on every row (sentinel fill); values are
checked against the oracle on sampled rows (every row for the decode shapes),
always including the first and last rows and rows on tile boundaries."""
import numpy as np
import pytest
import torch

import oracle
import moe_grouped_gemm_fp8_gb300 as dg
from moe_grouped_gemm_fp8_gb300 import workloads
import _parity as P

pytestmark = pytest.mark.gpu


def _sample_rows(m, seed, extra=48):
    rng = np.random.default_rng(seed)
    # 128- and 256-row tile boundaries (both tile heights run at these sizes)
    fixed = [0, 1, 2, 127, 128, 129, 255, 256, 257, m // 2, m - 257, m - 256, m - 129, m - 128,
             m - 2, m - 1]
    rows = set(r for r in fixed if 0 <= r < m)
    rows.update(rng.choice(m, size=min(extra, m), replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def _no_device_error():
    st, word = dg.get_device_error()
    assert st == 0, "device error word 0x%x" % word


@pytest.mark.parametrize("idx", range(len(workloads.PREFILL)))
def test_prefill_dense(idx):
    cfg = workloads.PREFILL[idx]
    m, n, k = cfg["m"], cfg["n"], cfg["k"]
    w = workloads.dense(m, n, k, cfg["seed"], with_c=True)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    args = (P.dev_codes(qa), P.dev_packed_sf(sa, m, k, 1), P.dev_codes(qb), P.dev_packed_sf(sb, n, k, 128))
    rows = _sample_rows(m, cfg["seed"])
    d = dg.fp8_gemm_nt(*args)
    o = oracle.gemm_nt_rows(qa, sa, qb, sb, rows)
    P.assert_close(P.bf16_to_f64(d[torch.from_numpy(rows).cuda()]), o, "prefill %s" % (cfg,))
    cbits = P.bf16_bits(w.c)
    dc = dg.fp8_gemm_nt(*args, c=w.c.cuda())
    oc = oracle.gemm_nt_rows(qa, sa, qb, sb, rows, cbits)
    P.assert_close(P.bf16_to_f64(dc[torch.from_numpy(rows).cuda()]), oc, "prefill+C %s" % (cfg,))
    _no_device_error()


@pytest.mark.parametrize("idx", range(len(workloads.DECODE)))
def test_decode_dense(idx):
    cfg = workloads.DECODE[idx]
    m, n, k = cfg["m"], cfg["n"], cfg["k"]
    w = workloads.dense(m, n, k, cfg["seed"])
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    d = dg.fp8_gemm_nt(P.dev_codes(qa), P.dev_packed_sf(sa, m, k, 1), P.dev_codes(qb),
                       P.dev_packed_sf(sb, n, k, 128))
    P.assert_close(P.bf16_to_f64(d), oracle.gemm_nt(qa, sa, qb, sb), "decode %s" % (cfg,))
    _no_device_error()


def test_contiguous_moe_config():
    cfg = workloads.CONTIG
    w = workloads.contiguous(cfg["num_groups"], cfg["n"], cfg["k"], cfg["seed"])
    n, k = cfg["n"], cfg["k"]
    m_sum = w.a.shape[0]
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    d = P.sentinel_like((m_sum, n))
    dg.m_grouped_fp8_gemm_nt_contiguous(P.dev_codes(qa), P.dev_packed_sf(sa, m_sum, k, 1),
                                        P.dev_codes(qb), P.dev_packed_sf(sb, n, k, 128),
                                        w.m_indices.cuda(), d=d)
    _no_device_error()
    mi = w.m_indices.numpy()
    bits = P.bf16_bits(d)
    valid = mi >= 0
    assert (bits[~valid] == P.SENTINEL_BITS).all(), "padding rows were written"
    assert not (bits[valid] == P.SENTINEL_BITS).all(axis=1).any(), "a valid row was not written"
    # sampled rows: per expert the first, last and random valid rows
    rng = np.random.default_rng(cfg["seed"])
    rows = []
    for g in range(cfg["num_groups"]):
        idx = np.nonzero(mi == g)[0]
        if idx.size:
            rows += [idx[0], idx[-1]] + rng.choice(idx, size=min(6, idx.size), replace=False).tolist()
    rows = np.array(sorted(set(int(r) for r in rows)), dtype=np.int64)
    o, written = oracle.gemm_contiguous(qa, sa, qb, sb, mi, rows=rows)
    assert written.all()
    P.assert_close(P.bf16_to_f64(d[torch.from_numpy(rows).cuda()]), o, "contiguous config")


def test_masked_moe_config():
    cfg = workloads.MASKED
    G, cap, n, k = cfg["num_groups"], cfg["cap"], cfg["n"], cfg["k"]
    w = workloads.masked(G, cap, n, k, cfg["seed"])
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    d = P.sentinel_like((G, cap, n))
    mm = w.masked_m.numpy()
    dg.m_grouped_fp8_gemm_nt_masked(P.dev_codes(qa), P.dev_packed_sf(sa, cap, k, 1),
                                    P.dev_codes(qb), P.dev_packed_sf(sb, n, k, 128),
                                    w.masked_m.cuda(), expected_m=int(mm.mean()), d=d)
    _no_device_error()
    bits = P.bf16_bits(d)
    for g in range(G):
        assert (bits[g, mm[g]:] == P.SENTINEL_BITS).all(), "group %d: rows past masked_m written" % g
        if mm[g]:
            assert not (bits[g, :mm[g]] == P.SENTINEL_BITS).all(axis=1).any()
    rng = np.random.default_rng(cfg["seed"])
    flat = []
    for g in range(G):
        if mm[g]:
            rr = {0, mm[g] - 1} | set(rng.choice(mm[g], size=min(6, mm[g]), replace=False).tolist())
            flat += [g * cap + r for r in rr]
    rows = np.array(sorted(flat), dtype=np.int64)
    o, written = oracle.gemm_masked(qa, sa, qb, sb, mm, rows=rows)
    assert written.all()
    got = P.bf16_to_f64(d.view(G * cap, n)[torch.from_numpy(rows).cuda()])
    P.assert_close(got, o, "masked config")


@pytest.mark.parametrize("counts", ["uniform128", "seeded"])
def test_masked_moe_every_tile_width_full_grid(counts):
    """The masked MoE shape at every tile width on all SMs: many CTAs with
    several tiles each and 5- and 6-stage pipelines, the setting in which a
    waiter that skips phases of a stage barrier would read stale scales."""
    import os
    cfg = workloads.MASKED
    G, cap, n, k = cfg["num_groups"], cfg["cap"], cfg["n"], cfg["k"]
    w = workloads.masked(G, cap, n, k, cfg["seed"], masked_m=[128] * G if counts == "uniform128" else None)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    mm = w.masked_m.numpy()
    rows = np.array(sorted({g * cap + r for g in range(G) for r in range(0, mm[g], 29)} |
                           {g * cap + mm[g] - 1 for g in range(G) if mm[g]}), dtype=np.int64)
    o, _ = oracle.gemm_masked(qa, sa, qb, sb, mm, rows=rows)
    dev = (P.dev_codes(qa), P.dev_packed_sf(sa, cap, k, 1), P.dev_codes(qb), P.dev_packed_sf(sb, n, k, 128))
    old = {k: os.environ.get(k) for k in ("DG_BLOCK_N", "DG_CTA_PAIR")}
    try:
        for pair, bn in ((0, 128), (0, 192), (0, 224), (0, 256), (1, 192), (1, 224), (1, 256)):
            os.environ["DG_BLOCK_N"] = str(bn)
            os.environ["DG_CTA_PAIR"] = str(pair)
            d = P.sentinel_like((G, cap, n))
            dg.m_grouped_fp8_gemm_nt_masked(*dev, w.masked_m.cuda(), d=d)
            _no_device_error()
            bits = P.bf16_bits(d)
            for g in range(G):
                assert (bits[g, mm[g]:] == P.SENTINEL_BITS).all(), "pair=%d bn=%d g=%d" % (pair, bn, g)
            got = P.bf16_to_f64(d.view(G * cap, n)[torch.from_numpy(rows).cuda()])
            P.assert_close(got, o, "masked pair=%d bn=%d" % (pair, bn))
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
