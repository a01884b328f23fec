"""GPU parity at the full workload sizes, in the launch configuration the
bench uses: dense small (M=128, N=256, K=512), dense prefill-like (M=4096,
five (N, K) pairs, with and without C), dense decode-like (M in {64, 128}),
contiguous MoE (8 experts, N=4096, K=7168) and masked MoE (16 experts x 256
rows, N=7168, K=2048).

Every written element is compared with the CPU oracle (FP64) on the same
seeded inputs, per tensor: sum((d - o)^2) / sum(o^2) <= 1e-5 and
max|d - o| <= 2e-2 * max|o|.  Which rows are written is checked bit for bit
on every row (sentinel fill).  The oracle runs the full products on the
host's cores (about 2 TFLOP for the prefill set with and without C, 2.3 for
the contiguous workload)."""
import os

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_gemm_fp8_gb300 as dg
from moe_grouped_gemm_fp8_gb300 import workloads
import _parity as P

pytestmark = pytest.mark.gpu


def _no_device_error():
    st, word = dg.get_device_error()
    assert st == 0, "device error word 0x%x" % word


def _dense_case(cfg, with_c):
    m, n, k = cfg["m"], cfg["n"], cfg["k"]
    w = workloads.dense(m, n, k, cfg["seed"], with_c=with_c)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    dev = (P.dev_codes(qa), P.dev_packed_sf(sa, m, k, 1), P.dev_codes(qb), P.dev_packed_sf(sb, n, k, 128))
    return w, (qa, sa, qb, sb), dev


def test_small_config():
    cfg = workloads.SMALL
    _, (qa, sa, qb, sb), dev = _dense_case(cfg, False)
    d = dg.fp8_gemm_nt(*dev, d=P.sentinel_like((cfg["m"], cfg["n"])))
    _no_device_error()
    P.assert_close(P.bf16_to_f64(d), oracle.gemm_nt(qa, sa, qb, sb), "small m=128 n=256 k=512", record=True)


@pytest.mark.parametrize("idx", range(len(workloads.PREFILL)))
def test_prefill_dense(idx):
    cfg = workloads.PREFILL[idx]
    m, n, k = cfg["m"], cfg["n"], cfg["k"]
    w, (qa, sa, qb, sb), dev = _dense_case(cfg, True)
    tag = "prefill m=%d n=%d k=%d" % (m, n, k)
    d = dg.fp8_gemm_nt(*dev, d=P.sentinel_like((m, n)))
    _no_device_error()
    P.assert_close(P.bf16_to_f64(d), oracle.gemm_nt(qa, sa, qb, sb), tag, record=True)
    del d
    dc = dg.fp8_gemm_nt(*dev, c=w.c.cuda(), d=P.sentinel_like((m, n)))
    _no_device_error()
    P.assert_close(P.bf16_to_f64(dc), oracle.gemm_nt(qa, sa, qb, sb, P.bf16_bits(w.c)), tag + " +C",
                   record=True)


@pytest.mark.parametrize("idx", range(len(workloads.DECODE)))
def test_decode_dense(idx):
    cfg = workloads.DECODE[idx]
    m, n, k = cfg["m"], cfg["n"], cfg["k"]
    _, (qa, sa, qb, sb), dev = _dense_case(cfg, False)
    d = dg.fp8_gemm_nt(*dev, d=P.sentinel_like((m, n)))
    _no_device_error()
    P.assert_close(P.bf16_to_f64(d), oracle.gemm_nt(qa, sa, qb, sb), "decode m=%d n=%d k=%d" % (m, n, k),
                   record=True)


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
    o, written = oracle.gemm_contiguous(qa, sa, qb, sb, mi)
    assert np.array_equal(written.astype(bool), valid)
    got = P.bf16_to_f64(d)[valid]
    del d, bits
    P.assert_close(got, o[valid], "contiguous G=8 rows=%d n=%d k=%d" % (int(valid.sum()), n, k), record=True)


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
    o, written = oracle.gemm_masked(qa, sa, qb, sb, mm)
    wr = written.astype(bool)
    assert np.array_equal(wr, np.arange(cap)[None, :] < mm[:, None])
    assert (bits[~wr] == P.SENTINEL_BITS).all(), "rows past masked_m were written"
    P.assert_close(P.bf16_to_f64(d)[wr], o[wr], "masked G=16 cap=256 rows=%d n=%d k=%d" % (int(mm.sum()), n, k),
                   record=True)


@pytest.mark.parametrize("counts", ["uniform128", "seeded"])
def test_masked_moe_every_tile_width_full_grid(counts):
    """The masked MoE shape at every tile width on all SMs: many CTAs with
    several tiles each and 5- and 6-stage pipelines, the setting in which a
    waiter that skips phases of a stage barrier would read stale scales.
    Every written element is compared."""
    cfg = workloads.MASKED
    G, cap, n, k = cfg["num_groups"], cfg["cap"], cfg["n"], cfg["k"]
    w = workloads.masked(G, cap, n, k, cfg["seed"], masked_m=[128] * G if counts == "uniform128" else None)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    mm = w.masked_m.numpy()
    o, written = oracle.gemm_masked(qa, sa, qb, sb, mm)
    wr = written.astype(bool)
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
            assert (bits[~wr] == P.SENTINEL_BITS).all(), "pair=%d bn=%d: rows past masked_m written" % (pair, bn)
            P.assert_close(P.bf16_to_f64(d)[wr], o[wr], "masked pair=%d bn=%d" % (pair, bn))
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
