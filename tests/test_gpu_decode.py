"""The decode kernel (dense NT with at most 128 rows of A): B's rows fill the
MMA's 128 lanes, A's rows are its N side (32, 64 or 128 tokens), and each
128-column strip's K blocks are split over a cluster of 1, 2, 4 or 8 CTAs
whose FP32 partials are added in rank order through distributed shared
memory.

Checked against the oracle at every cluster size and token width, on ragged
M and N (the last strip partly past N), K ranges that start inside a scale
word, with and without C (C aliasing D too), bit for bit where the FP32 sums
are exact, and with the columns of D past N (ldd > N) left untouched."""
import os
from contextlib import contextmanager

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_gemm_fp8_gb300 as dg
from moe_grouped_gemm_fp8_gb300 import workloads
import _parity as P

pytestmark = pytest.mark.gpu

_INT_CODE = {0: 0x00, 1: 0x38, 2: 0x40, 3: 0x44, 4: 0x48, -1: 0xB8, -2: 0xC0, -3: 0xC4, -4: 0xC8}


@contextmanager
def split(s):
    keys = ("DG_SPLIT_K", "DG_DECODE", "DG_BLOCK_M", "DG_BLOCK_N")
    old = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ.pop(k, None)
    if s:
        os.environ["DG_SPLIT_K"] = str(s)
    try:
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _no_device_error():
    st, word = dg.get_device_error()
    assert st == 0, "device error word 0x%x" % word


def _args(qa, sa, qb, sb, m, n, k):
    return (P.dev_codes(qa), P.dev_packed_sf(sa, m, k, 1), P.dev_codes(qb), P.dev_packed_sf(sb, n, k, 128))


# (M, N, K): token widths 32 / 64 / 128, ragged strips, K of 1 to 40 blocks
SHAPES = [(1, 128, 128), (7, 200, 1024), (32, 256, 512), (33, 1000, 2048), (64, 2112, 1536),
          (100, 384, 4096), (128, 640, 5120), (128, 136, 1152)]


@pytest.mark.parametrize("s", [1, 2, 4, 8])
@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("with_c", [False, True])
def test_decode_matches_oracle(s, M, N, K, with_c):
    kb = K // 128
    if s > kb:
        pytest.skip("more CTAs than K blocks")
    w = workloads.dense(M, N, K, seed=M * 7 + N + K + s, with_c=with_c)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    with split(s):
        p = dg.plan_fp8_gemm_nt_ws(M, N, K, with_c)
        if p["split_k"] != s or not p["swap_ab"]:
            pytest.skip("cluster size %d does not apply (K ranges over 8 scale words)" % s)
        assert p["block_n"] == 128 and p["block_m"] == (32 if M <= 32 else 64 if M <= 64 else 128)
        ldd = N + 24
        d = P.sentinel_like((M, ldd))
        dg.fp8_gemm_nt(*_args(qa, sa, qb, sb, M, N, K), c=w.c.cuda() if with_c else None, d=d[:, :N])
        _no_device_error()
    bits = P.bf16_bits(d)
    assert (bits[:, N:] == P.SENTINEL_BITS).all(), "columns past N were written"
    o = oracle.gemm_nt(qa, sa, qb, sb, P.bf16_bits(w.c) if with_c else None)
    P.assert_close(P.bf16_to_f64(d[:, :N]), o, "decode M=%d N=%d K=%d split %d C=%d" % (M, N, K, s, with_c))


def _int_operand(rng, rows, cols):
    v = rng.integers(-4, 5, size=(rows, cols))
    return np.vectorize(_INT_CODE.get)(v).astype(np.uint8)


@pytest.mark.parametrize("s", [1, 2, 4, 8])
@pytest.mark.parametrize("M", [5, 64, 128])
def test_decode_exact_integers(s, M):
    """Small-integer codes, per-row and per-block power-of-two scales that
    differ across the K blocks of a scale word, integer C aliasing D: every
    partial sum is exact, so D is the BF16 rounding of the oracle bit for bit."""
    N, K = 392, 3072
    rng = np.random.default_rng(M + 10 * s)
    qa, qb = _int_operand(rng, M, K), _int_operand(rng, N, K)
    sa = np.ldexp(1.0, rng.integers(-3, 4, size=(M, K // 128)))
    sb = np.ldexp(1.0, rng.integers(-3, 4, size=((N + 127) // 128, K // 128)))
    c = torch.from_numpy(rng.integers(-64, 65, size=(M, N)).astype(np.float32)).to(torch.bfloat16)
    want = oracle.bf16_rne(oracle.gemm_nt(qa, sa, qb, sb, P.bf16_bits(c)))
    with split(s):
        args = _args(qa, sa, qb, sb, M, N, K)
        got = P.bf16_bits(dg.fp8_gemm_nt(*args, c=c.cuda()))
        inplace = c.cuda()
        dg.fp8_gemm_nt(*args, c=inplace, d=inplace)
        _no_device_error()
    assert np.array_equal(got, want)
    assert np.array_equal(P.bf16_bits(inplace), want)


def test_decode_deterministic_and_matches_the_tiled_kernels():
    """Two calls give the same bits; the tiled kernels (DG_DECODE=0) agree
    within the tolerance."""
    M, N, K = 64, 4096, 7168
    w = workloads.dense(M, N, K, seed=9)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    with split(0):
        args = _args(qa, sa, qb, sb, M, N, K)
        d1 = dg.fp8_gemm_nt(*args)
        d2 = dg.fp8_gemm_nt(*args)
        assert dg.plan_fp8_gemm_nt_ws(M, N, K, False)["swap_ab"]
        os.environ["DG_DECODE"] = "0"
        assert not dg.plan_fp8_gemm_nt_ws(M, N, K, False)["swap_ab"]
        d3 = dg.fp8_gemm_nt(*args)
        _no_device_error()
    assert torch.equal(d1.view(torch.int16), d2.view(torch.int16))
    P.assert_close(P.bf16_to_f64(d1), P.bf16_to_f64(d3), "decode vs tiled")


def test_decode_with_pdl_in_a_graph():
    """PDL on (B prefetched into L2 before the wait), a chain of launches
    captured in a CUDA graph: replays match eager calls bit for bit."""
    M, N, K = 128, 2112, 7168
    w = workloads.dense(M, N, K, seed=4, with_c=True)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    args = _args(qa, sa, qb, sb, M, N, K)
    c = w.c.cuda()
    outs = [torch.empty(M, N, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    dg.set_pdl(True)
    try:
        with split(0):
            for d in outs:
                dg.fp8_gemm_nt(*args, c=c, d=d)
            torch.cuda.synchronize()
            ref = outs[0].clone()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for d in outs:
                    dg.fp8_gemm_nt(*args, c=c, d=d)
            for _ in range(2):
                for d in outs:
                    d.zero_()
                g.replay()
                torch.cuda.synchronize()
                for d in outs:
                    assert torch.equal(d.view(torch.int16), ref.view(torch.int16))
            _no_device_error()
    finally:
        dg.set_pdl(False)
    P.assert_close(P.bf16_to_f64(ref), oracle.gemm_nt(qa, sa, qb, sb, P.bf16_bits(w.c)), "decode pdl graph")
