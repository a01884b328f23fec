"""Stream-K form of the dense NT GEMM (dg_fp8_gemm_nt_ws): the K blocks of the
last waves' 256-row tiles are split between CTAs; the CTA holding a tile's
first K blocks adds the others' FP32 partial sums (read from the workspace
after their flags) and stores the tile.

Forced on small problems with few SMs (dg_set_num_sms) so that tiles are split
over two CTAs, over about six, and behind whole waves walked tile by tile;
checked against the oracle (tolerance, and bit for bit with exact integer
operands), with the workspace's flags back at zero after every call."""
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

FLAG_BYTES = dg.api.WORKSPACE_FLAG_BYTES


@contextmanager
def stream_k(bn, sms):
    old = {k: os.environ.get(k) for k in ("DG_STREAM_K", "DG_BLOCK_N", "DG_BLOCK_M")}
    os.environ["DG_STREAM_K"] = "1"
    os.environ["DG_BLOCK_N"] = str(bn)
    os.environ.pop("DG_BLOCK_M", None)
    dg.set_num_sms(sms)
    try:
        yield
    finally:
        dg.set_num_sms(0)
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _workspace(m, n, k, has_c, sms):
    need = dg.fp8_gemm_nt_workspace_size(m, n, k, has_c, sms)
    assert need > FLAG_BYTES, "stream-K not chosen for %s" % ((m, n, k, sms),)
    return torch.zeros(need, dtype=torch.uint8, device="cuda")


def _flags_clear(ws):
    torch.cuda.synchronize()
    assert int(ws[:FLAG_BYTES].count_nonzero()) == 0, "stream-K flags left set"


def _no_device_error():
    st, word = dg.get_device_error()
    assert st == 0, "device error word 0x%x" % word


# (M, N, K, SMs): T tiles of 256 x BN, K/128 blocks each, over SMs CTAs
CASES = [
    (512, 384, 2048, 8),     # 4 tiles, 8 CTAs: every tile split over 2 CTAs
    (512, 384, 2048, 20),    # 3.2 K blocks per CTA: tiles split over ~5 CTAs
    (1000, 376, 1024, 5),    # ragged M and N: 8 tiles over 5 CTAs
    (1536, 768, 1024, 7),    # 24 tiles: two waves tile by tile, the last ten split
]


@pytest.mark.parametrize("bn", [192, 224])
@pytest.mark.parametrize("M,N,K,sms", CASES)
@pytest.mark.parametrize("with_c", [False, True])
def test_stream_k_matches_oracle(bn, M, N, K, sms, with_c):
    w = workloads.dense(M, N, K, seed=M + N + K + sms, with_c=with_c)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    args = (P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    c = w.c.cuda() if with_c else None
    with stream_k(bn, sms):
        assert dg.plan_fp8_gemm_nt_ws(M, N, K, with_c, sms)["stream_k"]
        ws = _workspace(M, N, K, with_c, sms)
        for rep in range(2):  # the same workspace twice: its flags must be back at zero
            d = dg.fp8_gemm_nt(*args, c=c, d=P.sentinel_like((M, N)), workspace=ws)
            _no_device_error()
            _flags_clear(ws)
            o = oracle.gemm_nt(qa, sa, qb, sb, P.bf16_bits(w.c) if with_c else None)
            P.assert_close(P.bf16_to_f64(d), o, "stream-K bn=%d %s C=%d rep %d" % (bn, (M, N, K, sms), with_c, rep))


def _int_operand(rng, rows, cols):
    codes = {v: int(oracle.e4m3_encode(np.array([float(v)]))[0]) for v in range(-4, 5)}
    v = rng.integers(-4, 5, size=(rows, cols))
    return np.vectorize(codes.get)(v).astype(np.uint8)


@pytest.mark.parametrize("bn", [192, 224])
@pytest.mark.parametrize("M,N,K,sms", CASES)
def test_stream_k_exact_integers_with_c(bn, M, N, K, sms):
    """Integer operands with power-of-two scales and an integer C: every FP32
    partial sum is exact whichever CTA adds it, so D is the BF16 rounding of
    the oracle bit for bit; C may alias D."""
    rng = np.random.default_rng(7 * M + N + sms)
    qa, qb = _int_operand(rng, M, K), _int_operand(rng, N, K)
    ea = rng.integers(-2, 3, size=(M, K // 128))
    eb = rng.integers(-2, 3, size=((N + 127) // 128, K // 128))
    sa, sb = np.ldexp(1.0, ea), np.ldexp(1.0, eb)
    c = torch.from_numpy(rng.integers(-64, 65, size=(M, N)).astype(np.float32)).to(torch.bfloat16)
    want = oracle.bf16_rne(oracle.gemm_nt(qa, sa, qb, sb, P.bf16_bits(c)))
    args = (P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    with stream_k(bn, sms):
        ws = _workspace(M, N, K, True, sms)
        got = P.bf16_bits(dg.fp8_gemm_nt(*args, c=c.cuda(), workspace=ws))
        inplace = c.cuda()
        dg.fp8_gemm_nt(*args, c=inplace, d=inplace, workspace=ws)
        _no_device_error()
        _flags_clear(ws)
    assert np.array_equal(got, want)
    assert np.array_equal(P.bf16_bits(inplace), want)


def test_stream_k_deterministic_and_small_workspace_falls_back():
    """Two calls give the same bits; a workspace smaller than the query's
    figure runs the tile-by-tile walk (no error) and agrees within tolerance."""
    M, N, K, sms = 1536, 768, 1024, 7
    w = workloads.dense(M, N, K, seed=5)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    args = (P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    with stream_k(192, sms):
        ws = _workspace(M, N, K, False, sms)
        a1 = dg.fp8_gemm_nt(*args, workspace=ws)
        a2 = dg.fp8_gemm_nt(*args, workspace=ws)
        small = torch.zeros(FLAG_BYTES, dtype=torch.uint8, device="cuda")
        b = dg.fp8_gemm_nt(*args, workspace=small)
        _no_device_error()
    assert torch.equal(a1.view(torch.int16), a2.view(torch.int16))
    assert int(small.count_nonzero()) == 0
    o = oracle.gemm_nt(qa, sa, qb, sb)
    P.assert_close(P.bf16_to_f64(b), o, "fallback without stream-K")


def test_stream_k_in_a_cuda_graph():
    """Captured with the binding's own workspace (taken from the graph's pool,
    flags zeroed by a captured memset): every replay matches an eager call
    bit for bit."""
    M, N, K, sms = 512, 384, 2048, 20
    w = workloads.dense(M, N, K, seed=11, with_c=True)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    args = (P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    c = w.c.cuda()
    d = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    with stream_k(224, sms):
        dg.fp8_gemm_nt(*args, c=c, d=d)
        torch.cuda.synchronize()
        ref = d.clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            dg.fp8_gemm_nt(*args, c=c, d=d)
        for _ in range(3):
            d.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(d.view(torch.int16), ref.view(torch.int16))
        _no_device_error()
    P.assert_close(P.bf16_to_f64(ref), oracle.gemm_nt(qa, sa, qb, sb, P.bf16_bits(w.c)), "graph")
