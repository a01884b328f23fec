"""GPU parity of the K-grouped (weight-gradient) GEMM against the oracle:
experts stacked along K, MN-major E4M3 operands, FP32 output.  Bit-exact where
the FP32 accumulation is exact (small integers with power-of-two scales),
within the stated tolerance otherwise; empty experts must produce C (or 0)."""
import numpy as np
import pytest
import torch

import oracle
import moe_grouped_gemm_fp8_gb300 as dg
import _parity as P
from test_gpu_gemm import _INT_CODE, block_n

pytestmark = pytest.mark.gpu


def _no_device_error():
    st, word = dg.get_device_error()
    assert st == 0, "device error word 0x%x" % word


def _dev_cols_sf(s: np.ndarray, cols: int, sum_k: int) -> torch.Tensor:
    """Scales [sum_k/128, cols] (one per 128 rows of a column) -> packed
    layout through the library's transform (scales given per column)."""
    return P.dev_packed_sf(np.ascontiguousarray(s.T), cols, sum_k, 1)


def _prepare(a: np.ndarray, b: np.ndarray):
    qa, _, sa = oracle.quantize_cols(a)
    qb, _, sb = oracle.quantize_cols(b)
    sum_k, m = a.shape
    n = b.shape[1]
    dev = (P.dev_codes(qa), _dev_cols_sf(sa, m, sum_k), P.dev_codes(qb), _dev_cols_sf(sb, n, sum_k))
    return (qa, sa, qb, sb), dev


@pytest.mark.parametrize("bn", [128, 256])
def test_k_grouped_exact_small_integers(bn):
    rng = np.random.default_rng(61)
    ks = np.array([256, 0, 128, 512], dtype=np.int32)
    sum_k, M, N = int(ks.sum()), 144, 272
    av = rng.integers(-4, 5, size=(sum_k, M)); bv = rng.integers(-4, 5, size=(sum_k, N))
    qa = np.vectorize(_INT_CODE.get)(av).astype(np.uint8)
    qb = np.vectorize(_INT_CODE.get)(bv).astype(np.uint8)
    ea = rng.integers(-3, 4, size=(sum_k // 128, M)); eb = rng.integers(-3, 4, size=(sum_k // 128, N))
    sa, sb = np.ldexp(1.0, ea), np.ldexp(1.0, eb)
    c = rng.integers(-64, 64, size=(len(ks), M, N)).astype(np.float32)
    want = oracle.gemm_k_grouped(qa, sa, qb, sb, ks, c=c)
    with block_n(bn):
        d = dg.k_grouped_fp8_gemm_tn_contiguous(P.dev_codes(qa), _dev_cols_sf(sa, M, sum_k),
                                                P.dev_codes(qb), _dev_cols_sf(sb, N, sum_k),
                                                torch.from_numpy(ks).cuda(),
                                                c=torch.from_numpy(c).cuda())
    _no_device_error()
    got = d.cpu().double().numpy()
    assert np.array_equal(got, want), "max diff %g" % np.abs(got - want).max()


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("M,N,ks,with_c", [
    (128, 128, [128], False),
    (256, 384, [256, 0, 384, 128], True),
    (144, 208, [128, 640], True),
    (384, 512, [0, 0, 1152, 0], False),
])
def test_k_grouped_parity(bn, M, N, ks, with_c):
    ks = np.array(ks, dtype=np.int32)
    sum_k = int(ks.sum())
    g = torch.Generator().manual_seed(M * 7 + N + sum_k)
    a = torch.randn(sum_k, M, generator=g).numpy()
    b = torch.randn(sum_k, N, generator=g).numpy()
    c = torch.randn(len(ks), M, N, generator=g).numpy() if with_c else None
    host, dev = _prepare(a, b)
    want = oracle.gemm_k_grouped(*host, ks, c=c)
    with block_n(bn):
        d = torch.full((len(ks), M, N), float("nan"), device="cuda")
        dg.k_grouped_fp8_gemm_tn_contiguous(*dev, torch.from_numpy(ks).cuda(), d=d,
                                            c=None if c is None else torch.from_numpy(c).cuda())
    _no_device_error()
    got = d.cpu().double().numpy()
    for gi in range(len(ks)):
        if ks[gi] == 0:
            # an empty expert writes exactly C (or 0)
            exp = c[gi] if c is not None else np.zeros((M, N), dtype=np.float32)
            assert np.array_equal(got[gi], exp.astype(np.float64)), "expert %d" % gi
        else:
            P.assert_close(got[gi], want[gi], "expert %d bn=%d" % (gi, bn))


def test_k_grouped_c_aliases_d():
    ks = np.array([384, 256], dtype=np.int32)
    M, N = 128, 256
    g = torch.Generator().manual_seed(71)
    a = torch.randn(640, M, generator=g).numpy(); b = torch.randn(640, N, generator=g).numpy()
    c = torch.randn(2, M, N, generator=g).numpy()
    host, dev = _prepare(a, b)
    want = oracle.gemm_k_grouped(*host, ks, c=c)
    d = torch.from_numpy(c).cuda()
    dg.k_grouped_fp8_gemm_tn_contiguous(*dev, torch.from_numpy(ks).cuda(), d=d, c=d)
    _no_device_error()
    P.assert_close(d.cpu().double().numpy().reshape(-1, N), want.reshape(-1, N), "in place")


def test_k_grouped_all_experts_empty_copies_c():
    M, N = 32, 48
    c = torch.randn(3, M, N, device="cuda")
    d = torch.full_like(c, float("nan"))
    z = torch.empty(0, M, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    zb = torch.empty(0, N, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    sfa = torch.empty(dg.sf_packed_shape(M, 0), dtype=torch.int32, device="cuda")
    sfb = torch.empty(dg.sf_packed_shape(N, 0), dtype=torch.int32, device="cuda")
    ks = torch.zeros(3, dtype=torch.int32, device="cuda")
    dg.k_grouped_fp8_gemm_tn_contiguous(z, sfa, zb, sfb, ks, d=d, c=c)
    torch.cuda.synchronize()
    assert torch.equal(d, c)
    dg.k_grouped_fp8_gemm_tn_contiguous(z, sfa, zb, sfb, ks, d=d)
    torch.cuda.synchronize()
    assert torch.count_nonzero(d).item() == 0


def test_k_grouped_bad_size_is_flagged_and_counts_as_empty():
    M, N = 128, 128
    g = torch.Generator().manual_seed(73)
    a = torch.randn(384, M, generator=g).numpy(); b = torch.randn(384, N, generator=g).numpy()
    host, dev = _prepare(a, b)
    c = torch.randn(2, M, N, generator=g)
    ks = torch.tensor([100, 384], dtype=torch.int32, device="cuda")  # 100: not a multiple of 128
    d = dg.k_grouped_fp8_gemm_tn_contiguous(*dev, ks, c=c.cuda())
    st, word = dg.get_device_error()
    assert st == 6 and (word & 0xFF) == 6, (st, hex(word))
    assert torch.equal(d[0].cpu(), c[0])
    # expert 1 then starts at row 0 and spans the whole of A and B
    want = oracle.gemm_k_grouped(*host, np.array([0, 384], dtype=np.int32), c=c.numpy())
    P.assert_close(d[1].cpu().double().numpy(), want[1], "expert after a bad size")


def test_k_grouped_wgrad_like_sampled_rows():
    # 8 experts, M = 1024 (output features), N = 2048 (input features), token
    # counts U[128, 2048] rounded up to 128 with one empty expert
    rng = np.random.default_rng(79)
    ks = (rng.integers(1, 17, size=8) * 128).astype(np.int32)
    ks[3] = 0
    sum_k, M, N = int(ks.sum()), 1024, 2048
    g = torch.Generator().manual_seed(79)
    a = torch.randn(sum_k, M, generator=g).numpy()
    b = torch.randn(sum_k, N, generator=g).numpy()
    host, dev = _prepare(a, b)
    d = dg.k_grouped_fp8_gemm_tn_contiguous(*dev, torch.from_numpy(ks).cuda())
    _no_device_error()
    rows = np.array(sorted(set([gi * M + r for gi in range(8) for r in (0, 1, 127, 128, 511, M - 1)] +
                               rng.choice(8 * M, size=24, replace=False).tolist())), dtype=np.int64)
    want = oracle.gemm_k_grouped(*host, ks, rows=rows)
    got = d.reshape(-1, N)[torch.from_numpy(rows).cuda()].cpu().double().numpy()
    for i, r in enumerate(rows):
        if ks[r // M] == 0:
            assert not got[i].any()
    nz = ks[rows // M] > 0
    P.assert_close(got[nz], want[nz], "wgrad-like sampled rows")


@pytest.mark.parametrize("rows,cols", [(128, 16), (640, 36), (1024, 512), (384, 4)])
def test_quantize_cols_bit_exact(rows, cols):
    g = torch.Generator().manual_seed(rows + cols)
    x = (torch.randn(rows, cols, generator=g) * torch.logspace(-4, 4, cols)).contiguous()
    x[:128, 0] = 0.0  # an all-zero block: scale 1
    q_o, e_o, s_o = oracle.quantize_cols(x.numpy())
    q, sf = dg.quantize_fp8_cols(x.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(q.view(torch.uint8).cpu().numpy(), q_o)
    assert np.array_equal(sf.cpu().numpy(), oracle.pack_ue8m0_cols(e_o))
    q2, s2 = dg.quantize_fp8_cols(x.cuda(), packed=False)
    torch.cuda.synchronize()
    assert np.array_equal(q2.view(torch.uint8).cpu().numpy(), q_o)
    assert np.array_equal(s2.cpu().double().numpy(), s_o)


def test_k_grouped_end_to_end_with_device_quantisation():
    ks = np.array([384, 128, 0, 512], dtype=np.int32)
    sum_k, M, N = int(ks.sum()), 256, 384
    g = torch.Generator().manual_seed(83)
    a = torch.randn(sum_k, M, generator=g); b = torch.randn(sum_k, N, generator=g)
    qa, sfa = dg.quantize_fp8_cols(a.cuda())
    qb, sfb = dg.quantize_fp8_cols(b.cuda())
    d = dg.k_grouped_fp8_gemm_tn_contiguous(qa, sfa, qb, sfb, torch.from_numpy(ks).cuda())
    _no_device_error()
    ha = oracle.quantize_cols(a.numpy()); hb = oracle.quantize_cols(b.numpy())
    want = oracle.gemm_k_grouped(ha[0], ha[2], hb[0], hb[2], ks)
    got = d.cpu().double().numpy()
    for gi in range(len(ks)):
        if ks[gi]:
            P.assert_close(got[gi], want[gi], "expert %d" % gi)
        else:
            assert not got[gi].any()


@pytest.mark.parametrize("sms", [0, 5])
@pytest.mark.parametrize("M", [272, 512])
def test_k_grouped_multicast_pairs_match_single_ctas_bitwise(sms, M):
    """128 x 256 tiles in clusters of two CTAs on adjacent M blocks of one
    expert, each loading one of the B tile's two 128-column boxes into both
    (TMA multicast): the same bits as one CTA per tile, with C, an empty
    expert and (M = 272) an odd number of M blocks, whose last pair's second
    tile lies past M and writes nothing."""
    import os
    rng = np.random.default_rng(M + sms)
    ks = np.array([384, 0, 128, 640], dtype=np.int32)
    sum_k, N = int(ks.sum()), 528
    a = rng.standard_normal((sum_k, M)).astype(np.float32)
    b = rng.standard_normal((sum_k, N)).astype(np.float32)
    (qa, sa, qb, sb), dev = _prepare(a, b)
    c = torch.from_numpy(rng.standard_normal((len(ks), M, N)).astype(np.float32)).cuda()
    kst = torch.from_numpy(ks).cuda()
    out = {}
    old = {k: os.environ.get(k) for k in ("DG_MULTICAST", "DG_BLOCK_N")}
    os.environ["DG_BLOCK_N"] = "256"
    dg.set_num_sms(sms)
    try:
        for mc in ("1", "0"):
            os.environ["DG_MULTICAST"] = mc
            out[mc] = dg.k_grouped_fp8_gemm_tn_contiguous(*dev, kst, c=c).cpu()
            _no_device_error()
    finally:
        dg.set_num_sms(0)
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    assert torch.equal(out["1"].view(torch.int32), out["0"].view(torch.int32))
    want = oracle.gemm_k_grouped(qa, sa, qb, sb, ks, c=c.cpu().numpy())
    P.assert_close(out["1"].double().numpy(), want, "K-grouped multicast pairs M=%d" % M)
