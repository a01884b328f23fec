"""GPU parity of the dense GEMM in the NN, TN and TT operand layouts: the same
D = C + A @ B as NT with A and/or B stored transposed (MN-major).  The oracle
works on the K-major operands; the device receives the same E4M3 codes
transposed (a relabelling of storage, no arithmetic).  Bit-exact on small
integers with power-of-two scales, within the stated tolerance otherwise."""
import numpy as np
import pytest
import torch

import oracle
import moe_grouped_gemm_fp8_gb300 as dg
import _parity as P
from test_gpu_gemm import _INT_CODE, block_n

pytestmark = pytest.mark.gpu

LAYOUTS = ["nn", "tn", "tt"]


def _store(layout, qa, qb):
    """K-major codes qa [M,K], qb [N,K] -> the layout's storage."""
    a = np.ascontiguousarray(qa.T) if layout[0] == "t" else qa
    b = np.ascontiguousarray(qb) if layout[1] == "t" else np.ascontiguousarray(qb.T)
    return a, b


def _run(layout, qa, sa, qb, sb, m, n, k, c=None):
    a, b = _store(layout, qa, qb)
    fn = getattr(dg, "fp8_gemm_" + layout)
    d = fn(P.dev_codes(a), P.dev_packed_sf(sa, m, k, 1), P.dev_codes(b), P.dev_packed_sf(sb, n, k, 128),
           c=None if c is None else c.cuda())
    st, word = dg.get_device_error()
    assert st == 0, "device error word 0x%x" % word
    return d


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_layout_exact_small_integers(layout, bn):
    rng = np.random.default_rng(91)
    M, N, K = 208, 384, 512  # MN-major storage needs M, N % 16 == 0
    qa = np.vectorize(_INT_CODE.get)(rng.integers(-4, 5, size=(M, K))).astype(np.uint8)
    qb = np.vectorize(_INT_CODE.get)(rng.integers(-4, 5, size=(N, K))).astype(np.uint8)
    sa = np.ldexp(1.0, rng.integers(-3, 4, size=(M, K // 128)))
    sb = np.ldexp(1.0, rng.integers(-3, 4, size=((N + 127) // 128, K // 128)))
    with block_n(bn):
        d = _run(layout, qa, sa, qb, sb, M, N, K)
    want = oracle.bf16_rne(oracle.gemm_nt(qa, sa, qb, sb))
    assert np.array_equal(P.bf16_bits(d), want)


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("M,N,K,with_c", [(128, 256, 512, False), (208, 272, 384, True),
                                          (384, 512, 2048, True), (16, 128, 128, False)])
def test_layout_parity(layout, bn, M, N, K, with_c):
    g = torch.Generator().manual_seed(M + 3 * N + 7 * K)
    a = torch.randn(M, K, generator=g); b = torch.randn(N, K, generator=g)
    c = torch.randn(M, N, generator=g).to(torch.bfloat16) if with_c else None
    qa, _, sa = oracle.quantize(a.numpy(), 1)
    qb, _, sb = oracle.quantize(b.numpy(), 128)
    with block_n(bn):
        d = _run(layout, qa, sa, qb, sb, M, N, K, c)
    want = oracle.gemm_nt(qa, sa, qb, sb, None if c is None else P.bf16_bits(c))
    P.assert_close(P.bf16_to_f64(d), want, "%s bn=%d" % (layout, bn))


@pytest.mark.parametrize("layout", LAYOUTS)
def test_layout_prefill_shape_sampled(layout):
    M, N, K = 4096, 2112, 7168
    g = torch.Generator().manual_seed(97)
    a = torch.randn(M, K, generator=g); b = torch.randn(N, K, generator=g)
    qa, _, sa = oracle.quantize(a.numpy(), 1)
    qb, _, sb = oracle.quantize(b.numpy(), 128)
    d = _run(layout, qa, sa, qb, sb, M, N, K)
    rows = np.array([0, 1, 127, 128, 2047, 4095] + list(range(300, 4096, 397)), dtype=np.int64)
    want = oracle.gemm_nt_rows(qa, sa, qb, sb, rows)
    P.assert_close(P.bf16_to_f64(d[torch.from_numpy(rows).cuda()]), want, "%s prefill" % layout)
