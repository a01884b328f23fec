"""GPU parity of the FP32-scale GEMM (per-K-block partials promoted out of
TMEM and scaled on the CUDA cores) against the oracle, whose definition takes
any scale: bit-exact for small integers with power-of-two FP32 scales (every
partial and product exact in FP32), within the stated tolerance for arbitrary
scales."""
import numpy as np
import pytest
import torch

import oracle
import moe_grouped_gemm_fp8_gb300 as dg
import _parity as P
from test_gpu_gemm import _INT_CODE

pytestmark = pytest.mark.gpu


def _dev_scales(sa: np.ndarray, sb: np.ndarray, m: int):
    """sa [M, K/128] -> float32 [K/128, align(M, 4)] (K-block-major, padded);
    sb [ceil(N/128), K/128] as is."""
    kb = sa.shape[1]
    m_pad = (m + 3) // 4 * 4
    t = np.zeros((kb, m_pad), dtype=np.float32)
    t[:, :m] = sa.T
    return torch.from_numpy(t).cuda(), torch.from_numpy(np.ascontiguousarray(sb, dtype=np.float32)).cuda()


def _no_device_error():
    st, word = dg.get_device_error()
    assert st == 0, "device error word 0x%x" % word


def test_fp32_scales_exact_small_integers_pow2():
    rng = np.random.default_rng(131)
    M, N, K = 200, 264, 512
    qa = np.vectorize(_INT_CODE.get)(rng.integers(-4, 5, size=(M, K))).astype(np.uint8)
    qb = np.vectorize(_INT_CODE.get)(rng.integers(-4, 5, size=(N, K))).astype(np.uint8)
    sa = np.ldexp(1.0, rng.integers(-3, 4, size=(M, K // 128)))
    sb = np.ldexp(1.0, rng.integers(-3, 4, size=((N + 127) // 128, K // 128)))
    fa, fb = _dev_scales(sa, sb, M)
    d = dg.fp8_gemm_nt_fp32_sf(P.dev_codes(qa), fa, P.dev_codes(qb), fb)
    _no_device_error()
    want = oracle.bf16_rne(oracle.gemm_nt(qa, sa, qb, sb))
    assert np.array_equal(P.bf16_bits(d), want)


@pytest.mark.parametrize("M,N,K,with_c", [(128, 128, 128, False), (200, 264, 384, True),
                                          (300, 520, 1024, False), (5, 8, 256, True)])
def test_fp32_scales_arbitrary(M, N, K, with_c):
    g = torch.Generator().manual_seed(M + N + K)
    rng = np.random.default_rng(M * N + K)
    qa = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    qb = rng.integers(0, 256, size=(N, K)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    qb[(qb & 0x7F) == 0x7F] = 0x3C
    # arbitrary positive FP32 scales over several binades, rounded to FP32
    sa = (rng.uniform(0.5, 2.0, size=(M, K // 128)) * np.exp2(rng.integers(-8, 2, size=(M, K // 128)))).astype(np.float32).astype(np.float64)
    sb = (rng.uniform(0.5, 2.0, size=((N + 127) // 128, K // 128)) * np.exp2(rng.integers(-8, 2, size=((N + 127) // 128, K // 128)))).astype(np.float32).astype(np.float64)
    c = torch.randn(M, N, generator=g).to(torch.bfloat16) if with_c else None
    fa, fb = _dev_scales(sa, sb, M)
    d = dg.fp8_gemm_nt_fp32_sf(P.dev_codes(qa), fa, P.dev_codes(qb), fb,
                               c=None if c is None else c.cuda())
    _no_device_error()
    want = oracle.gemm_nt(qa, sa, qb, sb, None if c is None else P.bf16_bits(c))
    P.assert_close(P.bf16_to_f64(d), want, "fp32 scales %dx%dx%d" % (M, N, K))


def test_fp32_scales_prefill_shape_sampled():
    M, N, K = 4096, 7168, 7168
    g = torch.Generator().manual_seed(137)
    a = torch.randn(M, K, generator=g); b = torch.randn(N, K, generator=g)
    # amax / 448 scales, not rounded to powers of two
    a_blk = a.view(M, K // 128, 128).abs().amax(-1).clamp_min(1e-30) / 448.0
    b_blk = b.view(N // 128, 128, K // 128, 128).abs().amax(dim=(1, 3)).clamp_min(1e-30) / 448.0
    sa = a_blk.double().numpy(); sb = b_blk.double().numpy()
    qa = oracle.e4m3_encode((a.double().numpy().reshape(M, K // 128, 128) / sa[:, :, None]).reshape(M, K))
    qb = oracle.e4m3_encode((b.double().numpy().reshape(N // 128, 128, K // 128, 128)
                             / sb[:, None, :, None]).reshape(N, K))
    fa, fb = _dev_scales(sa, sb, M)
    d = dg.fp8_gemm_nt_fp32_sf(P.dev_codes(qa), fa, P.dev_codes(qb), fb)
    _no_device_error()
    rows = np.array([0, 1, 127, 128, 2048, 4095] + list(range(333, 4096, 401)), dtype=np.int64)
    want = oracle.gemm_nt_rows(qa, sa.astype(np.float32).astype(np.float64), qb,
                               sb.astype(np.float32).astype(np.float64), rows)
    P.assert_close(P.bf16_to_f64(d[torch.from_numpy(rows).cuda()]), want, "fp32 scales prefill")
