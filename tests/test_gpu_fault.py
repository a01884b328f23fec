"""Failure detection on the GPU without a GPU fault: a test hook makes the
producer of CTA 0 arm one pipeline stage without filling it, so the MMA
issuer's bounded wait expires.  The launch must end by itself with
DG_ERR_DEVICE_TIMEOUT recorded (read on the host), and the context must stay
usable: the next launch is correct."""
import os

import numpy as np
import pytest
import torch

import oracle
import moe_grouped_gemm_fp8_gb300 as dg
import _parity as P

pytestmark = pytest.mark.gpu

DG_ERR_DEVICE_TIMEOUT = 5
# CTA 0's first expired wait may be the MMA issuer's wait for the unfilled
# stage (3), the epilogue's wait for that tile's accumulator (4), the
# producer's drain of the stage (6) or the MMA drain (5), whichever deadline
# passes first
SITES = {3, 4, 5, 6}


def test_dropped_stage_times_out_and_context_survives():
    M, N, K = 256, 256, 1024
    g = torch.Generator().manual_seed(113)
    a = torch.randn(M, K, generator=g); b = torch.randn(N, K, generator=g)
    qa, _, sa = oracle.quantize(a.numpy(), 1)
    qb, _, sb = oracle.quantize(b.numpy(), 128)
    dev = (P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    assert dg.get_device_error()[0] == 0
    dg.set_wait_timeout_ns(2_000_000)  # 2 ms
    dg.debug_set_drop_load(3)  # K block 2 of CTA 0's first tile
    os.environ["DG_SPLIT_K"] = "1"  # the hook is in the single-CTA pipeline
    try:
        dg.fp8_gemm_nt(*dev)
        st, word = dg.get_device_error()
    finally:
        dg.debug_set_drop_load(0)
        os.environ.pop("DG_SPLIT_K", None)
        dg.set_wait_timeout_ns(2_000_000_000)
    assert st == DG_ERR_DEVICE_TIMEOUT, (st, hex(word))
    assert word & 0xFF == DG_ERR_DEVICE_TIMEOUT and (word >> 8) & 0xFFFF in SITES, hex(word)
    assert (word >> 32) == 0  # recorded by CTA 0
    # the context is intact: the same GEMM runs correctly (split-K path included)
    d = dg.fp8_gemm_nt(*dev)
    assert dg.get_device_error()[0] == 0
    P.assert_close(P.bf16_to_f64(d), oracle.gemm_nt(qa, sa, qb, sb), "after the injected timeout")


@pytest.mark.parametrize("decode", ["0", "1"], ids=["tiled", "swapped"])
def test_dropped_stage_in_a_split_k_cluster_times_out_everywhere(decode):
    """The same hook in a 4-CTA split-K cluster (the tiled kernel, and the
    decode kernel with swapped operand roles): CTA 0 never finishes its K
    slice, so the other CTAs' waits for its partials expire too; every CTA
    ends by itself, the error word holds a timeout, and the context stays
    usable."""
    M, N, K = 64, 256, 2048
    g = torch.Generator().manual_seed(114)
    a = torch.randn(M, K, generator=g); b = torch.randn(N, K, generator=g)
    qa, _, sa = oracle.quantize(a.numpy(), 1)
    qb, _, sb = oracle.quantize(b.numpy(), 128)
    dev = (P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    assert dg.get_device_error()[0] == 0
    dg.set_wait_timeout_ns(2_000_000)  # 2 ms
    dg.debug_set_drop_load(2)
    os.environ["DG_SPLIT_K"] = "4"
    os.environ["DG_DECODE"] = decode
    try:
        assert dg.plan_fp8_gemm_nt_ws(M, N, K)["swap_ab"] == (decode == "1")
        dg.fp8_gemm_nt(*dev)
        st, word = dg.get_device_error()
    finally:
        dg.debug_set_drop_load(0)
        os.environ.pop("DG_SPLIT_K", None)
        dg.set_wait_timeout_ns(2_000_000_000)
    assert st == DG_ERR_DEVICE_TIMEOUT, (st, hex(word))
    assert word & 0xFF == DG_ERR_DEVICE_TIMEOUT, hex(word)
    os.environ["DG_SPLIT_K"] = "4"
    try:
        d = dg.fp8_gemm_nt(*dev)
    finally:
        os.environ.pop("DG_SPLIT_K", None)
        os.environ.pop("DG_DECODE", None)
    assert dg.get_device_error()[0] == 0
    P.assert_close(P.bf16_to_f64(d), oracle.gemm_nt(qa, sa, qb, sb), "after the injected split-K timeout")


def test_dropped_stage_in_a_multicast_pair_times_out_everywhere():
    """The same hook in a 2-CTA cluster of 256-row tiles that share each B
    tile by TMA multicast: CTA 0 never fills one stage, so its peer's copy of
    that stage (which waits for CTA 0's half of B) never fills either; both
    CTAs' waits expire, both end by themselves (the abort marks the peer and
    both take the release/acquire cluster barrier), the error word holds a
    timeout, and the context stays usable."""
    M, N, K = 512, 384, 2048
    g = torch.Generator().manual_seed(115)
    a = torch.randn(M, K, generator=g); b = torch.randn(N, K, generator=g)
    qa, _, sa = oracle.quantize(a.numpy(), 1)
    qb, _, sb = oracle.quantize(b.numpy(), 128)
    dev = (P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    env = {"DG_SPLIT_K": "1", "DG_BLOCK_M": "256", "DG_BLOCK_N": "192", "DG_STREAM_K": "0", "DG_MULTICAST": "1"}
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        assert dg.plan_fp8_gemm_nt_ws(M, N, K)["multicast"]
        assert dg.get_device_error()[0] == 0
        dg.set_wait_timeout_ns(2_000_000)  # 2 ms
        dg.debug_set_drop_load(2)
        try:
            dg.fp8_gemm_nt(*dev)
            st, word = dg.get_device_error()
        finally:
            dg.debug_set_drop_load(0)
            dg.set_wait_timeout_ns(2_000_000_000)
        assert st == DG_ERR_DEVICE_TIMEOUT, (st, hex(word))
        assert word & 0xFF == DG_ERR_DEVICE_TIMEOUT, hex(word)
        d = dg.fp8_gemm_nt(*dev)
        assert dg.get_device_error()[0] == 0
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    P.assert_close(P.bf16_to_f64(d), oracle.gemm_nt(qa, sa, qb, sb), "after the injected multicast-pair timeout")
