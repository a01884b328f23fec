"""CPU-only checks of the tile choosers (dg_plan_fp8_gemm_nt and the two
M-grouped queries): the same host arithmetic the calls use to pick their
launch, queried without a GPU.  Pins the choices measured fastest on GB300
(152 SMs) for the prefill, decode, contiguous and masked workloads, and checks
invariants any choice must satisfy."""
import ctypes as C
import os
from contextlib import contextmanager

import numpy as np
import pytest

import moe_grouped_gemm_fp8_gb300 as dg
from moe_grouped_gemm_fp8_gb300 import _lib, workloads

SMS = 152
OVERRIDES = ("DG_BLOCK_M", "DG_BLOCK_N", "DG_SPLIT_K", "DG_CTA_PAIR", "DG_STREAM_K", "DG_MULTICAST",
             "DG_TALL_EPI8")


@pytest.fixture(scope="module", autouse=True)
def built():
    from moe_grouped_gemm_fp8_gb300 import build
    build.build()


@contextmanager
def env(**kw):
    old = {k: os.environ.get(k) for k in OVERRIDES}
    for k in OVERRIDES:
        os.environ.pop(k, None)
    os.environ.update({k: str(v) for k, v in kw.items()})
    try:
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def plan(m, n, k, has_c=False, sms=SMS):
    p = dg.plan_fp8_gemm_nt(m, n, k, has_c, sms)
    return p["block_m"], p["block_n"], p["split_k"], p["cta_pair"]


# (N, K, with C) -> (block_m, block_n) at M = 4096: the tiles the prefill
# sweeps on GB300 measured fastest (or within noise of it), every tile forced
# in turn; 256-row tiles drain their accumulator with eight epilogue warps
PREFILL_CHOICE = {
    (2112, 7168, False): (128, 256), (2112, 7168, True): (128, 256),
    (24576, 1536, False): (256, 224), (24576, 1536, True): (256, 224),
    (7168, 16384, False): (256, 192), (7168, 16384, True): (256, 192),
    (4096, 7168, False): (256, 224), (4096, 7168, True): (256, 224),
    (7168, 2048, False): (256, 192), (7168, 2048, True): (256, 192),
}


@pytest.mark.parametrize("has_c", [False, True])
def test_prefill_shapes_take_the_measured_tiles(has_c):
    with env():
        for cfg in workloads.PREFILL:
            want = PREFILL_CHOICE[(cfg["n"], cfg["k"], has_c)]
            assert plan(cfg["m"], cfg["n"], cfg["k"], has_c) == want + (1, False), cfg


# decode (M = 64, 128): the swapped-operand kernel where its strips' K blocks
# split over clusters of 4 (measured faster on GB300), the tiled kernels
# elsewhere: split-K over 2 where 128-column tiles leave SMs idle, none where
# they fill the GPU (N = 24576); 64-row A slots for M = 64.
# (N, K) -> (block_n, split_k, swap_ab)
DECODE_CHOICE = {
    (2112, 7168): (128, 4, True),
    (24576, 1536): (192, 1, False),
    (7168, 16384): (128, 2, False),
    (4096, 7168): (128, 4, True),
    (7168, 2048): (128, 2, False),
}


def plan_swap(m, n, k, has_c=False, sms=SMS):
    p = dg.plan_fp8_gemm_nt_ws(m, n, k, has_c, sms)
    return p["block_m"], p["block_n"], p["split_k"], p["cta_pair"], p["swap_ab"]


@pytest.mark.parametrize("m", [64, 128])
def test_decode_shapes(m):
    with env():
        for cfg in workloads.PREFILL:
            bn, ks, swap = DECODE_CHOICE[(cfg["n"], cfg["k"])]
            assert plan_swap(m, cfg["n"], cfg["k"]) == (m if m == 64 else 128, bn, ks, False, swap), cfg
            assert plan(m, cfg["n"], cfg["k"]) == (m if m == 64 else 128, bn, ks, False), cfg


def test_decode_split_rules():
    """The swapped-operand kernel runs one wave of clusters: S CTAs per
    strip, at most 152 CTAs, at most floor(19 / S) clusters per 19-SM GPC,
    every CTA's K range within 8 scale words (29 K blocks)."""
    with env():
        # 17 strips: 17 clusters of 8 would take two waves, so 4
        assert plan_swap(64, 2112, 7168)[2:] == (4, False, True)
        # 8 strips of 7 K blocks: clusters of 8 (each CTA one K block or more)
        assert plan_swap(32, 1000, 1024)[2:] == (8, False, True) and plan_swap(32, 1000, 1024)[0] == 32
        # K of 2 blocks: at most 2 CTAs per strip: clusters of 2 are left to the tiled kernels
        assert plan_swap(64, 1024, 256)[4] is False
        # 17 strips of 132 K blocks: 4 CTAs would take 33 blocks (9 scale words)
        # each, 8 would not fit in one wave: the tiled kernels
        assert plan_swap(64, 2112, 132 * 128)[4] is False
        # 16 strips of 128 K blocks: clusters of 8, 16 blocks (4 scale words) each
        assert plan_swap(64, 2048, 16384)[2:] == (8, False, True)
    with env(DG_SPLIT_K=2):
        assert plan_swap(64, 7168, 2048)[2:] == (2, False, True)
    with env(DG_SPLIT_K=8):  # 17 clusters of 8 do not fit in one wave: tiled kernels
        assert plan_swap(64, 2112, 7168)[4] is False


def test_invariants_over_random_shapes():
    rng = np.random.default_rng(5)
    with env():
        for _ in range(400):
            m = int(rng.choice([1, 7, 64, 65, 127, 128, 129, 255, 256, 257, 1000, 4096, 16384]))
            n = 8 * int(rng.integers(1, 4000))
            k = 128 * int(rng.integers(1, 130))
            sms = int(rng.choice([1, 2, 8, 66, 132, 152]))
            bm, bn, ks, pair, swap = plan_swap(m, n, k, bool(rng.integers(0, 2)), sms)
            kb = k // 128
            m_blocks = -(-m // 128)
            if swap:
                # decode kernel: one wave of clusters of 4 or 8 CTAs, each CTA
                # at least one K block and at most 8 scale words of them
                strips = -(-n // 128)
                assert m <= 128 and bn == 128 and bm == (32 if m <= 32 else 64 if m <= 64 else 128)
                assert ks in (4, 8) and strips * ks <= sms and ks <= kb and not pair
                assert strips <= max(1, sms // 19) * (19 // ks)
                for r in range(ks):
                    k0, k1 = kb * r // ks, kb * (r + 1) // ks
                    assert k1 > k0 and ((k1 - 1) >> 2) - (k0 >> 2) + 1 <= 8
                continue
            assert bn in (128, 192, 224, 256)
            assert ks in (1, 2, 4) and not pair
            if ks > 1:
                # only when the split's clusters fit on the SMs, every CTA's K slice non-empty
                assert bn == 128 and m_blocks * (-(-n // 128)) * ks <= sms
                assert (ks - 1) * (-(-kb // ks)) < kb
            assert bm in (64, 128, 256)
            if bm == 64:
                assert m <= 64 and bn in (128, 192)
            if bm == 256:
                assert m > 128 and bn in (192, 224) and ks == 1
            if m <= 64 and ks == 1 and bn in (128, 192):
                assert bm == 64


def test_environment_overrides():
    with env(DG_BLOCK_N=192):
        assert plan(4096, 7168, 16384) == (128, 192, 1, False)  # a forced width means 128-row tiles
    with env(DG_BLOCK_M=256):
        assert plan(4096, 2112, 7168) == (256, 192, 1, False)
    with env(DG_BLOCK_M=256, DG_BLOCK_N=224):
        assert plan(4096, 2112, 7168) == (256, 224, 1, False)
    with env(DG_BLOCK_M=128):
        assert plan(4096, 7168, 16384)[0] == 128
    with env(DG_SPLIT_K=1):
        assert plan(64, 4096, 7168)[2] == 1
    with env(DG_SPLIT_K=2):
        assert plan(64, 4096, 7168) == (64, 128, 2, False)
    with env(DG_SPLIT_K=4):
        assert plan(64, 4096, 256)[2] == 2  # 2 K blocks cannot feed 4 CTAs
    with env(DG_CTA_PAIR=1):
        bm, bn, ks, pair = plan(4096, 7168, 16384)
        assert pair and bm == 256 and bn in (192, 224, 256)


def test_fewer_sms_change_the_split():
    with env():
        assert plan(64, 2112, 7168, sms=SMS)[2] == 4
        assert plan(64, 2112, 7168, sms=40)[2] == 2   # 17 tiles x 2 <= 40 < 17 x 4
        assert plan(64, 2112, 7168, sms=20)[2] == 1


def test_argument_checks():
    L = _lib.lib()
    out = [C.c_int32(-1) for _ in range(4)]
    refs = [C.byref(o) for o in out]
    assert L.dg_plan_fp8_gemm_nt(128, 256, 512, 0, SMS, *refs) == 0
    assert L.dg_plan_fp8_gemm_nt(0, 256, 512, 0, SMS, *refs) == 0
    assert [o.value for o in out] == [0, 0, 0, 0]                       # empty: nothing launched
    assert L.dg_plan_fp8_gemm_nt(128, 256, 500, 0, SMS, *refs) == 2      # K % 128
    assert L.dg_plan_fp8_gemm_nt(128, 260, 512, 0, SMS, *refs) == 2      # N % 8
    assert L.dg_plan_fp8_gemm_nt(-1, 256, 512, 0, SMS, *refs) == 1
    assert L.dg_plan_fp8_gemm_nt(128, 256, 512, 0, 0, *refs) == 1        # no SMs
    assert L.dg_plan_fp8_gemm_nt(128, 256, 512, 0, SMS, None, *refs[1:]) == 1


# ------------------------------------------------------------------ M-grouped forms

def test_contiguous_workload_takes_256_row_pairs():
    # 8 experts of the seed-31 contiguous workload: 40448 padded rows, N=4096, K=7168
    with env():
        assert dg.plan_m_grouped_fp8_gemm_nt_contiguous(40448, 4096, 7168, 8) == {"block_m": 256, "block_n": 224}
    with env(DG_BLOCK_M=128):
        assert dg.plan_m_grouped_fp8_gemm_nt_contiguous(40448, 4096, 7168, 8)["block_m"] == 128


def test_contiguous_pairs_only_when_the_pair_table_fits():
    with env():
        for m_blocks, groups in ((10, 3), (300, 8), (2000, 40), (2100, 8), (100, 600)):
            p = dg.plan_m_grouped_fp8_gemm_nt_contiguous(128 * m_blocks, 4096, 7168, groups)
            assert p["block_n"] in (128, 192, 224, 256)
            if p["block_m"] == 256:
                assert groups <= 512 and (m_blocks + groups + 1) // 2 <= 1024 and p["block_n"] in (192, 224)


def test_masked_workload_streams_256_columns():
    # 16 experts x 256 rows, N=7168, K=2048; the bench passes the mean count (102)
    with env():
        assert dg.plan_m_grouped_fp8_gemm_nt_masked(16, 256, 7168, 2048, 102) == \
            {"block_m": 128, "block_n": 256, "cta_pair": False}
        # without a hint the capacity (2 blocks per expert) drives the estimate
        assert dg.plan_m_grouped_fp8_gemm_nt_masked(16, 256, 7168, 2048, 0)["block_n"] == 224
    with env(DG_CTA_PAIR=1):
        p = dg.plan_m_grouped_fp8_gemm_nt_masked(16, 256, 7168, 2048, 102)
        assert p["cta_pair"] and p["block_m"] == 256


def test_grouped_argument_checks():
    L = _lib.lib()
    o = [C.c_int32(-1) for _ in range(3)]
    r = [C.byref(x) for x in o]
    assert L.dg_plan_m_grouped_fp8_gemm_nt_contiguous(0, 4096, 7168, 8, SMS, r[0], r[1]) == 0
    assert [x.value for x in o[:2]] == [0, 0]
    assert L.dg_plan_m_grouped_fp8_gemm_nt_contiguous(1000, 4096, 7168, 8, SMS, r[0], r[1]) == 2   # M % 128
    assert L.dg_plan_m_grouped_fp8_gemm_nt_contiguous(1024, 4096, 7168, 8, 0, r[0], r[1]) == 1     # no SMs
    assert L.dg_plan_m_grouped_fp8_gemm_nt_contiguous(1024, 4096, 7168, 8, SMS, None, r[1]) == 1
    assert L.dg_plan_m_grouped_fp8_gemm_nt_masked(16, 256, 7168, 2000, 0, SMS, *r) == 2          # K % 128
    assert L.dg_plan_m_grouped_fp8_gemm_nt_masked(16, 256, 7168, 2048, -1, SMS, *r) == 1         # expected_m
    assert L.dg_plan_m_grouped_fp8_gemm_nt_masked(100000, 16, 7168, 2048, 0, SMS, *r) == 7       # groups
    assert L.dg_plan_m_grouped_fp8_gemm_nt_masked(0, 256, 7168, 2048, 0, SMS, *r) == 0
    assert [x.value for x in o] == [0, 0, 0]


# ------------------------------------------------------------------ stream-K


def plan_ws(m, n, k, has_c=False, sms=SMS):
    p = dg.plan_fp8_gemm_nt_ws(m, n, k, has_c, sms)
    return p["block_m"], p["block_n"], p["split_k"], p["cta_pair"], p["stream_k"]


@pytest.mark.parametrize("has_c", [False, True])
def test_stream_k_needs_its_fixed_cost_repaid(has_c):
    """With a workspace the plan is dg_fp8_gemm_nt's unless stream-K's
    estimate, which carries the measured cost of the partial sums (~22 K
    blocks per CTA), wins by 10%: on 152 SMs no prefill or decode shape does
    (M = 4096, (N, K) = (2112, 7168), whose last wave is mostly empty, measured
    slower with stream-K than with 128 x 256 tiles); 17 long tiles on 16 SMs
    (a second wave of one tile) do."""
    with env():
        for cfg in workloads.PREFILL + workloads.DECODE:
            m, n, k = cfg["m"], cfg["n"], cfg["k"]
            assert plan_ws(m, n, k, has_c) == plan(m, n, k, has_c) + (False,)
            assert dg.fp8_gemm_nt_workspace_size(m, n, k, has_c, SMS) == 0
        got = plan_ws(4352, 192, 16384, has_c, sms=16)  # 17 tiles of 256 x 192 on 16 SMs
        assert got[0] == 256 and got[4], got
        assert dg.fp8_gemm_nt_workspace_size(4352, 192, 16384, has_c, 16) == 32 * 1024 + 16 * 256 * got[1] * 4


def test_stream_k_overrides():
    with env():
        os.environ["DG_STREAM_K"] = "0"
        try:
            assert not plan_ws(4352, 192, 16384, sms=16)[4]
            assert dg.fp8_gemm_nt_workspace_size(4352, 192, 16384, False, 16) == 0
            os.environ["DG_STREAM_K"] = "1"
            assert plan_ws(512, 384, 128)[4] is False     # 4 K blocks for 152 SMs: nothing to share
            assert plan_ws(4096, 7168, 2048)[:2] == (256, 224)  # 512 tiles: the 192-wide ones fill 4 waves
            assert plan_ws(512, 384, 2048, sms=8)[4]      # 4 tiles over 8 SMs
            os.environ["DG_BLOCK_N"] = "224"
            assert plan_ws(512, 384, 2048, sms=8)[:2] == (256, 224)
        finally:
            os.environ.pop("DG_STREAM_K", None)
            os.environ.pop("DG_BLOCK_N", None)


# ------------------------------------------------------------------ multicast


def test_multicast_pairs_go_with_256_row_tiles_walked_tile_by_tile():
    """Clusters of two CTAs sharing B by TMA multicast are used exactly when
    the dense plan takes 256-row tiles with eight epilogue warps, tile by
    tile: never with 128-row tiles, stream-K, CTA pairs, split-K or the
    decode kernel; DG_MULTICAST = 0 (or the four-warp epilogue) turns them
    off."""
    with env():
        seen = 0
        for cfg in workloads.PREFILL + workloads.DECODE:
            for has_c in (False, True):
                p = dg.plan_fp8_gemm_nt_ws(cfg["m"], cfg["n"], cfg["k"], has_c, SMS)
                tall = p["block_m"] == 256 and not p["cta_pair"] and not p["swap_ab"]
                assert p["multicast"] == (tall and not p["stream_k"]), (cfg, has_c, p)
                seen += p["multicast"]
        assert seen >= 4  # the prefill shapes that take 256-row tiles
        assert not dg.plan_fp8_gemm_nt_ws(4352, 192, 16384, False, 16)["multicast"]  # stream-K
    with env(DG_BLOCK_M=128):
        assert not dg.plan_fp8_gemm_nt_ws(4096, 7168, 16384, False, SMS)["multicast"]
    with env(DG_MULTICAST=0):
        assert not dg.plan_fp8_gemm_nt_ws(4096, 7168, 16384, False, SMS)["multicast"]
    with env(DG_TALL_EPI8=0):
        assert not dg.plan_fp8_gemm_nt_ws(4096, 7168, 16384, False, SMS)["multicast"]
    with env(DG_CTA_PAIR=1):
        p = dg.plan_fp8_gemm_nt_ws(4096, 7168, 16384, False, SMS)
        assert p["cta_pair"] and not p["multicast"]
    with env():
        assert dg.plan_fp8_gemm_nt_ws(4096, 7168, 16384, False, SMS)["multicast"]
