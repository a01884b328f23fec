"""GPU parity of the GEMMs against the oracle on small and ragged shapes:
bit-exact where the FP32 accumulation is exact, within the stated tolerance
otherwise; rows and columns the kernel must not write are compared bit for bit
against a sentinel fill."""
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


# (CTA pair, tile width): single-CTA 128-row tiles at every width, and
# 256-row tiles on 2-CTA clusters at the widths they support
CONFIGS = [(0, 128), (0, 192), (0, 224), (0, 256), (1, 192), (1, 224), (1, 256)]
CONFIG_IDS = ["%s%d" % ("pair" if p else "cta", b) for p, b in CONFIGS]


@contextmanager
def tile_config(cfg):
    pair, bn = cfg if isinstance(cfg, tuple) else (None, cfg)
    old = {k: os.environ.get(k) for k in ("DG_BLOCK_N", "DG_CTA_PAIR")}
    if bn:
        os.environ["DG_BLOCK_N"] = str(bn)
    if pair is not None:
        os.environ["DG_CTA_PAIR"] = str(pair)
    try:
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


block_n = tile_config


def _int_operand(rng, rows, cols):
    v = rng.integers(-4, 5, size=(rows, cols))
    return np.vectorize(_INT_CODE.get)(v).astype(np.uint8)


def _no_device_error():
    st, word = dg.get_device_error()
    assert st == 0, "device error word 0x%x" % word


@pytest.mark.parametrize("bn", CONFIGS, ids=CONFIG_IDS)
@pytest.mark.parametrize("M,N,K", [(200, 264, 384), (128, 512, 1024), (5, 8, 128)])
def test_dense_exact_small_integers(bn, M, N, K):
    """Integer operands with power-of-two scales: every FP32 partial sum is
    exact, so D must equal the BF16 rounding of the oracle bit for bit."""
    rng = np.random.default_rng(M + N + K)
    qa, qb = _int_operand(rng, M, K), _int_operand(rng, N, K)
    ea = rng.integers(-2, 3, size=(M, K // 128))
    eb = rng.integers(-2, 3, size=((N + 127) // 128, K // 128))
    sa, sb = np.ldexp(1.0, ea), np.ldexp(1.0, eb)
    want = oracle.bf16_rne(oracle.gemm_nt(qa, sa, qb, sb))
    with block_n(bn):
        d = dg.fp8_gemm_nt(P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1),
                           P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    got = P.bf16_bits(d)
    bad = np.argwhere(got != want)
    assert bad.size == 0, "first mismatches (row, col): %s" % bad[:8].tolist()
    _no_device_error()


def test_dense_identity_b_is_exact():
    K = 256
    x = torch.randn(300, K, generator=torch.Generator().manual_seed(3))
    qa, _, sa = P.quantize(x, 1)
    qb = np.where(np.eye(K, dtype=bool), 0x38, 0x00).astype(np.uint8)
    sb = np.ones((2, 2))
    want = oracle.bf16_rne(oracle.gemm_nt(qa, sa, qb, sb))
    d = dg.fp8_gemm_nt(P.dev_codes(qa), P.dev_packed_sf(sa, 300, K, 1), P.dev_codes(qb),
                       P.dev_packed_sf(sb, K, K, 128))
    assert np.array_equal(P.bf16_bits(d), want)


def test_small_config_dense_128x256x512():
    w = workloads.dense(**workloads.SMALL)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    o = oracle.gemm_nt(qa, sa, qb, sb)
    d = dg.fp8_gemm_nt(P.dev_codes(qa), P.dev_packed_sf(sa, 128, 512, 1), P.dev_codes(qb),
                       P.dev_packed_sf(sb, 256, 512, 128))
    P.assert_close(P.bf16_to_f64(d), o, "dense 128x256x512")
    _no_device_error()


@pytest.mark.parametrize("bn", CONFIGS, ids=CONFIG_IDS)
@pytest.mark.parametrize("with_c", [False, True])
@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (100, 136, 640), (300, 392, 384), (129, 264, 1024), (257, 520, 256)])
def test_dense_ragged(bn, with_c, M, N, K):
    w = workloads.dense(M, N, K, seed=M * 7 + N + K, with_c=with_c)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    cb = P.bf16_bits(w.c) if with_c else None
    o = oracle.gemm_nt(qa, sa, qb, sb, cb)
    # D lives inside a wider sentinel-filled buffer: columns past N must stay untouched
    ldd = N + 24
    buf = P.sentinel_like((M, ldd))
    d = buf[:, :N]
    c = w.c.cuda() if with_c else None
    with block_n(bn):
        dg.fp8_gemm_nt(P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb),
                       P.dev_packed_sf(sb, N, K, 128), d=d, c=c)
    P.assert_close(P.bf16_to_f64(d), o, "dense %dx%dx%d" % (M, N, K))
    assert (P.bf16_bits(buf[:, N:]) == P.SENTINEL_BITS).all()
    _no_device_error()


@pytest.mark.parametrize("ks", [1, 4])
@pytest.mark.parametrize("M", [1, 7, 33, 64, 127])
def test_short_m_block_ignores_stale_shared_memory(ks, M):
    """A single M block shorter than 128 rows loads only round_up(M, 8) rows of
    A; the rest of the A tile holds whatever an earlier launch left there.  A
    launch whose A is all NaN codes runs first, then the short one must still
    match the oracle on every row it writes."""
    N, K = 392, 2048
    nan_a = torch.full((512, K), 0x7F, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    w = workloads.dense(M, N, K, seed=700 + M, with_c=True)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    o = oracle.gemm_nt(qa, sa, qb, sb, P.bf16_bits(w.c))
    b_dev, sfb_dev = P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128)
    ones = P.dev_packed_sf(np.ones((512, K // 128)), 512, K, 1)
    buf = P.sentinel_like((M, N + 24))
    d = buf[:, :N]
    with block_n(128), split_k(ks):
        dg.fp8_gemm_nt(nan_a, ones, b_dev, sfb_dev)
        dg.fp8_gemm_nt(P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), b_dev, sfb_dev, d=d, c=w.c.cuda())
    P.assert_close(P.bf16_to_f64(d), o, "M=%d after a NaN launch" % M)
    assert (P.bf16_bits(buf[:, N:]) == P.SENTINEL_BITS).all()
    _no_device_error()


@contextmanager
def tall_tiles(bn):
    """256-row tiles of width bn on one CTA each (no CTA pair, no split-K,
    which the plan would otherwise take for the smaller shapes)."""
    old = {k: os.environ.get(k) for k in ("DG_BLOCK_M", "DG_BLOCK_N", "DG_CTA_PAIR", "DG_SPLIT_K")}
    os.environ["DG_BLOCK_M"] = "256"
    os.environ["DG_BLOCK_N"] = str(bn)
    os.environ["DG_CTA_PAIR"] = "0"
    os.environ["DG_SPLIT_K"] = "1"
    try:
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


@pytest.mark.parametrize("bn", [192, 224])
@pytest.mark.parametrize("with_c", [False, True])
@pytest.mark.parametrize("M,N,K", [(129, 264, 384), (300, 392, 1024), (512, 448, 640), (700, 200, 1536)])
def test_dense_256_row_tiles(bn, with_c, M, N, K):
    """256-row tiles: two 128-row MMAs per K step share the B tile; ragged M
    leaves the second half partly or wholly outside the problem."""
    w = workloads.dense(M, N, K, seed=M + 3 * N + K + bn, with_c=with_c)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    cb = P.bf16_bits(w.c) if with_c else None
    o = oracle.gemm_nt(qa, sa, qb, sb, cb)
    buf = P.sentinel_like((M, N + 24))
    d = buf[:, :N]
    with tall_tiles(bn):
        dg.fp8_gemm_nt(P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb),
                       P.dev_packed_sf(sb, N, K, 128), d=d, c=w.c.cuda() if with_c else None)
    P.assert_close(P.bf16_to_f64(d), o, "256-row tiles BN=%d %dx%dx%d" % (bn, M, N, K))
    assert (P.bf16_bits(buf[:, N:]) == P.SENTINEL_BITS).all()
    _no_device_error()


@pytest.mark.parametrize("bn", [192, 224])
def test_dense_256_row_tiles_exact_many_tiles_per_sm(bn):
    """Exact integer products (bit-exact BF16 of the oracle) with few SMs, so
    every CTA runs many 256-row tiles through its single accumulator."""
    rng = np.random.default_rng(31 + bn)
    M, N, K = 600, 520, 1024
    qa, qb = _int_operand(rng, M, K), _int_operand(rng, N, K)
    ea = rng.integers(-2, 3, size=(M, K // 128))
    eb = rng.integers(-2, 3, size=((N + 127) // 128, K // 128))
    sa, sb = np.ldexp(1.0, ea), np.ldexp(1.0, eb)
    want = oracle.bf16_rne(oracle.gemm_nt(qa, sa, qb, sb))
    args = (P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    dg.set_num_sms(3)
    try:
        with tall_tiles(bn):
            got = P.bf16_bits(dg.fp8_gemm_nt(*args))
    finally:
        dg.set_num_sms(0)
    assert np.array_equal(got, want)
    _no_device_error()


@pytest.mark.parametrize("bn", [192, 224])
@pytest.mark.parametrize("sms", [0, 5])
@pytest.mark.parametrize("M,N,K", [(600, 520, 1024), (1024, 1000, 640), (257, 448, 2048)])
def test_dense_multicast_pairs_match_single_ctas_bitwise(bn, sms, M, N, K):
    """256-row tiles in clusters of two CTAs that load half of each B tile
    into both (TMA multicast) compute what one CTA per tile computes, bit for
    bit, with and without C; with an odd number of 256-row blocks the last
    pair's second tile lies past M and writes nothing (sentinel columns and
    rows stay untouched)."""
    w = workloads.dense(M, N, K, seed=M + N + K + bn, with_c=True)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    args = (P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    c = w.c.cuda()
    out = {}
    old = {k: os.environ.get(k) for k in ("DG_MULTICAST", "DG_STREAM_K")}
    os.environ["DG_STREAM_K"] = "0"  # tile by tile (stream-K tiles are never paired)
    dg.set_num_sms(sms)
    try:
        for mc in ("1", "0"):
            os.environ["DG_MULTICAST"] = mc
            with tall_tiles(bn):
                assert dg.plan_fp8_gemm_nt_ws(M, N, K, True, sms or 152)["multicast"] == (mc == "1")
                for with_c in (False, True):
                    buf = P.sentinel_like((M, N + 24))
                    dg.fp8_gemm_nt(*args, d=buf[:, :N], c=c if with_c else None)
                    assert (P.bf16_bits(buf[:, N:]) == P.SENTINEL_BITS).all()
                    out[mc, with_c] = P.bf16_bits(buf[:, :N])
                    if mc == "1" and with_c:
                        d_mc = buf[:, :N].clone()
    finally:
        dg.set_num_sms(0)
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    for with_c in (False, True):
        assert np.array_equal(out["1", with_c], out["0", with_c])
    o = oracle.gemm_nt(qa, sa, qb, sb, P.bf16_bits(w.c))
    P.assert_close(P.bf16_to_f64(d_mc), o, "multicast pairs BN=%d %dx%dx%d" % (bn, M, N, K))
    _no_device_error()


@pytest.mark.parametrize("tiles", ["auto", "256x192", "256x224"])
def test_dense_c_aliases_d(tiles):
    """D may be C itself: every element's C is read before its D is written
    (the 128-row epilogue fetches C a chunk ahead, the 256-row one a half
    ahead)."""
    M, N, K = 192 if tiles == "auto" else 520, 256 if tiles == "auto" else 392, 512
    w = workloads.dense(M, N, K, seed=5, with_c=True)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    args = (P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    if tiles == "auto":
        ref = dg.fp8_gemm_nt(*args, c=w.c.cuda())
        inplace = w.c.cuda().clone()
        dg.fp8_gemm_nt(*args, d=inplace, c=inplace)
    else:
        with tall_tiles(int(tiles.split("x")[1])):
            ref = dg.fp8_gemm_nt(*args, c=w.c.cuda())
            inplace = w.c.cuda().clone()
            dg.fp8_gemm_nt(*args, d=inplace, c=inplace)
    assert torch.equal(inplace.view(torch.int16), ref.view(torch.int16))


def _contig_setup(G, N, K, counts, seed):
    w = workloads.contiguous(G, N, K, seed=seed, counts=counts)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    m_sum = w.a.shape[0]
    dev = (P.dev_codes(qa), P.dev_packed_sf(sa, m_sum, K, 1), P.dev_codes(qb),
           P.dev_packed_sf(sb, N, K, 128))
    return w, (qa, sa, qb, sb), dev


@pytest.mark.parametrize("bn", CONFIGS, ids=CONFIG_IDS)
def test_contiguous_routing_and_values(bn):
    G, N, K = 4, 264, 384
    w, (qa, sa, qb, sb), dev = _contig_setup(G, N, K, [100, 0, 250, 128], seed=77)
    mi = w.m_indices.numpy()
    o, written = oracle.gemm_contiguous(qa, sa, qb, sb, mi)
    d = P.sentinel_like((mi.size, N))
    with block_n(bn):
        dg.m_grouped_fp8_gemm_nt_contiguous(*dev, w.m_indices.cuda(), d=d)
    bits = P.bf16_bits(d)
    wr = written.astype(bool)
    assert np.array_equal(wr, mi >= 0)
    assert (bits[~wr] == P.SENTINEL_BITS).all(), "padding rows were written"
    P.assert_close(P.bf16_to_f64(d)[wr], o[wr], "contiguous")
    _no_device_error()


@pytest.mark.parametrize("bn", [192, 224])
@pytest.mark.parametrize("sms", [0, 5])
def test_contiguous_256_row_tiles(bn, sms):
    """256-row tiles pair two 128-row blocks of one expert: experts with odd
    block counts end with a half-empty pair, padding rows stay untouched, an
    expert with no rows gets no pair; with few SMs each CTA runs many pairs."""
    G, N, K = 6, 264, 384
    w, (qa, sa, qb, sb), dev = _contig_setup(G, N, K, [100, 0, 250, 128, 600, 384], seed=81 + bn)
    mi = w.m_indices.numpy()
    o, written = oracle.gemm_contiguous(qa, sa, qb, sb, mi)
    d = P.sentinel_like((mi.size, N))
    dg.set_num_sms(sms)
    try:
        with tall_tiles(bn):
            dg.m_grouped_fp8_gemm_nt_contiguous(*dev, w.m_indices.cuda(), d=d)
    finally:
        dg.set_num_sms(0)
    bits = P.bf16_bits(d)
    wr = written.astype(bool)
    assert np.array_equal(wr, mi >= 0)
    assert (bits[~wr] == P.SENTINEL_BITS).all(), "padding rows were written"
    P.assert_close(P.bf16_to_f64(d)[wr], o[wr], "contiguous, 256-row tiles")
    _no_device_error()


@pytest.mark.parametrize("bn", [192, 224])
def test_contiguous_256_row_tiles_match_128_row_tiles_bitwise(bn):
    """Each output element is the same sum in the same K order whichever way
    the blocks are paired, so both tile heights give identical bits."""
    G, N, K = 5, 448, 1024
    w, _, dev = _contig_setup(G, N, K, [300, 520, 0, 129, 1000], seed=90)
    mi = w.m_indices.cuda()
    d128 = P.sentinel_like((mi.numel(), N))
    d256 = P.sentinel_like((mi.numel(), N))
    os.environ["DG_BLOCK_M"] = "128"
    try:
        dg.m_grouped_fp8_gemm_nt_contiguous(*dev, mi, d=d128)
    finally:
        os.environ.pop("DG_BLOCK_M", None)
    with tall_tiles(bn):
        dg.m_grouped_fp8_gemm_nt_contiguous(*dev, mi, d=d256)
    assert torch.equal(d128.view(torch.int16), d256.view(torch.int16))
    _no_device_error()


@pytest.mark.parametrize("G,count", [(600, 128), (4, 67200)])
def test_contiguous_256_row_tiles_fall_back_past_the_pair_table(G, count):
    """More experts than the pair table holds (600 > 512), or more 128-row
    blocks than it can pair (4 x 525 blocks > 2 x 1024): 256-row tiles are
    refused on the host and the 128-row kernel runs, bit-identical."""
    N, K = 64, 128
    w, _, dev = _contig_setup(G, N, K, [count] * G, seed=91)
    mi = w.m_indices.cuda()
    d_ref = P.sentinel_like((mi.numel(), N))
    d_req = P.sentinel_like((mi.numel(), N))
    os.environ["DG_BLOCK_M"] = "128"
    try:
        dg.m_grouped_fp8_gemm_nt_contiguous(*dev, mi, d=d_ref)
    finally:
        os.environ.pop("DG_BLOCK_M", None)
    with tall_tiles(192):
        dg.m_grouped_fp8_gemm_nt_contiguous(*dev, mi, d=d_req)
    assert torch.equal(d_ref.view(torch.int16), d_req.view(torch.int16))
    _no_device_error()


def test_contiguous_single_group_equals_dense():
    G, N, K = 1, 256, 512
    w, (qa, sa, qb, sb), dev = _contig_setup(G, N, K, [384], seed=78)
    d = dg.m_grouped_fp8_gemm_nt_contiguous(*dev, w.m_indices.cuda())
    dd = dg.fp8_gemm_nt(dev[0], dev[1], dev[2][0], dev[3][0])
    assert torch.equal(d.view(torch.int16), dd.view(torch.int16))


@pytest.mark.parametrize("tall", [0, 192])
def test_contiguous_bad_index_is_flagged_not_written(tall):
    G, N, K = 2, 128, 256
    w, (qa, sa, qb, sb), dev = _contig_setup(G, N, K, [128, 200], seed=79)
    mi = w.m_indices.clone()
    mi[128 + 5] = 7          # an expert id >= G inside expert 1's block
    mi[128 * 2] = 9          # a whole block tagged with an expert id >= G
    d = P.sentinel_like((mi.numel(), N))
    dg.get_device_error()
    if tall:
        with tall_tiles(tall):
            dg.m_grouped_fp8_gemm_nt_contiguous(*dev, mi.cuda(), d=d)
    else:
        os.environ["DG_BLOCK_M"] = "128"
        try:
            dg.m_grouped_fp8_gemm_nt_contiguous(*dev, mi.cuda(), d=d)
        finally:
            os.environ.pop("DG_BLOCK_M", None)
    st, word = dg.get_device_error()
    assert st == 6, "expected DG_ERR_DEVICE_BAD_INDEX, got %d (0x%x)" % (st, word)
    bits = P.bf16_bits(d)
    assert (bits[128 + 5] == P.SENTINEL_BITS).all()
    assert (bits[256:384] == P.SENTINEL_BITS).all()
    o, _ = oracle.gemm_contiguous(qa, sa, qb, sb, w.m_indices.numpy())
    P.assert_close(P.bf16_to_f64(d)[:128], o[:128], "block 0 unaffected")


def _masked_setup(G, cap, N, K, mm, seed):
    w = workloads.masked(G, cap, N, K, seed=seed, masked_m=mm)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    dev = (P.dev_codes(qa), P.dev_packed_sf(sa, cap, K, 1), P.dev_codes(qb),
           P.dev_packed_sf(sb, N, K, 128))
    return w, (qa, sa, qb, sb), dev


@pytest.mark.parametrize("bn", CONFIGS, ids=CONFIG_IDS)
@pytest.mark.parametrize("cap", [200, 256, 64])
def test_masked_rows_and_values(bn, cap):
    G, N, K = 4, 272, 256
    mm = [0, cap, 77 % (cap + 1), min(129, cap)]
    w, (qa, sa, qb, sb), dev = _masked_setup(G, cap, N, K, mm, seed=cap)
    o, written = oracle.gemm_masked(qa, sa, qb, sb, np.array(mm, np.int32))
    d = P.sentinel_like((G, cap, N))
    with block_n(bn):
        dg.m_grouped_fp8_gemm_nt_masked(*dev, w.masked_m.cuda(), expected_m=64, d=d)
    bits = P.bf16_bits(d)
    wr = written.astype(bool)
    assert (bits[~wr] == P.SENTINEL_BITS).all(), "rows past masked_m were written"
    P.assert_close(P.bf16_to_f64(d)[wr], o[wr], "masked")
    _no_device_error()


def test_masked_count_out_of_range_is_clamped_and_flagged():
    G, cap, N, K = 2, 128, 128, 256
    w, (qa, sa, qb, sb), dev = _masked_setup(G, cap, N, K, [cap, 3], seed=5)
    mm = torch.tensor([cap + 50, -4], dtype=torch.int32)
    d = P.sentinel_like((G, cap, N))
    dg.get_device_error()
    dg.m_grouped_fp8_gemm_nt_masked(*dev, mm.cuda(), d=d)
    st, _ = dg.get_device_error()
    assert st == 6
    bits = P.bf16_bits(d)
    assert (bits[1] == P.SENTINEL_BITS).all()
    o, _ = oracle.gemm_masked(qa, sa, qb, sb, np.array([cap, 0], np.int32))
    P.assert_close(P.bf16_to_f64(d)[0], o[0], "clamped group 0")


def test_masked_all_zero_writes_nothing():
    G, cap, N, K = 3, 128, 128, 128
    w, _, dev = _masked_setup(G, cap, N, K, [0, 0, 0], seed=6)
    d = P.sentinel_like((G, cap, N))
    dg.m_grouped_fp8_gemm_nt_masked(*dev, w.masked_m.cuda(), d=d)
    assert (P.bf16_bits(d) == P.SENTINEL_BITS).all()
    _no_device_error()



@pytest.mark.parametrize("tiles", [("cta", 128), ("cta", 192), ("cta", 224), ("cta", 256),
                                   ("pair", 256), ("tall", 192), ("tall", 224)],
                         ids=lambda t: "%s%d" % t)
def test_dense_c_exact_many_tiles_per_sm(tiles):
    """D = C + A@B.T with exact integer products and an integer C (so the FP32
    sum is exact and D is the bit-exact BF16 rounding of the oracle) on three
    SMs: every CTA runs many ragged tiles, and each tile's C is fetched while
    its accumulator is still being computed."""
    kind, bn = tiles
    rng = np.random.default_rng(41 + bn)
    M, N, K = 600, 520, 1024
    qa, qb = _int_operand(rng, M, K), _int_operand(rng, N, K)
    ea = rng.integers(-2, 3, size=(M, K // 128))
    eb = rng.integers(-2, 3, size=((N + 127) // 128, K // 128))
    sa, sb = np.ldexp(1.0, ea), np.ldexp(1.0, eb)
    c = torch.from_numpy(rng.integers(-64, 65, size=(M, N)).astype(np.float32)).to(torch.bfloat16)
    want = oracle.bf16_rne(oracle.gemm_nt(qa, sa, qb, sb, P.bf16_bits(c)))
    args = (P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    ctx = tall_tiles(bn) if kind == "tall" else tile_config((1 if kind == "pair" else 0, bn))
    dg.set_num_sms(3)
    try:
        with ctx:
            got = P.bf16_bits(dg.fp8_gemm_nt(*args, c=c.cuda()))
    finally:
        dg.set_num_sms(0)
    assert np.array_equal(got, want)
    _no_device_error()

def test_num_sms_limit_does_not_change_results():
    """The tile-by-tile walk gives the same bits on any number of SMs (the
    stream-K form, whose K split follows the SM count, is tested apart)."""
    M, N, K = 512, 1024, 512
    w = workloads.dense(M, N, K, seed=9)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    args = (P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    full = dg.fp8_gemm_nt(*args, workspace=False)
    dg.set_num_sms(7)
    try:
        few = dg.fp8_gemm_nt(*args, workspace=False)
    finally:
        dg.set_num_sms(0)
    assert torch.equal(full.view(torch.int16), few.view(torch.int16))


@pytest.mark.parametrize("K", [128, 640, 1536])
def test_scale_ring_with_many_short_tiles(K):
    """Few SMs, many tiles per CTA and K-block counts that are not multiples of
    four: the scale buffers and TMEM scale slots cycle through every slot."""
    M, N = 1024, 2048
    w = workloads.dense(M, N, K, seed=K)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    args = (P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    rows = np.arange(0, M, 37)
    o = oracle.gemm_nt_rows(qa, sa, qb, sb, rows)
    for bn in CONFIGS:
        dg.set_num_sms(6)
        try:
            with block_n(bn):
                d = dg.fp8_gemm_nt(*args)
        finally:
            dg.set_num_sms(0)
        P.assert_close(P.bf16_to_f64(d)[rows], o, "K=%d cfg=%s" % (K, bn))
    _no_device_error()


@contextmanager
def split_k(ks):
    old = os.environ.get("DG_SPLIT_K")
    os.environ["DG_SPLIT_K"] = str(ks)
    try:
        yield
    finally:
        if old is None:
            os.environ.pop("DG_SPLIT_K", None)
        else:
            os.environ["DG_SPLIT_K"] = old


@pytest.mark.parametrize("ks", [2, 4])
@pytest.mark.parametrize("with_c", [False, True])
@pytest.mark.parametrize("M,N,K", [(64, 264, 2048), (128, 136, 4096), (200, 512, 2560), (1, 8, 1024), (300, 392, 1536)])
def test_dense_split_k(ks, with_c, M, N, K):
    """K split over a cluster of CTAs, partial sums reduced through
    distributed shared memory; rows/columns past the problem stay untouched."""
    w = workloads.dense(M, N, K, seed=M + N + K + ks, with_c=with_c)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    cb = P.bf16_bits(w.c) if with_c else None
    o = oracle.gemm_nt(qa, sa, qb, sb, cb)
    buf = P.sentinel_like((M, N + 24))
    d = buf[:, :N]
    with split_k(ks):
        dg.fp8_gemm_nt(P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb),
                       P.dev_packed_sf(sb, N, K, 128), d=d, c=w.c.cuda() if with_c else None)
    P.assert_close(P.bf16_to_f64(d), o, "split-K %d %dx%dx%d" % (ks, M, N, K))
    assert (P.bf16_bits(buf[:, N:]) == P.SENTINEL_BITS).all()
    _no_device_error()


@pytest.mark.parametrize("ks", [2, 4])
def test_dense_split_k_many_tiles_per_cluster(ks):
    """Few SMs, so each cluster runs many tiles in turn: the exchange buffers
    are reused from tile to tile, and the last M block (44 rows) has quarters
    with no rows, which every CTA of the cluster skips."""
    M, N, K = 300, 392, 1536
    w = workloads.dense(M, N, K, seed=900 + ks, with_c=True)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    o = oracle.gemm_nt(qa, sa, qb, sb, P.bf16_bits(w.c))
    buf = P.sentinel_like((M, N + 24))
    d = buf[:, :N]
    dg.set_num_sms(2 * ks)
    try:
        with split_k(ks):
            dg.fp8_gemm_nt(P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb),
                           P.dev_packed_sf(sb, N, K, 128), d=d, c=w.c.cuda())
    finally:
        dg.set_num_sms(0)
    P.assert_close(P.bf16_to_f64(d), o, "split-K %d, 2 clusters" % ks)
    assert (P.bf16_bits(buf[:, N:]) == P.SENTINEL_BITS).all()
    _no_device_error()


@pytest.mark.parametrize("ks", [2, 4])
def test_dense_split_k_exact_and_deterministic(ks):
    """Exact integer products: the rank-ordered reduction must give the BF16
    rounding of the oracle bit for bit, and the same bits on every run."""
    rng = np.random.default_rng(17 + ks)
    M, N, K = 96, 392, 4096
    qa, qb = _int_operand(rng, M, K), _int_operand(rng, N, K)
    ea = rng.integers(-2, 3, size=(M, K // 128))
    eb = rng.integers(-2, 3, size=((N + 127) // 128, K // 128))
    sa, sb = np.ldexp(1.0, ea), np.ldexp(1.0, eb)
    want = oracle.bf16_rne(oracle.gemm_nt(qa, sa, qb, sb))
    args = (P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    with split_k(ks):
        first = P.bf16_bits(dg.fp8_gemm_nt(*args))
        again = P.bf16_bits(dg.fp8_gemm_nt(*args))
    assert np.array_equal(first, want)
    assert np.array_equal(first, again)
    _no_device_error()


@pytest.mark.parametrize("tile", [(128, 256), (256, 192), (256, 224)], ids=["128x256", "256x192", "256x224"])
@pytest.mark.parametrize("c_layout", ["sector_aligned", "offset_16_bytes"])
@pytest.mark.parametrize("M,N,K", [(300, 392, 512), (520, 1000, 1024)])
def test_c_row_loads(tile, c_layout, M, N, K):
    """The register-held epilogues read C row by row, with 32-byte loads when
    C's base and row stride are multiples of 32 bytes and 16-byte ones
    otherwise; N % 16 == 8 leaves a last 8-column piece per row.  Both forms,
    several tiles per CTA (the next tile's C is fetched during the current
    tile's stores), against the oracle."""
    w = workloads.dense(M, N, K, seed=3 * M + N, with_c=True)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    o = oracle.gemm_nt(qa, sa, qb, sb, P.bf16_bits(w.c))
    if c_layout == "sector_aligned":
        cbuf = torch.zeros(M, N + 8, dtype=torch.bfloat16, device="cuda")  # row stride a multiple of 32 bytes
        c = cbuf[:, :N]
    else:
        cbuf = torch.zeros(M, N + 24, dtype=torch.bfloat16, device="cuda")
        c = cbuf[:, 8:8 + N]  # base 16 bytes past a 32-byte boundary
    c.copy_(w.c.cuda())
    old = {k: os.environ.get(k) for k in ("DG_BLOCK_M", "DG_BLOCK_N")}
    os.environ["DG_BLOCK_M"], os.environ["DG_BLOCK_N"] = str(tile[0]), str(tile[1])
    dg.set_num_sms(2)  # several tiles per CTA
    try:
        assert (dg.plan_fp8_gemm_nt(M, N, K, True, 2)["block_m"], dg.plan_fp8_gemm_nt(M, N, K, True, 2)["block_n"]) == tile
        d = dg.fp8_gemm_nt(P.dev_codes(qa), P.dev_packed_sf(sa, M, K, 1), P.dev_codes(qb),
                           P.dev_packed_sf(sb, N, K, 128), c=c)
        _no_device_error()
    finally:
        dg.set_num_sms(0)
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    P.assert_close(P.bf16_to_f64(d), o, "C row loads %s %s %dx%dx%d" % (tile, c_layout, M, N, K))


@pytest.mark.parametrize("bn", [(0, 128), (0, 224)], ids=["cta128", "cta224"])
@pytest.mark.parametrize("tall", [False, True], ids=["128row", "256row"])
def test_contiguous_layout_aligned_to_the_set_alignment(bn, tall):
    """Segments padded to the alignment the setter chose (256 here): the
    kernels work on 128-row blocks, so any multiple of 128 is a valid
    contiguous layout; routing and values as with 128."""
    dg.set_mk_alignment_for_contiguous_layout(256)
    try:
        align = dg.get_mk_alignment_for_contiguous_layout()
        assert align == 256
        G, N, K = 4, 264, 512
        w = workloads.contiguous(G, N, K, seed=91, counts=[100, 0, 300, 256], align=align)
        assert all(int(p) % 256 == 0 for p in w.padded)
        qa, _, sa = P.quantize(w.a, 1)
        qb, _, sb = P.quantize(w.b, 128)
        m_sum = w.a.shape[0]
        dev = (P.dev_codes(qa), P.dev_packed_sf(sa, m_sum, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
        mi = w.m_indices.numpy()
        o, written = oracle.gemm_contiguous(qa, sa, qb, sb, mi)
        d = P.sentinel_like((m_sum, N))
        old = os.environ.get("DG_BLOCK_M")
        os.environ["DG_BLOCK_M"] = "256" if tall else "128"
        try:
            with block_n(bn if not tall else (None, 224)):
                dg.m_grouped_fp8_gemm_nt_contiguous(*dev, w.m_indices.cuda(), d=d)
        finally:
            if old is None:
                os.environ.pop("DG_BLOCK_M", None)
            else:
                os.environ["DG_BLOCK_M"] = old
        bits = P.bf16_bits(d)
        wr = written.astype(bool)
        assert (bits[~wr] == P.SENTINEL_BITS).all(), "padding rows were written"
        P.assert_close(P.bf16_to_f64(d)[wr], o[wr], "contiguous, 256-row alignment")
        _no_device_error()
    finally:
        dg.set_mk_alignment_for_contiguous_layout(128)
