"""Pins for the CPU oracle against facts fixed outside it.

Each test checks the oracle against something other than itself: the OCP
OFP8 E4M3 definition and its anchor table, torch's own float8/bfloat16
conversions (library routines), closed forms, exact integer arithmetic, and
brute force on tiny shapes.  The inputs are built so that a plausible mistake
(a dropped term, a transposed scale index, a wrong sign or block index) fails
at least one of them.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ofp8_value(code: int) -> float:
    """Second, independent reading of the OCP OFP8 E4M3 encoding."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** (-6)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def _torch_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


# --------------------------------------------------------------------------- E4M3


def test_e4m3_table_all_codes():
    table = oracle.e4m3_table()
    ref = np.array([_ofp8_value(c) for c in range(256)])
    lib = _torch_decode(np.arange(256))
    for c in range(256):
        if np.isnan(ref[c]):
            assert np.isnan(table[c]) and np.isnan(lib[c]), hex(c)
        else:
            assert table[c] == ref[c] == lib[c], hex(c)
            assert np.signbit(table[c]) == bool(c & 0x80), hex(c)


def test_e4m3_anchor_fixture():
    table = oracle.e4m3_table()
    n = 0
    with open(os.path.join(GOLDEN, "e4m3_anchors.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            code_s, val_s = line.split()
            code, val = int(code_s, 16), float(val_s)
            if np.isnan(val):
                assert np.isnan(table[code])
            else:
                assert table[code] == val and np.signbit(table[code]) == np.signbit(val)
            n += 1
    assert n >= 10


def test_e4m3_encode_roundtrips_every_finite_code():
    table = oracle.e4m3_table()
    codes = np.array([c for c in range(256) if not np.isnan(table[c])], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(table[codes]), codes)


def test_e4m3_encode_ties_go_to_even_code():
    table = oracle.e4m3_table()
    for c in range(0, 126):
        lo, hi = table[c], table[c + 1]
        mid = (lo + hi) / 2.0  # exact in FP64
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode([mid])[0] == want, (c, mid)
        assert oracle.e4m3_encode([-mid])[0] == (want | 0x80)
        # just off the tie rounds to the nearer neighbour
        assert oracle.e4m3_encode([np.nextafter(mid, 0)])[0] == c
        assert oracle.e4m3_encode([np.nextafter(mid, 1e9)])[0] == c + 1


def test_e4m3_encode_matches_torch_inside_range():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(200000) * s for s in (1e-3, 0.1, 1.0, 30.0, 150.0)])
    x = x[np.abs(x) < 448.0].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates_and_keeps_sign_of_zero():
    got = oracle.e4m3_encode([448.0, 464.0, 480.0, 1e30, np.inf, -500.0, -np.inf, -1e-30, 0.0, np.nan])
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x80, 0x00, 0x7F]


# --------------------------------------------------------------------------- scale rule


def test_scale_exponent_is_minimal_power_of_two():
    rng = np.random.default_rng(3)
    amaxes = np.concatenate([rng.lognormal(0, 6, 5000), [448.0, 448.0 * 2 ** -7, 1.0, 2.0 ** -30]])
    for amax in amaxes:
        e = oracle.scale_exponent(amax)
        assert 448.0 * 2.0 ** e >= amax
        assert 448.0 * 2.0 ** (e - 1) < amax


def test_scale_exponent_boundaries():
    for k in range(-20, 21):
        exact = 448.0 * 2.0 ** k
        assert oracle.scale_exponent(exact) == k
        assert oracle.scale_exponent(np.nextafter(exact, np.inf)) == k + 1
        assert oracle.scale_exponent(np.nextafter(exact, 0)) == k
    assert oracle.scale_exponent(0.0) == 0
    assert oracle.scale_exponent(1e300) == 127
    assert oracle.scale_exponent(1e-300) == -127


# --------------------------------------------------------------------------- quantize


@pytest.mark.parametrize("block_rows,rows,cols", [(1, 37, 384), (128, 300, 512), (128, 64, 128)])
def test_quantize_roundtrip_bound_and_minimality(block_rows, rows, cols):
    g = torch.Generator().manual_seed(rows * 7 + cols)
    x = (torch.randn(rows, cols, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 3)).numpy()
    q, e, s = oracle.quantize(x, block_rows)
    assert np.array_equal(s, np.ldexp(1.0, e))
    deq = _torch_decode(q)
    assert not np.isnan(deq).any()
    rb = (rows + block_rows - 1) // block_rows
    for i in range(rb):
        r0, r1 = i * block_rows, min(rows, (i + 1) * block_rows)
        for j in range(cols // 128):
            xs = x[r0:r1, j * 128:(j + 1) * 128].astype(np.float64)
            sc = s[i, j]
            err = np.abs(xs - deq[r0:r1, j * 128:(j + 1) * 128] * sc)
            assert (err <= np.maximum(2.0 ** -4 * np.abs(xs), 2.0 ** -10 * sc)).all()
            ratio = np.abs(xs) / sc
            assert ratio.max() <= 448.0
            assert ratio.max() > 224.0  # e is minimal


def test_quantize_block_indexing_structured():
    """Block (i, j) holds values of magnitude 2^(i + 3j); any mix-up of the
    row-block / column-block indices gives a different exponent grid."""
    rows, cols = 256 + 40, 5 * 128
    x = np.zeros((rows, cols), dtype=np.float32)
    for i in range(3):
        for j in range(5):
            blk = x[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            blk[...] = 0.5
            blk[min(3, blk.shape[0] - 1), 5] = 2.0 ** (i + 3 * j)
    q, e, _ = oracle.quantize(x, 128)
    for i in range(3):
        for j in range(5):
            # 448 * 2^e >= 2^(i+3j) with e minimal: 2^(i+3j) / 448 in (2^(e-1), 2^e]
            assert e[i, j] == i + 3 * j - 8, (i, j, e[i, j])
    q1, e1, _ = oracle.quantize(x, 1)
    assert e1.shape == (rows, 5)
    assert e1[3, 2] == 0 + 3 * 2 - 8 and e1[4, 2] == -9  # 0.5 -> e = -9 (448/1024 < 0.5 <= 448/512)


# --------------------------------------------------------------------------- UE8M0 packing


def test_pack_ue8m0_hand_example():
    mn, kblocks = 5, 6
    e = np.array([[r - kb for kb in range(kblocks)] for r in range(mn)], dtype=np.int32)
    packed = oracle.pack_ue8m0(e, mn, 1).view(np.uint32)
    assert packed.shape == (2, 8)
    # word (j=0, r=1): bytes e+127 of K blocks 0..3 = 128, 127, 126, 125 (LSB first)
    assert packed[0, 1] == 0x7D7E7F80
    # word (j=1, r=4): K blocks 4, 5 -> 127, 126; bytes 2..3 (no K block) are zero
    assert packed[1, 4] == 0x00007E7F
    assert packed[0, 0] == 0x7C7D7E7F
    assert (packed[:, 5:] == 0).all()  # rows past mn up to the 16-byte alignment


def test_pack_ue8m0_block_rows_values():
    e = np.array([[[-3, 4], [7, 0]], [[5, -6], [1, 2]]], dtype=np.int32)  # G=2, 2 row blocks, 2 K blocks
    packed = oracle.pack_ue8m0(e, 200, 128).view(np.uint32)
    assert packed.shape == (2, 1, 200)
    assert (packed[0, 0, :128] == ((4 + 127) << 8 | (-3 + 127))).all()
    assert (packed[0, 0, 128:200] == ((0 + 127) << 8 | (7 + 127))).all()
    assert (packed[1, 0, :128] == ((-6 + 127) << 8 | (5 + 127))).all()
    assert (packed[1, 0, 128:] == ((2 + 127) << 8 | (1 + 127))).all()


# --------------------------------------------------------------------------- GEMM: exact cases

_INT_CODES = {v: c for c, v in ((c, _ofp8_value(c)) for c in range(256)) if v in (0.0, 1.0, 2.0, 3.0, 4.0, -1.0, -2.0, -3.0, -4.0) and not (c & 0x80 and v == 0.0)}


def _small_int_operands(rng, rows, cols):
    vals = rng.integers(-4, 5, size=(rows, cols))
    codes = np.vectorize(lambda v: _INT_CODES[float(v)])(vals).astype(np.uint8)
    return vals, codes


def test_gemm_exact_small_integers_with_pow2_scales():
    rng = np.random.default_rng(11)
    M, N, K = 7, 136, 384
    av, qa = _small_int_operands(rng, M, K)
    bv, qb = _small_int_operands(rng, N, K)
    ea = rng.integers(-3, 4, size=(M, K // 128))
    eb = rng.integers(-3, 4, size=((N + 127) // 128, K // 128))
    o = oracle.gemm_nt(qa, np.ldexp(1.0, ea), qb, np.ldexp(1.0, eb))
    for m in range(M):
        for n in range(N):
            want = Fraction(0)
            for k in range(K):
                want += Fraction(int(av[m, k]) * int(bv[n, k])) * Fraction(2) ** int(ea[m, k // 128] + eb[n // 128, k // 128])
            assert Fraction(o[m, n]) == want, (m, n)


def test_gemm_with_c_adds_c_once():
    rng = np.random.default_rng(12)
    M, N, K = 5, 24, 256
    _, qa = _small_int_operands(rng, M, K)
    _, qb = _small_int_operands(rng, N, K)
    sa = np.ones((M, 2)); sb = np.ones((1, 2))
    cvals = rng.integers(-50, 50, size=(M, N)).astype(np.float32)
    cbits = torch.from_numpy(cvals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    o0 = oracle.gemm_nt(qa, sa, qb, sb)
    o1 = oracle.gemm_nt(qa, sa, qb, sb, cbits)
    assert np.array_equal(o1, o0 + cvals.astype(np.float64))


def test_gemm_identity_b_returns_dequantised_a():
    K = 256
    g = torch.Generator().manual_seed(5)
    x = torch.randn(9, K, generator=g).numpy()
    qa, ea, sa = oracle.quantize(x, 1)
    qb = np.where(np.eye(K, dtype=bool), 0x38, 0x00).astype(np.uint8)  # 1.0 on the diagonal
    o = oracle.gemm_nt(qa, sa, qb, np.ones((2, 2)))
    want = _torch_decode(qa) * np.repeat(sa, 128, axis=1)
    assert np.array_equal(o, want)


def test_gemm_permutation_b_permutes_columns():
    K = 384
    rng = np.random.default_rng(2)
    perm = rng.permutation(K)
    g = torch.Generator().manual_seed(6)
    x = torch.randn(4, K, generator=g).numpy()
    qa, _, sa = oracle.quantize(x, 1)
    qb = np.zeros((K, K), dtype=np.uint8)
    qb[np.arange(K), perm] = 0x38
    sb = np.ldexp(1.0, rng.integers(-2, 3, size=(3, 3)))
    o = oracle.gemm_nt(qa, sa, qb, sb)
    deq = _torch_decode(qa) * np.repeat(sa, 128, axis=1)
    want = deq[:, perm] * sb[np.arange(K)[:, None] // 128, perm[:, None] // 128].T
    assert np.array_equal(o, want)


@pytest.mark.parametrize("M", [1, 2, 5, 16, 17])
@pytest.mark.parametrize("N,K", [(8, 128), (16, 256), (24, 128), (136, 256)])
def test_gemm_brute_force_tiny(M, N, K):
    g = torch.Generator().manual_seed(M * 1000 + N * 10 + K)
    a = torch.randn(M, K, generator=g).numpy()
    b = torch.randn(N, K, generator=g).numpy()
    qa, _, sa = oracle.quantize(a, 1)
    qb, _, sb = oracle.quantize(b, 128)
    cbits = torch.randn(M, N, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    o = oracle.gemm_nt(qa, sa, qb, sb, cbits)
    # naive triple loop over independently dequantised FP64 matrices
    A = _torch_decode(qa) * np.repeat(sa, 128, axis=1)
    B = _torch_decode(qb) * np.repeat(np.repeat(sb, 128, axis=0)[:N], 128, axis=1)
    Cm = torch.from_numpy(cbits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    want = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            s = Cm[m, n]
            for k in range(K):
                s += A[m, k] * B[n, k]
            want[m, n] = s
    np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-12)


def test_gemm_rows_matches_full():
    g = torch.Generator().manual_seed(9)
    a = torch.randn(40, 256, generator=g).numpy(); b = torch.randn(72, 256, generator=g).numpy()
    qa, _, sa = oracle.quantize(a, 1); qb, _, sb = oracle.quantize(b, 128)
    full = oracle.gemm_nt(qa, sa, qb, sb)
    rows = np.array([39, 0, 17, 17])
    assert np.array_equal(oracle.gemm_nt_rows(qa, sa, qb, sb, rows), full[rows])


# --------------------------------------------------------------------------- grouped special cases


def _quant_groups(b):
    qs, ss = [], []
    for g in range(b.shape[0]):
        q, _, s = oracle.quantize(b[g], 128)
        qs.append(q); ss.append(s)
    return np.stack(qs), np.stack(ss)


def test_contiguous_single_group_equals_dense():
    g = torch.Generator().manual_seed(21)
    a = torch.randn(256, 256, generator=g).numpy(); b = torch.randn(1, 48, 256, generator=g).numpy()
    qa, _, sa = oracle.quantize(a, 1); qb, sb = _quant_groups(b)
    o, w = oracle.gemm_contiguous(qa, sa, qb, sb, np.zeros(256, np.int32))
    assert w.all()
    assert np.array_equal(o, oracle.gemm_nt(qa, sa, qb[0], sb[0]))


def test_contiguous_routing_and_padding():
    g = torch.Generator().manual_seed(22)
    G, N, K = 3, 40, 256
    mi = np.array([1] * 100 + [-1] * 28 + [0] * 128 + [2] * 3 + [-1] * 125 + [7] * 5 + [-1] * 123, np.int32)
    a = torch.randn(mi.size, K, generator=g).numpy(); b = torch.randn(G, N, K, generator=g).numpy()
    qa, _, sa = oracle.quantize(a, 1); qb, sb = _quant_groups(b)
    o, w = oracle.gemm_contiguous(qa, sa, qb, sb, mi)
    assert np.array_equal(w.astype(bool), (mi >= 0) & (mi < G))
    for r in range(mi.size):
        if w[r]:
            want = oracle.gemm_nt(qa[r:r + 1], sa[r:r + 1], qb[mi[r]], sb[mi[r]])[0]
            assert np.array_equal(o[r], want)
    # permuting the expert order permutes the rows' results
    perm = np.array([2, 0, 1])
    inv = np.argsort(perm)
    mi_p = np.where((mi >= 0) & (mi < G), inv[np.clip(mi, 0, G - 1)], mi).astype(np.int32)
    o_p, w_p = oracle.gemm_contiguous(qa, sa, qb[perm], sb[perm], mi_p)
    assert np.array_equal(w_p, w) and np.array_equal(o_p[w.astype(bool)], o[w.astype(bool)])


def test_masked_full_capacity_equals_per_group_dense_and_zero_writes_nothing():
    g = torch.Generator().manual_seed(23)
    G, cap, N, K = 3, 130, 32, 256
    a = torch.randn(G, cap, K, generator=g).numpy(); b = torch.randn(G, N, K, generator=g).numpy()
    qa = np.empty((G, cap, K), np.uint8); sa = np.empty((G, cap, K // 128))
    for i in range(G):
        qa[i], _, sa[i] = oracle.quantize(a[i], 1)
    qb, sb = _quant_groups(b)
    o, w = oracle.gemm_masked(qa, sa, qb, sb, np.array([cap, 0, 77], np.int32))
    assert w[0].all() and not w[1].any() and w[2, :77].all() and not w[2, 77:].any()
    assert np.array_equal(o[0], oracle.gemm_nt(qa[0], sa[0], qb[0], sb[0]))
    assert np.array_equal(o[2, :77], oracle.gemm_nt(qa[2, :77], sa[2, :77], qb[2], sb[2]))
    # out-of-range counts clamp to [0, cap]
    o2, w2 = oracle.gemm_masked(qa, sa, qb, sb, np.array([cap + 5, -3, 77], np.int32))
    assert np.array_equal(w2, w) and np.array_equal(o2[w2.astype(bool)], o[w.astype(bool)])


def test_masked_rows_subset_matches_full():
    g = torch.Generator().manual_seed(24)
    G, cap, N, K = 2, 16, 16, 128
    a = torch.randn(G, cap, K, generator=g).numpy(); b = torch.randn(G, N, K, generator=g).numpy()
    qa = np.empty((G, cap, K), np.uint8); sa = np.empty((G, cap, 1))
    for i in range(G):
        qa[i], _, sa[i] = oracle.quantize(a[i], 1)
    qb, sb = _quant_groups(b)
    mm = np.array([9, 16], np.int32)
    o, w = oracle.gemm_masked(qa, sa, qb, sb, mm)
    rows = np.array([0, 8, 9, 31, 16])
    o_r, w_r = oracle.gemm_masked(qa, sa, qb, sb, mm, rows=rows)
    assert np.array_equal(w_r, w.reshape(-1)[rows])
    assert np.array_equal(o_r[w_r.astype(bool)], o.reshape(-1, N)[rows][w_r.astype(bool)])


# --------------------------------------------------------------------------- bf16 rounding


def test_bf16_rne_matches_torch_for_fp32_values():
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-30, 30, 100000), [0.0, -0.0, 1.0, 3e38]])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_rne(x.astype(np.float64)), ref)


def test_bf16_rne_ties_to_even_from_double():
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7: ties to even (1.0)
    assert oracle.bf16_rne([1.0 + 2.0 ** -8])[0] == 0x3F80
    # 1 + 3*2^-8 is the midpoint between 1+2^-7 (odd) and 1+2^-6 (even)
    assert oracle.bf16_rne([1.0 + 3 * 2.0 ** -8])[0] == 0x3F82
    # a double just above the midpoint rounds up (no double rounding through FP32)
    assert oracle.bf16_rne([1.0 + 2.0 ** -8 + 2.0 ** -40])[0] == 0x3F81


# --------------------------------------------------------------------------- K-grouped (weight gradients)


def test_quantize_cols_is_row_quantize_of_the_transpose():
    # one scale per 128 rows of a column = the 1x128 row grouping of x.T
    g = torch.Generator().manual_seed(21)
    x = (torch.randn(384, 72, generator=g) * torch.logspace(-3, 3, 72)).numpy()
    q, e, s = oracle.quantize_cols(x)
    qt, et, st = oracle.quantize(np.ascontiguousarray(x.T), 1)
    assert np.array_equal(q, qt.T) and np.array_equal(e, et.T) and np.array_equal(s, st.T)


def test_pack_ue8m0_cols_hand_example():
    e = np.array([[0, 1, -1], [2, 0, 0], [-3, 5, 1], [0, 0, 0], [7, -7, 2]], dtype=np.int32)  # [kb=5, cols=3]
    p = oracle.pack_ue8m0_cols(e)
    assert p.shape == (2, 4)
    assert p[0, 0] == 127 | (129 << 8) | (124 << 16) | (127 << 24)
    assert p[0, 1] == 128 | (127 << 8) | (132 << 16) | (127 << 24)
    assert p[1, 0] == 134 and p[1, 1] == 120 and p[1, 2] == 129 and p[1, 3] == 0
    assert np.all(p[:, 3] == 0)


def _kg_small_ints(rng, sum_k, cols):
    vals = rng.integers(-4, 5, size=(sum_k, cols))
    codes = np.vectorize(lambda v: _INT_CODES[float(v)])(vals).astype(np.uint8)
    return vals, codes


def test_k_grouped_exact_small_integers_with_pow2_scales():
    rng = np.random.default_rng(31)
    ks = np.array([256, 0, 128, 384], dtype=np.int32)
    sum_k, M, N = int(ks.sum()), 6, 10
    av, qa = _kg_small_ints(rng, sum_k, M)
    bv, qb = _kg_small_ints(rng, sum_k, N)
    ea = rng.integers(-3, 4, size=(sum_k // 128, M))
    eb = rng.integers(-3, 4, size=(sum_k // 128, N))
    cv = rng.integers(-20, 20, size=(len(ks), M, N)).astype(np.float32)
    o = oracle.gemm_k_grouped(qa, np.ldexp(1.0, ea), qb, np.ldexp(1.0, eb), ks, c=cv)
    start = np.concatenate([[0], np.cumsum(ks)])
    for g in range(len(ks)):
        for m in range(M):
            for n in range(N):
                want = Fraction(int(cv[g, m, n]))
                for k in range(start[g], start[g + 1]):
                    want += Fraction(int(av[k, m]) * int(bv[k, n])) * Fraction(2) ** int(ea[k // 128, m] + eb[k // 128, n])
                assert Fraction(o[g, m, n]) == want, (g, m, n)


@pytest.mark.parametrize("ks", [[128], [256, 128], [0, 384, 0, 128]])
def test_k_grouped_brute_force_tiny(ks):
    ks = np.array(ks, dtype=np.int32)
    sum_k, M, N = int(ks.sum()), 9, 24
    g = torch.Generator().manual_seed(int(sum_k) + len(ks))
    a = torch.randn(sum_k, M, generator=g).numpy()
    b = torch.randn(sum_k, N, generator=g).numpy()
    c = torch.randn(len(ks), M, N, generator=g).numpy()
    qa, _, sa = oracle.quantize_cols(a)
    qb, _, sb = oracle.quantize_cols(b)
    o = oracle.gemm_k_grouped(qa, sa, qb, sb, ks, c=c)
    # naive loop over independently dequantised FP64 matrices
    A = _torch_decode(qa) * np.repeat(sa, 128, axis=0)
    B = _torch_decode(qb) * np.repeat(sb, 128, axis=0)
    start = np.concatenate([[0], np.cumsum(ks)])
    for gi in range(len(ks)):
        want = c[gi].astype(np.float64).copy()
        for m in range(M):
            for n in range(N):
                s = want[m, n]
                for k in range(start[gi], start[gi + 1]):
                    s += A[k, m] * B[k, n]
                want[m, n] = s
        np.testing.assert_allclose(o[gi], want, rtol=1e-12, atol=1e-12)


def test_k_grouped_split_of_a_group_is_additive_and_empty_group_is_c():
    rng = np.random.default_rng(41)
    sum_k, M, N = 512, 5, 8
    _, qa = _kg_small_ints(rng, sum_k, M)
    _, qb = _kg_small_ints(rng, sum_k, N)
    sa = np.ldexp(1.0, rng.integers(-2, 3, size=(4, M)))
    sb = np.ldexp(1.0, rng.integers(-2, 3, size=(4, N)))
    whole = oracle.gemm_k_grouped(qa, sa, qb, sb, [512])
    parts = oracle.gemm_k_grouped(qa, sa, qb, sb, [128, 384])
    assert np.array_equal(whole[0], parts[0] + parts[1])
    cv = rng.standard_normal((3, M, N)).astype(np.float32)
    o = oracle.gemm_k_grouped(qa, sa, qb, sb, [0, 512, 0], c=cv)
    assert np.array_equal(o[0], cv[0].astype(np.float64)) and np.array_equal(o[2], cv[2].astype(np.float64))
    assert np.array_equal(o[1], whole[0] + cv[1].astype(np.float64))


def test_k_grouped_rows_subset_and_argument_checks():
    g = torch.Generator().manual_seed(43)
    ks = np.array([128, 256], dtype=np.int32)
    a = torch.randn(384, 16, generator=g).numpy(); b = torch.randn(384, 40, generator=g).numpy()
    qa, _, sa = oracle.quantize_cols(a); qb, _, sb = oracle.quantize_cols(b)
    full = oracle.gemm_k_grouped(qa, sa, qb, sb, ks)
    rows = np.array([31, 0, 16, 17])
    sub = oracle.gemm_k_grouped(qa, sa, qb, sb, ks, rows=rows)
    assert np.array_equal(sub, full.reshape(-1, 40)[rows])
    with pytest.raises(ValueError):
        oracle.gemm_k_grouped(qa, sa, qb, sb, [128, 200])  # not a multiple of 128
    with pytest.raises(ValueError):
        oracle.gemm_k_grouped(qa, sa, qb, sb, [128, 128])  # does not cover sum_k
