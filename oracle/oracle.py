"""ctypes wrapper around ``liboracle.so`` (the plain C CPU oracle).

TEST INFRASTRUCTURE ONLY.  Arrays are numpy; every function copies its
inputs to contiguous arrays of the C type first.  The C source states the
definitions and cites the pages they follow.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = C.CDLL(path)
        p = C.c_void_p
        i64 = C.c_int64
        L.or_e4m3_table.argtypes = [p]
        L.or_e4m3_decode.argtypes = [C.c_uint8]
        L.or_e4m3_decode.restype = C.c_double
        L.or_e4m3_encode.argtypes = [C.c_double]
        L.or_e4m3_encode.restype = C.c_uint8
        L.or_e4m3_encode_array.argtypes = [p, i64, p]
        L.or_bf16_rne_array.argtypes = [p, i64, p]
        L.or_scale_exponent.argtypes = [C.c_double]
        L.or_scale_exponent.restype = C.c_int
        L.or_set_threads.argtypes = [C.c_int]
        L.or_get_threads.restype = C.c_int
        L.or_quantize.argtypes = [p, i64, i64, C.c_int, p, p, p]
        L.or_quantize.restype = C.c_int
        L.or_pack_ue8m0.argtypes = [p, i64, i64, i64, C.c_int, p]
        L.or_pack_ue8m0.restype = C.c_int
        L.or_gemm_nt.argtypes = [p, p, p, p, p, i64, i64, i64, p]
        L.or_gemm_nt.restype = C.c_int
        L.or_gemm_nt_rows.argtypes = [p, p, p, p, p, i64, i64, p, i64, p]
        L.or_gemm_nt_rows.restype = C.c_int
        L.or_gemm_contiguous.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, i64, p, p]
        L.or_gemm_contiguous.restype = C.c_int
        L.or_gemm_masked.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, i64, p, p]
        L.or_gemm_masked.restype = C.c_int
        L.or_quantize_cols.argtypes = [p, i64, i64, p, p, p]
        L.or_quantize_cols.restype = C.c_int
        L.or_gemm_k_grouped.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, p, i64, p]
        L.or_gemm_k_grouped.restype = C.c_int
        _LIB = L
    return _LIB


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def set_threads(n: int) -> None:
    lib().or_set_threads(int(n))


def get_threads() -> int:
    return int(lib().or_get_threads())


def e4m3_table() -> np.ndarray:
    out = np.empty(256, dtype=np.float64)
    lib().or_e4m3_table(_ptr(out))
    return out


def e4m3_encode(x) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().or_e4m3_encode_array(_ptr(x), x.size, _ptr(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    return e4m3_table()[_c(codes, np.uint8)]


def bf16_rne(x) -> np.ndarray:
    """FP64 -> BF16 bit patterns (uint16), round to nearest, ties to even."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().or_bf16_rne_array(_ptr(x), x.size, _ptr(out))
    return out


def scale_exponent(amax: float) -> int:
    return int(lib().or_scale_exponent(float(amax)))


def quantize(x, block_rows: int):
    """FP32 [rows, cols] -> (codes uint8 [rows, cols], exponents int32
    [ceil(rows/block_rows), cols/128], scales float64 (2^e), same shape)."""
    x = _c(x, np.float32)
    assert x.ndim == 2
    rows, cols = x.shape
    rb = (rows + block_rows - 1) // block_rows
    q = np.empty((rows, cols), dtype=np.uint8)
    e = np.empty((rb, cols // 128), dtype=np.int32)
    s = np.empty((rb, cols // 128), dtype=np.float64)
    rc = lib().or_quantize(_ptr(x), rows, cols, block_rows, _ptr(q), _ptr(e), _ptr(s))
    if rc != 0:
        raise ValueError("or_quantize rejected its arguments (rc=%d)" % rc)
    return q, e, s


def pack_ue8m0(sf_exp, mn: int, block_rows: int) -> np.ndarray:
    """exponents [G, ceil(mn/block_rows), kblocks] (or without G) ->
    packed int32 [G, ceil(kblocks/4), align(mn, 4)] (G dim kept iff given)."""
    e = _c(sf_exp, np.int32)
    squeeze = e.ndim == 2
    if squeeze:
        e = e[None]
    groups, _, kblocks = e.shape
    mn_pad = (mn + 3) // 4 * 4
    out = np.empty((groups, (kblocks + 3) // 4, mn_pad), dtype=np.int32)
    rc = lib().or_pack_ue8m0(_ptr(e), groups, mn, kblocks, block_rows, _ptr(out))
    if rc != 0:
        raise ValueError("or_pack_ue8m0 rejected its arguments (rc=%d)" % rc)
    return out[0] if squeeze else out


def gemm_nt(qa, sa, qb, sb, c_bf16_bits=None) -> np.ndarray:
    """o = C + dequant(A) @ dequant(B)^T in FP64.  qa [M,K] codes,
    sa [M,K/128], qb [N,K], sb [ceil(N/128),K/128], C as uint16 bf16 bits."""
    qa, qb = _c(qa, np.uint8), _c(qb, np.uint8)
    sa, sb = _c(sa, np.float64), _c(sb, np.float64)
    M, K = qa.shape
    N = qb.shape[0]
    cc = None if c_bf16_bits is None else _c(c_bf16_bits, np.uint16)
    o = np.empty((M, N), dtype=np.float64)
    rc = lib().or_gemm_nt(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), _ptr(cc), M, N, K, _ptr(o))
    if rc != 0:
        raise ValueError("or_gemm_nt rejected its arguments (rc=%d)" % rc)
    return o


def gemm_nt_rows(qa, sa, qb, sb, rows, c_bf16_bits=None) -> np.ndarray:
    qa, qb = _c(qa, np.uint8), _c(qb, np.uint8)
    sa, sb = _c(sa, np.float64), _c(sb, np.float64)
    rows = _c(rows, np.int64)
    K = qa.shape[1]
    N = qb.shape[0]
    cc = None if c_bf16_bits is None else _c(c_bf16_bits, np.uint16)
    o = np.empty((rows.size, N), dtype=np.float64)
    rc = lib().or_gemm_nt_rows(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), _ptr(cc), N, K,
                               _ptr(rows), rows.size, _ptr(o))
    if rc != 0:
        raise ValueError("or_gemm_nt_rows rejected its arguments (rc=%d)" % rc)
    return o


def gemm_contiguous(qa, sa, qb, sb, m_indices, rows=None):
    """Returns (o [m_sum or len(rows), N], written uint8)."""
    qa, qb = _c(qa, np.uint8), _c(qb, np.uint8)
    sa, sb = _c(sa, np.float64), _c(sb, np.float64)
    mi = _c(m_indices, np.int32)
    m_sum, K = qa.shape
    G, N, _ = qb.shape
    r = None if rows is None else _c(rows, np.int64)
    n_out = m_sum if r is None else r.size
    o = np.empty((n_out, N), dtype=np.float64)
    w = np.empty(n_out, dtype=np.uint8)
    rc = lib().or_gemm_contiguous(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), _ptr(mi), m_sum, G, N, K,
                                  _ptr(r), 0 if r is None else r.size, _ptr(o), _ptr(w))
    if rc != 0:
        raise ValueError("or_gemm_contiguous rejected its arguments (rc=%d)" % rc)
    return o, w


def gemm_masked(qa, sa, qb, sb, masked_m, rows=None):
    """qa [G,cap,K], sa [G,cap,K/128]; returns (o, written) shaped [G,cap,N] /
    [G,cap] (or flat by list position when rows is given)."""
    qa, qb = _c(qa, np.uint8), _c(qb, np.uint8)
    sa, sb = _c(sa, np.float64), _c(sb, np.float64)
    mm = _c(masked_m, np.int32)
    G, cap, K = qa.shape
    N = qb.shape[1]
    r = None if rows is None else _c(rows, np.int64)
    if r is None:
        o = np.empty((G, cap, N), dtype=np.float64)
        w = np.empty((G, cap), dtype=np.uint8)
    else:
        o = np.empty((r.size, N), dtype=np.float64)
        w = np.empty(r.size, dtype=np.uint8)
    rc = lib().or_gemm_masked(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), _ptr(mm), G, cap, N, K,
                              _ptr(r), 0 if r is None else r.size, _ptr(o), _ptr(w))
    if rc != 0:
        raise ValueError("or_gemm_masked rejected its arguments (rc=%d)" % rc)
    return o, w


def quantize_cols(x):
    """FP32 [rows, cols], rows % 128 == 0 -> (codes uint8 [rows, cols],
    exponents int32 [rows/128, cols], scales float64 (2^e), same shape): one
    scale per 128 rows of each column."""
    x = _c(x, np.float32)
    assert x.ndim == 2
    rows, cols = x.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    e = np.empty((rows // 128, cols), dtype=np.int32)
    s = np.empty((rows // 128, cols), dtype=np.float64)
    rc = lib().or_quantize_cols(_ptr(x), rows, cols, _ptr(q), _ptr(e), _ptr(s))
    if rc != 0:
        raise ValueError("or_quantize_cols rejected its arguments (rc=%d)" % rc)
    return q, e, s


def pack_ue8m0_cols(sf_exp) -> np.ndarray:
    """Column-wise exponents [kblocks, cols] -> packed int32
    [ceil(kblocks/4), align(cols, 4)]: the same word layout as pack_ue8m0 with
    one scale per row, the columns playing the rows (a transposition only)."""
    e = _c(sf_exp, np.int32)
    return pack_ue8m0(np.ascontiguousarray(e.T), e.shape[1], 1)


def gemm_k_grouped(qa, sa, qb, sb, ks, c=None, rows=None) -> np.ndarray:
    """o[g] = C[g] + A_g^T B_g in FP64.  qa [sum_k, M] codes, sa [sum_k/128, M];
    qb [sum_k, N], sb [sum_k/128, N]; ks [G] rows per expert; c FP32 [G, M, N]
    or None.  Returns [G, M, N], or [len(rows), N] for flat rows g * M + m."""
    qa, qb = _c(qa, np.uint8), _c(qb, np.uint8)
    sa, sb = _c(sa, np.float64), _c(sb, np.float64)
    ks = _c(ks, np.int32)
    sum_k, M = qa.shape
    N = qb.shape[1]
    G = ks.size
    cc = None if c is None else _c(c, np.float32)
    r = None if rows is None else _c(rows, np.int64)
    o = np.empty((G, M, N) if r is None else (r.size, N), dtype=np.float64)
    rc = lib().or_gemm_k_grouped(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), _ptr(ks), G, M, N, sum_k,
                                 _ptr(cc), _ptr(r), 0 if r is None else r.size, _ptr(o))
    if rc != 0:
        raise ValueError("or_gemm_k_grouped rejected its arguments (rc=%d)" % rc)
    return o


__all__ = [
    "lib", "set_threads", "get_threads", "e4m3_table", "e4m3_encode", "e4m3_decode", "bf16_rne",
    "scale_exponent", "quantize", "pack_ue8m0", "gemm_nt", "gemm_nt_rows", "gemm_contiguous",
    "gemm_masked", "quantize_cols", "pack_ue8m0_cols", "gemm_k_grouped",
]
