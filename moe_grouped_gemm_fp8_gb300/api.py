"""Torch-facing wrappers of the C ABI in include/dg.h.

Argument marshalling only: dtype/device/shape checks, output allocation by
torch, ``data_ptr()`` and the current CUDA stream.  Every step of the
computation runs in libdg.so's kernels; there is no fallback.

Naming follows "DeepGEMM: kernels GEMM FP8 limpos e eficientes por meio de
scaling granular" (pt.news.hada.io), sections "Interface GEMM e restrições de
layout", "GEMM denso e grouped" and "Utilitários e variáveis de ambiente".
"""
import ctypes as C
from typing import Optional, Tuple

import torch

from . import _lib

FP8_DTYPES = (torch.float8_e4m3fn, torch.uint8)


class DGError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s failed: %s (%s)" % (what, _lib.status_name(status),
                                                 _lib.lib().dg_status_string(status).decode()))
        self.status = int(status)


def _check(status: int, what: str) -> None:
    if status != _lib.DG_OK:
        raise DGError(status, what)


# The current stream's raw handle without building a torch.cuda.Stream object
# (which costs ~3 us per call on the Grace host).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> C.c_void_p:
    if stream is None:
        if _raw_stream is not None:
            return C.c_void_p(_raw_stream(torch.cuda.current_device()))
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def _on_current_device(stream, *tensors) -> None:
    """The library launches on the current CUDA device: every tensor (and an
    explicit torch stream) must live there.  A pointer of another device would
    reach a kernel that cannot use it."""
    dev = torch.cuda.current_device()
    for t in tensors:
        if t is not None and t.device.index != dev:
            raise ValueError("tensor on %s, but the current CUDA device is cuda:%d "
                             "(use torch.cuda.device(...) around the call)" % (t.device, dev))
    if isinstance(stream, torch.cuda.Stream) and stream.device.index != dev:
        raise ValueError("stream of %s, but the current CUDA device is cuda:%d" % (stream.device, dev))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtypes, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype not in dtypes or not t.is_cuda or t.dim() != ndim:
        if t.dtype not in dtypes:
            raise TypeError("%s: dtype %s not in %s" % (name, t.dtype, dtypes))
        if not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % name)
        raise ValueError("%s must have %d dims, got %s" % (name, ndim, tuple(t.shape)))


def get_tma_aligned_size(x: int, element_size: int) -> int:
    return int(_lib.lib().dg_get_tma_aligned_size(int(x), int(element_size)))


def get_mk_alignment_for_contiguous_layout() -> int:
    return int(_lib.lib().dg_get_mk_alignment_for_contiguous_layout())


def set_mk_alignment_for_contiguous_layout(alignment: int) -> None:
    """A positive multiple of 128 up to 4096 (the value the getter returns)."""
    _check(_lib.lib().dg_set_mk_alignment_for_contiguous_layout(int(alignment)),
           "dg_set_mk_alignment_for_contiguous_layout")


def plan_fp8_gemm_nt(m: int, n: int, k: int, has_c: bool = False, num_sms: int = 152) -> dict:
    """The tile configuration fp8_gemm_nt chooses for an M x N x K problem on
    a device with num_sms SMs, computed on the host (no GPU needed):
    {"block_m": 64 | 128 | 256, "block_n": ..., "split_k": 1 | 2 | 4,
    "cta_pair": bool}; all zero for an empty problem."""
    out = [C.c_int32(0) for _ in range(4)]
    st = _lib.lib().dg_plan_fp8_gemm_nt(int(m), int(n), int(k), 1 if has_c else 0, int(num_sms),
                                        *[C.byref(o) for o in out])
    _check(st, "dg_plan_fp8_gemm_nt")
    bm, bn, sk, pair = (int(o.value) for o in out)
    return {"block_m": bm, "block_n": bn, "split_k": sk, "cta_pair": bool(pair)}


def plan_fp8_gemm_nt_ws(m: int, n: int, k: int, has_c: bool = False, num_sms: int = 152) -> dict:
    """The tile configuration fp8_gemm_nt chooses with a large enough
    workspace: plan_fp8_gemm_nt's keys plus "stream_k", "swap_ab" (the
    decode kernel, operand roles swapped; fp8_gemm_nt chooses it too) and
    "multicast" (256-row tiles in clusters of two sharing B by TMA multicast;
    fp8_gemm_nt chooses it too)."""
    out = [C.c_int32(0) for _ in range(7)]
    st = _lib.lib().dg_plan_fp8_gemm_nt_ws(int(m), int(n), int(k), 1 if has_c else 0, int(num_sms),
                                           *[C.byref(o) for o in out])
    _check(st, "dg_plan_fp8_gemm_nt_ws")
    bm, bn, sk, pair, strk, swap, mc = (int(o.value) for o in out)
    return {"block_m": bm, "block_n": bn, "split_k": sk, "cta_pair": bool(pair), "stream_k": bool(strk),
            "swap_ab": bool(swap), "multicast": bool(mc)}


def plan_m_grouped_fp8_gemm_nt_contiguous(m_sum: int, n: int, k: int, num_groups: int,
                                          num_sms: int = 152) -> dict:
    """The tile configuration m_grouped_fp8_gemm_nt_contiguous chooses, on the
    host: {"block_m": 128 | 256, "block_n": ...}; zeros for an empty problem."""
    out = [C.c_int32(0) for _ in range(2)]
    _check(_lib.lib().dg_plan_m_grouped_fp8_gemm_nt_contiguous(
        int(m_sum), int(n), int(k), int(num_groups), int(num_sms), *[C.byref(o) for o in out]),
        "dg_plan_m_grouped_fp8_gemm_nt_contiguous")
    return {"block_m": int(out[0].value), "block_n": int(out[1].value)}


def plan_m_grouped_fp8_gemm_nt_masked(num_groups: int, max_m: int, n: int, k: int,
                                      expected_m: int = 0, num_sms: int = 152) -> dict:
    """The tile configuration m_grouped_fp8_gemm_nt_masked chooses, on the
    host: {"block_m": 128 | 256, "block_n": ..., "cta_pair": bool}."""
    out = [C.c_int32(0) for _ in range(3)]
    _check(_lib.lib().dg_plan_m_grouped_fp8_gemm_nt_masked(
        int(num_groups), int(max_m), int(n), int(k), int(expected_m), int(num_sms),
        *[C.byref(o) for o in out]), "dg_plan_m_grouped_fp8_gemm_nt_masked")
    return {"block_m": int(out[0].value), "block_n": int(out[1].value), "cta_pair": bool(out[2].value)}


def set_num_sms(n: int) -> None:
    _check(_lib.lib().dg_set_num_sms(int(n)), "dg_set_num_sms")
    # the binding's workspaces are sized for the SM count (a fresh one has
    # its flags zeroed; the old ones are released stream-ordered)
    _WORKSPACES.clear()


def get_num_sms() -> int:
    return int(_lib.lib().dg_get_num_sms())


def set_pdl(enable: bool) -> None:
    """Programmatic dependent launch for every kernel of the library."""
    _check(_lib.lib().dg_set_pdl(1 if enable else 0), "dg_set_pdl")


def get_pdl() -> bool:
    return bool(_lib.lib().dg_get_pdl())


def set_wait_timeout_ns(ns: int) -> None:
    _check(_lib.lib().dg_set_wait_timeout_ns(int(ns)), "dg_set_wait_timeout_ns")


def debug_set_drop_load(k: int) -> None:
    """Test hook: with k > 0 the next dense NT launches leave the stage of K
    block k - 1 of CTA 0's first tile unfilled, so the kernel's bounded waits
    must end the launch with DG_ERR_DEVICE_TIMEOUT; 0 turns it off."""
    _check(_lib.lib().dg_debug_set_drop_load(int(k)), "dg_debug_set_drop_load")


def debug_plant_check(on: bool) -> None:
    """Test hook of the debug library (DG_DEBUG_LIBRARY=1): the next dense NT
    launches record DG_ERR_DEVICE_CHECK from the MMA issuer's TMEM check.  The
    release library refuses on=True (it carries no checks)."""
    _check(_lib.lib().dg_debug_plant_check(1 if on else 0), "dg_debug_plant_check")


def get_device_error(stream=None) -> Tuple[int, int]:
    """Synchronises the stream; returns (status, raw word) and clears the word.
    After a timeout the binding's own workspaces are zero-filled again (an
    aborted stream-K launch may leave flags set)."""
    detail = C.c_uint64(0)
    st = _lib.lib().dg_get_device_error(_stream(stream), C.byref(detail))
    if int(st) == 5:  # DG_ERR_DEVICE_TIMEOUT
        for ws in _WORKSPACES.values():
            ws[:min(ws.numel(), WORKSPACE_FLAG_BYTES)].zero_()
        torch.cuda.synchronize()
    return int(st), int(detail.value)


def sf_packed_shape(mn: int, k: int, groups: Optional[int] = None):
    kp = (k // 128 + 3) // 4
    shape = (kp, (mn + 3) // 4 * 4)  # rows padded to 16 bytes (dg_get_tma_aligned_size(mn, 4))
    return shape if groups is None else (groups,) + shape


def quantize_fp8(x: torch.Tensor, block_rows: int, packed: bool = True, out=None, stream=None):
    """FP32 [rows, cols] or [G, rows, cols] -> (E4M3 codes, scales).

    block_rows=1: 1x128 row groups (activations); 128: 128x128 blocks
    (weights).  packed=True gives the int32 UE8M0 layout the GEMMs take;
    packed=False FP32 scales [G?, ceil(rows/block_rows), cols/128].
    out=(q, sf) writes into preallocated tensors of those shapes."""
    if x.dim() not in (2, 3):
        raise ValueError("x must be [rows, cols] or [groups, rows, cols]")
    _need(x, "x", (torch.float32,), x.dim())
    x = x.contiguous()
    grouped = x.dim() == 3
    groups = x.shape[0] if grouped else 1
    rows, cols = x.shape[-2], x.shape[-1]
    if packed:
        sf_shape = sf_packed_shape(rows, cols, groups if grouped else None)
        sf_dtype = torch.int32
    else:
        sf_shape = ((groups,) if grouped else ()) + ((rows + block_rows - 1) // block_rows, cols // 128)
        sf_dtype = torch.float32
    if out is None:
        q = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device=x.device)
        sf = torch.empty(sf_shape, dtype=sf_dtype, device=x.device)
    else:
        q, sf = out
        _need(q, "q", FP8_DTYPES, x.dim())
        _need(sf, "sf", (sf_dtype,), len(sf_shape))
        if tuple(q.shape) != tuple(x.shape) or tuple(sf.shape) != tuple(sf_shape) or \
                not q.is_contiguous() or not sf.is_contiguous():
            raise ValueError("out tensors must be contiguous %s / %s" % (tuple(x.shape), sf_shape))
    _on_current_device(stream, x, q, sf)
    st = _lib.lib().dg_quantize_fp8(_ptr(x), _ptr(q), _ptr(sf), groups, rows, cols, int(block_rows),
                                    _lib.DG_SF_UE8M0_PACKED if packed else _lib.DG_SF_FP32,
                                    _stream(stream))
    _check(st, "dg_quantize_fp8")
    return q, sf


def quantize_fp8_cols(x: torch.Tensor, packed: bool = True, out=None, stream=None):
    """FP32 [rows, cols] (rows % 128 == 0) -> (E4M3 codes, scales) with one
    scale per 128 rows of each column, the grouping of the K-grouped GEMM's
    operands.  packed=True gives int32 [ceil(rows/512), align(cols, 4)];
    packed=False FP32 [rows/128, cols]."""
    _need(x, "x", (torch.float32,), 2)
    x = x.contiguous()
    rows, cols = x.shape
    if packed:
        sf_shape, sf_dtype = sf_packed_shape(cols, rows), torch.int32
    else:
        sf_shape, sf_dtype = (rows // 128, cols), torch.float32
    if out is None:
        q = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device=x.device)
        sf = torch.empty(sf_shape, dtype=sf_dtype, device=x.device)
    else:
        q, sf = out
        _need(q, "q", FP8_DTYPES, 2)
        _need(sf, "sf", (sf_dtype,), 2)
        if tuple(q.shape) != tuple(x.shape) or tuple(sf.shape) != tuple(sf_shape) or \
                not q.is_contiguous() or not sf.is_contiguous():
            raise ValueError("out tensors must be contiguous %s / %s" % (tuple(x.shape), sf_shape))
    _on_current_device(stream, x, q, sf)
    st = _lib.lib().dg_quantize_fp8_cols(_ptr(x), _ptr(q), _ptr(sf), rows, cols,
                                         _lib.DG_SF_UE8M0_PACKED if packed else _lib.DG_SF_FP32,
                                         _stream(stream))
    _check(st, "dg_quantize_fp8_cols")
    return q, sf


def transform_sf_into_required_layout(sf: torch.Tensor, mn: int, k: int, block_rows: int,
                                      stream=None) -> torch.Tensor:
    """FP32 scales [G?, ceil(mn/block_rows), ceil(k/128)] -> packed UE8M0
    int32 [G?, ceil(k/512), align(mn, 4)]."""
    _need(sf, "sf", (torch.float32,), sf.dim())
    grouped = sf.dim() == 3
    groups = sf.shape[0] if grouped else 1
    sf = sf.contiguous()
    out = torch.empty(sf_packed_shape(mn, k, groups if grouped else None), dtype=torch.int32,
                      device=sf.device)
    _on_current_device(stream, sf, out)
    st = _lib.lib().dg_transform_sf(_ptr(sf), _ptr(out), groups, int(mn), int(k), int(block_rows),
                                    _stream(stream))
    _check(st, "dg_transform_sf")
    return out


# Workspaces of dg_fp8_gemm_nt_ws kept by the binding, one per (device,
# stream): flag words zeroed when allocated, left zero by every launch.
_WORKSPACES = {}


def fp8_gemm_nt_workspace_size(m: int, n: int, k: int, has_c: bool = False,
                               num_sms: Optional[int] = None) -> int:
    """Bytes of workspace the stream-K form of fp8_gemm_nt needs for this
    problem (0: it would not use stream-K)."""
    out = C.c_uint64(0)
    _check(_lib.lib().dg_fp8_gemm_nt_workspace_size(int(m), int(n), int(k), 1 if has_c else 0,
                                                    int(num_sms if num_sms else get_num_sms()),
                                                    C.byref(out)), "dg_fp8_gemm_nt_workspace_size")
    return int(out.value)


# Leading bytes of a stream-K workspace that hold its flag words (dg.h).
WORKSPACE_FLAG_BYTES = 32 * 1024


def _new_workspace(nbytes: int, device) -> torch.Tensor:
    """A workspace of nbytes with its flag words zeroed (the partial-sum
    slots after them need no initialisation)."""
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    ws[:min(nbytes, WORKSPACE_FLAG_BYTES)].zero_()
    return ws


# The widest 256-row tile the stream-K form uses; the binding's own workspace
# holds a partial slot of 256 x this many floats per SM, the most any call
# can ask for, so a call needs no query to decide (dg_fp8_gemm_nt_ws plans
# with it and takes stream-K only where that is faster).
_WS_MAX_BLOCK_N = 224


def _stream_workspace(stream_handle, device) -> torch.Tensor:
    """The binding's workspace for this device and stream (its handle), of
    the largest size a stream-K launch on the current SM count can use
    (about 35 MB on 152 SMs); created with zeroed flags on first use."""
    key = (device.index, stream_handle or 0)
    ws = _WORKSPACES.get(key)
    if ws is None:
        nbytes = WORKSPACE_FLAG_BYTES + get_num_sms() * 2 * 128 * _WS_MAX_BLOCK_N * 4
        ws = _WORKSPACES[key] = _new_workspace(nbytes, device)
    return ws


def fp8_gemm_nt(a: torch.Tensor, sfa: torch.Tensor, b: torch.Tensor, sfb: torch.Tensor,
                d: Optional[torch.Tensor] = None, c: Optional[torch.Tensor] = None,
                stream=None, workspace=None) -> torch.Tensor:
    """D = C + A @ B.T with A [M,K], B [N,K] E4M3 and packed UE8M0 scales.

    workspace: None lets the call use a workspace kept by this binding (one
    buffer per device and stream; inside a CUDA-graph capture one from the
    graph's pool) for the stream-K form when that is faster; False runs
    without one (dg_fp8_gemm_nt); a uint8 CUDA tensor is used as given (its
    flag words zero before its first use, see dg_fp8_gemm_nt_ws)."""
    _need(a, "a", FP8_DTYPES, 2)
    _need(b, "b", FP8_DTYPES, 2)
    _need(sfa, "sfa", (torch.int32,), 2)
    _need(sfb, "sfb", (torch.int32,), 2)
    m, k = a.shape
    n = b.shape[0]
    if b.shape[1] != k:
        raise ValueError("K mismatch: a %s, b %s" % (tuple(a.shape), tuple(b.shape)))
    if tuple(sfa.shape) != sf_packed_shape(m, k) or tuple(sfb.shape) != sf_packed_shape(n, k):
        raise ValueError("scale shapes %s / %s, expected %s / %s" % (
            tuple(sfa.shape), tuple(sfb.shape), sf_packed_shape(m, k), sf_packed_shape(n, k)))
    if a.stride(1) != 1 or b.stride(1) != 1 or not sfa.is_contiguous() or not sfb.is_contiguous():
        raise ValueError("a and b need unit stride along K; scales must be contiguous")
    if d is None:
        d = torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    _need(d, "d", (torch.bfloat16,), 2)
    if tuple(d.shape) != (m, n) or d.stride(1) != 1:
        raise ValueError("d must be [M, N] with unit column stride")
    if c is not None:
        _need(c, "c", (torch.bfloat16,), 2)
        if tuple(c.shape) != (m, n) or c.stride(1) != 1:
            raise ValueError("c must be [M, N] with unit column stride")
    _on_current_device(stream, a, sfa, b, sfb, c, d)
    st = _stream(stream)
    ws = None
    if workspace is None:
        if torch.cuda.is_current_stream_capturing():
            # a captured call gets its own workspace from the graph's pool,
            # only when its plan uses one
            need = fp8_gemm_nt_workspace_size(m, n, k, c is not None)
            if need:
                ws = _new_workspace(need, d.device)
        else:
            ws = _stream_workspace(st.value, d.device)
    elif workspace is not False:
        _need(workspace, "workspace", (torch.uint8,), 1)
        _on_current_device(stream, workspace)
        ws = workspace
    # pointers go to ctypes as plain ints (the argtypes are void*)
    cp = c.data_ptr() if c is not None else None
    ldc = c.stride(0) if c is not None else 0
    if ws is None:
        rc = _lib.lib().dg_fp8_gemm_nt(a.data_ptr(), sfa.data_ptr(), b.data_ptr(), sfb.data_ptr(), cp,
                                       d.data_ptr(), m, n, k, a.stride(0), b.stride(0), ldc, d.stride(0), st)
        if rc:
            _check(rc, "dg_fp8_gemm_nt")
    else:
        rc = _lib.lib().dg_fp8_gemm_nt_ws(a.data_ptr(), sfa.data_ptr(), b.data_ptr(), sfb.data_ptr(), cp,
                                          d.data_ptr(), m, n, k, a.stride(0), b.stride(0), ldc, d.stride(0),
                                          ws.data_ptr(), ws.numel(), st)
        if rc:
            _check(rc, "dg_fp8_gemm_nt_ws")
    return d


def fp8_gemm_nt_fp32_sf(a: torch.Tensor, sfa: torch.Tensor, b: torch.Tensor, sfb: torch.Tensor,
                        d: Optional[torch.Tensor] = None, c: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """D = C + A @ B.T with arbitrary FP32 scales: sfa float32 [ceil(K/128),
    align(M, 4)] (one per 1x128 group of A, K-block-major), sfb float32
    [ceil(N/128), K/128] (one per 128x128 block of B)."""
    _need(a, "a", FP8_DTYPES, 2)
    _need(b, "b", FP8_DTYPES, 2)
    _need(sfa, "sfa", (torch.float32,), 2)
    _need(sfb, "sfb", (torch.float32,), 2)
    m, k = a.shape
    n = b.shape[0]
    if b.shape[1] != k:
        raise ValueError("K mismatch: a %s, b %s" % (tuple(a.shape), tuple(b.shape)))
    want_a = ((k + 127) // 128, get_tma_aligned_size(m, 4))
    want_b = ((n + 127) // 128, k // 128)
    if tuple(sfa.shape) != want_a or tuple(sfb.shape) != want_b:
        raise ValueError("scale shapes %s / %s, expected %s / %s" % (
            tuple(sfa.shape), tuple(sfb.shape), want_a, want_b))
    if a.stride(1) != 1 or b.stride(1) != 1 or not sfa.is_contiguous() or not sfb.is_contiguous():
        raise ValueError("a and b need unit stride along K; scales must be contiguous")
    if d is None:
        d = torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    _need(d, "d", (torch.bfloat16,), 2)
    if tuple(d.shape) != (m, n) or d.stride(1) != 1:
        raise ValueError("d must be [M, N] with unit column stride")
    if c is not None:
        _need(c, "c", (torch.bfloat16,), 2)
        if tuple(c.shape) != (m, n) or c.stride(1) != 1:
            raise ValueError("c must be [M, N] with unit column stride")
    _on_current_device(stream, a, sfa, b, sfb, c, d)
    st = _lib.lib().dg_fp8_gemm_nt_fp32_sf(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(c), _ptr(d),
                                           m, n, k, a.stride(0), b.stride(0),
                                           c.stride(0) if c is not None else 0, d.stride(0),
                                           _stream(stream))
    _check(st, "dg_fp8_gemm_nt_fp32_sf")
    return d


def _dense_layout(layout: str, a, sfa, b, sfb, d, c, stream):
    """Shared marshalling of fp8_gemm_{nn, tn, tt}: A is [M,K] ('n') or
    [K,M] ('t'); B is [K,N] ('n') or [N,K] ('t')."""
    _need(a, "a", FP8_DTYPES, 2)
    _need(b, "b", FP8_DTYPES, 2)
    _need(sfa, "sfa", (torch.int32,), 2)
    _need(sfb, "sfb", (torch.int32,), 2)
    a_t, b_t = layout[0] == "t", layout[1] == "t"
    k, m = a.shape if a_t else a.shape[::-1]
    n, kb = b.shape if b_t else b.shape[::-1]
    if kb != k:
        raise ValueError("K mismatch: a %s, b %s" % (tuple(a.shape), tuple(b.shape)))
    if tuple(sfa.shape) != sf_packed_shape(m, k) or tuple(sfb.shape) != sf_packed_shape(n, k):
        raise ValueError("scale shapes %s / %s, expected %s / %s" % (
            tuple(sfa.shape), tuple(sfb.shape), sf_packed_shape(m, k), sf_packed_shape(n, k)))
    if a.stride(1) != 1 or b.stride(1) != 1 or not sfa.is_contiguous() or not sfb.is_contiguous():
        raise ValueError("a and b need a unit inner stride; scales must be contiguous")
    if d is None:
        d = torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    _need(d, "d", (torch.bfloat16,), 2)
    if tuple(d.shape) != (m, n) or d.stride(1) != 1:
        raise ValueError("d must be [M, N] with unit column stride")
    if c is not None:
        _need(c, "c", (torch.bfloat16,), 2)
        if tuple(c.shape) != (m, n) or c.stride(1) != 1:
            raise ValueError("c must be [M, N] with unit column stride")
    fn = "dg_fp8_gemm_" + layout
    _on_current_device(stream, a, sfa, b, sfb, c, d)
    st = getattr(_lib.lib(), fn)(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(c), _ptr(d), m, n, k,
                                 a.stride(0), b.stride(0), c.stride(0) if c is not None else 0,
                                 d.stride(0), _stream(stream))
    _check(st, fn)
    return d


def fp8_gemm_nn(a, sfa, b, sfb, d=None, c=None, stream=None) -> torch.Tensor:
    """D = C + A @ B with A [M,K] and B [K,N] (N innermost)."""
    return _dense_layout("nn", a, sfa, b, sfb, d, c, stream)


def fp8_gemm_tn(a, sfa, b, sfb, d=None, c=None, stream=None) -> torch.Tensor:
    """D = C + A^T @ B with A stored [K,M] and B [K,N]."""
    return _dense_layout("tn", a, sfa, b, sfb, d, c, stream)


def fp8_gemm_tt(a, sfa, b, sfb, d=None, c=None, stream=None) -> torch.Tensor:
    """D = C + A^T @ B^T with A stored [K,M] and B [N,K]."""
    return _dense_layout("tt", a, sfa, b, sfb, d, c, stream)


def m_grouped_fp8_gemm_nt_contiguous(a: torch.Tensor, sfa: torch.Tensor, b: torch.Tensor,
                                     sfb: torch.Tensor, m_indices: torch.Tensor,
                                     d: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Rows of A [m_sum,K] routed to experts B [G,N,K] by m_indices (-1 = padding)."""
    _need(a, "a", FP8_DTYPES, 2)
    _need(b, "b", FP8_DTYPES, 3)
    _need(sfa, "sfa", (torch.int32,), 2)
    _need(sfb, "sfb", (torch.int32,), 3)
    _need(m_indices, "m_indices", (torch.int32,), 1)
    m_sum, k = a.shape
    g, n, kb = b.shape
    if kb != k or m_indices.numel() != m_sum:
        raise ValueError("shape mismatch")
    if tuple(sfa.shape) != sf_packed_shape(m_sum, k) or tuple(sfb.shape) != sf_packed_shape(n, k, g):
        raise ValueError("scale shapes do not match the packed layout")
    for t, name in ((a, "a"), (b, "b"), (sfa, "sfa"), (sfb, "sfb"), (m_indices, "m_indices")):
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    if d is None:
        d = torch.empty((m_sum, n), dtype=torch.bfloat16, device=a.device)
    _need(d, "d", (torch.bfloat16,), 2)
    if tuple(d.shape) != (m_sum, n) or not d.is_contiguous():
        raise ValueError("d must be contiguous [m_sum, N]")
    _on_current_device(stream, a, sfa, b, sfb, d, m_indices)
    st = _lib.lib().dg_m_grouped_fp8_gemm_nt_contiguous(
        _ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(d), _ptr(m_indices), m_sum, n, k, g,
        _stream(stream))
    _check(st, "dg_m_grouped_fp8_gemm_nt_contiguous")
    return d


def k_grouped_fp8_gemm_tn_contiguous(a: torch.Tensor, sfa: torch.Tensor, b: torch.Tensor,
                                     sfb: torch.Tensor, ks: torch.Tensor,
                                     d: Optional[torch.Tensor] = None,
                                     c: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Experts stacked along K: A [sum_k, M], B [sum_k, N] (E4M3, M / N
    innermost), ks [G] int32 on the device (rows per expert, multiples of
    128).  D[g] = C[g] + A_g^T B_g, FP32 [G, M, N]."""
    _need(a, "a", FP8_DTYPES, 2)
    _need(b, "b", FP8_DTYPES, 2)
    _need(sfa, "sfa", (torch.int32,), 2)
    _need(sfb, "sfb", (torch.int32,), 2)
    _need(ks, "ks", (torch.int32,), 1)
    sum_k, m = a.shape
    kb, n = b.shape
    g = ks.numel()
    if kb != sum_k:
        raise ValueError("shape mismatch")
    if tuple(sfa.shape) != sf_packed_shape(m, sum_k) or tuple(sfb.shape) != sf_packed_shape(n, sum_k):
        raise ValueError("scale shapes do not match the packed layout")
    for t, name in ((a, "a"), (b, "b"), (sfa, "sfa"), (sfb, "sfb"), (ks, "ks")):
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    if d is None:
        d = torch.empty((g, m, n), dtype=torch.float32, device=a.device)
    _need(d, "d", (torch.float32,), 3)
    if tuple(d.shape) != (g, m, n) or not d.is_contiguous():
        raise ValueError("d must be contiguous [G, M, N]")
    if c is not None:
        _need(c, "c", (torch.float32,), 3)
        if tuple(c.shape) != (g, m, n) or not c.is_contiguous():
            raise ValueError("c must be contiguous [G, M, N]")
    _on_current_device(stream, a, sfa, b, sfb, c, d, ks)
    st = _lib.lib().dg_k_grouped_fp8_gemm_tn_contiguous(
        _ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(c), _ptr(d), _ptr(ks), m, n, sum_k, g,
        _stream(stream))
    _check(st, "dg_k_grouped_fp8_gemm_tn_contiguous")
    return d


def m_grouped_fp8_gemm_nt_masked(a: torch.Tensor, sfa: torch.Tensor, b: torch.Tensor,
                                 sfb: torch.Tensor, masked_m: torch.Tensor, expected_m: int = 0,
                                 d: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """A [G,max_m,K] x B [G,N,K]; rows >= masked_m[g] are left untouched."""
    _need(a, "a", FP8_DTYPES, 3)
    _need(b, "b", FP8_DTYPES, 3)
    _need(sfa, "sfa", (torch.int32,), 3)
    _need(sfb, "sfb", (torch.int32,), 3)
    _need(masked_m, "masked_m", (torch.int32,), 1)
    g, max_m, k = a.shape
    gb, n, kb = b.shape
    if gb != g or kb != k or masked_m.numel() != g:
        raise ValueError("shape mismatch")
    if tuple(sfa.shape) != sf_packed_shape(max_m, k, g) or tuple(sfb.shape) != sf_packed_shape(n, k, g):
        raise ValueError("scale shapes do not match the packed layout")
    for t, name in ((a, "a"), (b, "b"), (sfa, "sfa"), (sfb, "sfb"), (masked_m, "masked_m")):
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    if d is None:
        d = torch.empty((g, max_m, n), dtype=torch.bfloat16, device=a.device)
    _need(d, "d", (torch.bfloat16,), 3)
    if tuple(d.shape) != (g, max_m, n) or not d.is_contiguous():
        raise ValueError("d must be contiguous [G, max_m, N]")
    _on_current_device(stream, a, sfa, b, sfb, d, masked_m)
    st = _lib.lib().dg_m_grouped_fp8_gemm_nt_masked(
        _ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), _ptr(d), _ptr(masked_m), g, max_m, n, k,
        int(expected_m), _stream(stream))
    _check(st, "dg_m_grouped_fp8_gemm_nt_masked")
    return d
