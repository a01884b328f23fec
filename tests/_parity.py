"""Helpers shared by the GPU parity tests: oracle-side quantisation of the
seeded inputs, upload of the oracle's codes to the device, and the tolerance
stated for the BF16 outputs.

The oracle quantises; the device receives the oracle's E4M3 codes and FP32
scales and builds its own packed scale layout with dg_transform_sf.  No value
flows from the CUDA path into the oracle.
"""
import numpy as np
import torch

import oracle
import moe_grouped_gemm_fp8_gb300 as dg

# Tolerance on the BF16 outputs over the rows the kernel writes:
# sum((d - o)^2) / sum(o^2) <= 1e-5 and max|d - o| <= 2e-2 * max|o|.
# BF16 round-to-nearest alone gives an expected relative squared error of
# about u^2 / 3 = 1.3e-6 (u = 2^-9), so the bound leaves room for the FP32
# accumulation order while catching any wrong term, sign or index.
REL_SQ_TOL = 1e-5
MAX_ABS_TOL = 2e-2

SENTINEL_BITS = 0x7F3C  # a finite BF16 pattern no GEMM result here produces


def quantize(x: torch.Tensor, block_rows: int):
    """Oracle quantisation of an FP32 [rows, cols] or [G, rows, cols] tensor.
    Returns (codes uint8, exponents int32, scales float64) with a leading
    group dim iff x has one."""
    x = x.numpy()
    if x.ndim == 2:
        return oracle.quantize(x, block_rows)
    qs, es, ss = zip(*(oracle.quantize(x[g], block_rows) for g in range(x.shape[0])))
    return np.stack(qs), np.stack(es), np.stack(ss)


def dev_codes(q: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(q)).cuda().view(torch.float8_e4m3fn)


def dev_packed_sf(s: np.ndarray, mn: int, k: int, block_rows: int) -> torch.Tensor:
    """Device packed UE8M0 scales built by the library's own transform."""
    sf = torch.from_numpy(np.ascontiguousarray(s, dtype=np.float32)).cuda()
    return dg.transform_sf_into_required_layout(sf, mn, k, block_rows)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().double().numpy()


def sentinel_like(shape, device="cuda") -> torch.Tensor:
    return torch.full(shape, SENTINEL_BITS, dtype=torch.int16, device=device).view(torch.bfloat16)


# (label, elements compared, sum((d-o)^2)/sum(o^2), max|d-o| / max|o|) of every
# comparison made with record=True; printed at the end of the session.
REPORT = []


def assert_close(d: np.ndarray, o: np.ndarray, what: str = "", record: bool = False):
    """d, o: FP64 arrays of the written rows."""
    assert d.shape == o.shape, (d.shape, o.shape)
    if o.size == 0:
        return
    assert np.isfinite(d).all(), "%s: non-finite output" % what
    err = d - o
    denom = float(np.einsum("i,i->", o.ravel(), o.ravel()))
    num = float(np.einsum("i,i->", err.ravel(), err.ravel()))
    rel = num / denom if denom > 0 else num
    mx = float(np.abs(err).max())
    omax = float(np.abs(o).max())
    lim = MAX_ABS_TOL * omax
    if record:
        REPORT.append((what, int(o.size), rel, mx / omax if omax > 0 else mx))
    assert rel <= REL_SQ_TOL, "%s: relative squared error %.3e > %.0e" % (what, rel, REL_SQ_TOL)
    assert mx <= lim, "%s: max abs error %.4g > %.4g" % (what, mx, lim)
    return rel, mx
