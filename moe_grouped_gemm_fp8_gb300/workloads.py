"""Seeded synthetic inputs for the FP8 GEMM family.

This module holds only random-number generation and the shapes of the
workloads; it holds none of the method's arithmetic (no quantisation, no
scaling, no GEMM), so both the CUDA path and the CPU oracle can draw their
inputs from it.  Every tensor is created on the CPU from a
``torch.Generator`` seeded explicitly, in FP32 (BF16 for C).

Workload recipe (the shapes of the method's intended use: dense layers and the
two M-grouped MoE layouts of "DeepGEMM: kernels GEMM FP8 limpos e eficientes
por meio de scaling granular", section "GEMM denso e grouped"):

* dense NT small: M=128, N=256, K=512;
* dense NT prefill-like: M=4096 and (N, K) in PREFILL_NK, with and without C;
* dense NT decode-like: M in {64, 128} and the same (N, K);
* contiguous M-grouped: 8 experts, B [8, 4096, 7168]; per-expert token counts
  uniform in [256, 8192], each segment padded to a multiple of 128 rows, the
  padding rows zero in A and tagged -1 in ``m_indices``;
* masked M-grouped: 16 experts of capacity 256, B [16, 7168, 2048];
  ``masked_m`` uniform in [0, 256]; every row of A is random (rows past
  ``masked_m`` hold data the GEMM must ignore);
* K-grouped (MoE weight gradients): 8 experts, M=4096, N=7168; per-expert
  token counts uniform in [256, 8192], each padded to a multiple of 128 rows
  along K, the padding rows zero in both operands.

A, B and C entries are N(0, 1).
"""
from dataclasses import dataclass
from typing import Optional

import torch

PREFILL_NK = [(2112, 7168), (24576, 1536), (7168, 16384), (4096, 7168), (7168, 2048)]
DECODE_M = (64, 128)
CONTIG_ALIGN = 128  # segment alignment of the contiguous layout (M block size)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


@dataclass
class Dense:
    a: torch.Tensor           # [M, K] float32
    b: torch.Tensor           # [N, K] float32
    c: Optional[torch.Tensor]  # [M, N] bfloat16 or None


def dense(m: int, n: int, k: int, seed: int, with_c: bool = False) -> Dense:
    g = _gen(seed)
    a = torch.randn(m, k, generator=g, dtype=torch.float32)
    b = torch.randn(n, k, generator=g, dtype=torch.float32)
    c = None
    if with_c:
        gc = _gen(seed + 100)
        c = torch.randn(m, n, generator=gc, dtype=torch.float32).to(torch.bfloat16)
    return Dense(a, b, c)


@dataclass
class Contiguous:
    a: torch.Tensor          # [m_sum, K] float32, padding rows zero
    b: torch.Tensor          # [G, N, K] float32
    m_indices: torch.Tensor  # [m_sum] int32, -1 on padding rows
    counts: torch.Tensor     # [G] int64 real rows per expert
    padded: torch.Tensor     # [G] int64 rows per expert incl. padding


def contiguous(num_groups: int, n: int, k: int, seed: int, lo: int = 256, hi: int = 8192,
               align: int = CONTIG_ALIGN, counts: Optional[list] = None) -> Contiguous:
    """Expert segments in ascending expert order, each padded to ``align``."""
    g = _gen(seed)
    if counts is None:
        cnt = torch.randint(lo, hi + 1, (num_groups,), generator=g, dtype=torch.int64)
    else:
        cnt = torch.tensor(counts, dtype=torch.int64)
    padded = (cnt + align - 1) // align * align
    m_sum = int(padded.sum())
    a = torch.zeros(m_sum, k, dtype=torch.float32)
    m_indices = torch.full((m_sum,), -1, dtype=torch.int32)
    row = 0
    for e in range(num_groups):
        c_e, p_e = int(cnt[e]), int(padded[e])
        if c_e:
            a[row:row + c_e] = torch.randn(c_e, k, generator=g, dtype=torch.float32)
            m_indices[row:row + c_e] = e
        row += p_e
    b = torch.randn(num_groups, n, k, generator=g, dtype=torch.float32)
    return Contiguous(a, b, m_indices, cnt, padded)


@dataclass
class Masked:
    a: torch.Tensor         # [G, cap, K] float32 (all rows random)
    b: torch.Tensor         # [G, N, K] float32
    masked_m: torch.Tensor  # [G] int32


def masked(num_groups: int, cap: int, n: int, k: int, seed: int,
           masked_m: Optional[list] = None) -> Masked:
    g = _gen(seed)
    if masked_m is None:
        mm = torch.randint(0, cap + 1, (num_groups,), generator=g, dtype=torch.int64).to(torch.int32)
    else:
        mm = torch.tensor(masked_m, dtype=torch.int32)
    a = torch.randn(num_groups, cap, k, generator=g, dtype=torch.float32)
    b = torch.randn(num_groups, n, k, generator=g, dtype=torch.float32)
    return Masked(a, b, mm)


@dataclass
class KGrouped:
    a: torch.Tensor   # [sum_k, M] float32 (experts stacked along K), padding rows zero
    b: torch.Tensor   # [sum_k, N] float32, padding rows zero
    ks: torch.Tensor  # [G] int32 rows per expert incl. padding (multiples of 128)
    counts: torch.Tensor  # [G] int64 real rows per expert


def k_grouped(num_groups: int, m: int, n: int, seed: int, lo: int = 256, hi: int = 8192,
              align: int = CONTIG_ALIGN, counts: Optional[list] = None) -> KGrouped:
    g = _gen(seed)
    if counts is None:
        cnt = torch.randint(lo, hi + 1, (num_groups,), generator=g, dtype=torch.int64)
    else:
        cnt = torch.tensor(counts, dtype=torch.int64)
    padded = (cnt + align - 1) // align * align
    sum_k = int(padded.sum())
    a = torch.zeros(sum_k, m, dtype=torch.float32)
    b = torch.zeros(sum_k, n, dtype=torch.float32)
    row = 0
    for e in range(num_groups):
        c_e = int(cnt[e])
        if c_e:
            a[row:row + c_e] = torch.randn(c_e, m, generator=g, dtype=torch.float32)
            b[row:row + c_e] = torch.randn(c_e, n, generator=g, dtype=torch.float32)
        row += int(padded[e])
    return KGrouped(a, b, padded.to(torch.int32), cnt)


# Named workloads with their seeds (one seed per shape, C drawn from seed+100).
SMALL = dict(m=128, n=256, k=512, seed=0)
PREFILL = [dict(m=4096, n=n, k=k, seed=1 + i) for i, (n, k) in enumerate(PREFILL_NK)]
DECODE = [dict(m=m, n=n, k=k, seed=(11 if m == 64 else 21) + i)
          for m in DECODE_M for i, (n, k) in enumerate(PREFILL_NK)]
CONTIG = dict(num_groups=8, n=4096, k=7168, seed=31)
MASKED = dict(num_groups=16, cap=256, n=7168, k=2048, seed=41)
KGROUPED = dict(num_groups=8, m=4096, n=7168, seed=51)
