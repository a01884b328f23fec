"""CPU-only checks of the seeded input recipe (moe_grouped_gemm_fp8_gb300.workloads):
determinism per seed, shapes and dtypes, and the structure the grouped layouts
rely on (padding to 128 rows, -1 tags, zero padding rows, counts in range)."""
import torch

from moe_grouped_gemm_fp8_gb300 import workloads


def test_dense_is_seeded_and_shaped():
    w1 = workloads.dense(100, 136, 256, seed=7, with_c=True)
    w2 = workloads.dense(100, 136, 256, seed=7, with_c=True)
    w3 = workloads.dense(100, 136, 256, seed=8, with_c=True)
    assert w1.a.shape == (100, 256) and w1.b.shape == (136, 256) and w1.c.shape == (100, 136)
    assert w1.a.dtype == torch.float32 and w1.c.dtype == torch.bfloat16
    assert torch.equal(w1.a, w2.a) and torch.equal(w1.b, w2.b) and torch.equal(w1.c, w2.c)
    assert not torch.equal(w1.a, w3.a)
    assert workloads.dense(100, 136, 256, seed=7).c is None
    # C comes from its own stream (seed + 100): A and B do not change with it
    assert torch.equal(workloads.dense(100, 136, 256, seed=7).a, w1.a)


def test_contiguous_segments_are_padded_and_tagged():
    w = workloads.contiguous(5, 64, 128, seed=31, lo=1, hi=300)
    assert w.counts.min() >= 1 and w.counts.max() <= 300
    assert torch.equal(w.padded, (w.counts + 127) // 128 * 128)
    m_sum = int(w.padded.sum())
    assert w.a.shape == (m_sum, 128) and w.m_indices.shape == (m_sum,) and w.b.shape == (5, 64, 128)
    row = 0
    for e in range(5):
        c, p = int(w.counts[e]), int(w.padded[e])
        assert (w.m_indices[row:row + c] == e).all() and (w.m_indices[row + c:row + p] == -1).all()
        assert (w.a[row + c:row + p] == 0).all() and (w.a[row:row + c].abs().sum(1) > 0).all()
        row += p
    # every 128-row block holds one expert, then only padding
    for blk in w.m_indices.view(-1, 128):
        first = int(blk[0])
        assert first >= 0 and ((blk == first) | (blk == -1)).all()
        tail = (blk == -1).nonzero()
        if len(tail):
            assert (blk[int(tail[0]):] == -1).all()


def test_contiguous_explicit_counts_and_empty_expert():
    w = workloads.contiguous(3, 32, 128, seed=1, counts=[130, 0, 5])
    assert w.padded.tolist() == [256, 0, 128]
    assert (w.m_indices == 1).sum() == 0


def test_masked_counts_in_range():
    w = workloads.masked(16, 256, 64, 128, seed=41)
    assert w.a.shape == (16, 256, 128) and w.b.shape == (16, 64, 128)
    assert w.masked_m.dtype == torch.int32
    assert int(w.masked_m.min()) >= 0 and int(w.masked_m.max()) <= 256
    assert torch.equal(w.masked_m, workloads.masked(16, 256, 64, 128, seed=41).masked_m)


def test_k_grouped_padding_rows_are_zero():
    w = workloads.k_grouped(4, 48, 40, seed=51, lo=1, hi=300)
    assert w.ks.dtype == torch.int32 and ((w.ks % 128) == 0).all()
    assert torch.equal(w.ks.to(torch.int64), (w.counts + 127) // 128 * 128)
    row = 0
    for e in range(4):
        c, p = int(w.counts[e]), int(w.ks[e])
        assert (w.a[row + c:row + p] == 0).all() and (w.b[row + c:row + p] == 0).all()
        row += p
    assert row == w.a.shape[0] == w.b.shape[0]


def test_named_workloads_match_the_stated_configurations():
    assert [(c["m"], c["n"], c["k"]) for c in workloads.PREFILL] == \
        [(4096, n, k) for n, k in workloads.PREFILL_NK]
    assert [c["seed"] for c in workloads.PREFILL] == [1, 2, 3, 4, 5]
    assert sorted({c["m"] for c in workloads.DECODE}) == [64, 128]
    assert workloads.CONTIG == dict(num_groups=8, n=4096, k=7168, seed=31)
    assert workloads.MASKED == dict(num_groups=16, cap=256, n=7168, k=2048, seed=41)
