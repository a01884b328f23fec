"""The masked GEMM under CUDA-graph capture: the per-expert counts live on
the device only, so one captured graph serves any counts written into the
same tensor before a replay ("GEMM denso e grouped": masked grouped GEMM for
decoding with CUDA graphs, where the CPU does not know the token counts)."""
import numpy as np
import pytest
import torch

import oracle
import moe_grouped_gemm_fp8_gb300 as dg
from moe_grouped_gemm_fp8_gb300 import workloads
import _parity as P

pytestmark = pytest.mark.gpu


def test_masked_gemm_replays_with_new_counts():
    G, cap, N, K = 6, 256, 512, 512
    w = workloads.masked(G, cap, N, K, seed=61, masked_m=[0] * G)
    qa, _, sa = P.quantize(w.a, 1)
    qb, _, sb = P.quantize(w.b, 128)
    dev = (P.dev_codes(qa), P.dev_packed_sf(sa, cap, K, 1), P.dev_codes(qb), P.dev_packed_sf(sb, N, K, 128))
    mm_dev = torch.zeros(G, dtype=torch.int32, device="cuda")
    d = P.sentinel_like((G, cap, N))
    # first call outside the capture: per-device set-up happens here
    dg.m_grouped_fp8_gemm_nt_masked(*dev, mm_dev, expected_m=128, d=d)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dg.m_grouped_fp8_gemm_nt_masked(*dev, mm_dev, expected_m=128, d=d)
    for counts in ([256, 0, 17, 128, 129, 200], [1, 255, 0, 64, 256, 3]):
        d.copy_(P.sentinel_like((G, cap, N)))
        mm_dev.copy_(torch.tensor(counts, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        mm = np.array(counts, np.int32)
        o, written = oracle.gemm_masked(qa, sa, qb, sb, mm)
        bits = P.bf16_bits(d)
        wr = written.astype(bool)
        assert (bits[~wr] == P.SENTINEL_BITS).all(), counts
        P.assert_close(P.bf16_to_f64(d)[wr], o[wr], "graph replay %s" % counts)
    st, word = dg.get_device_error()
    assert st == 0, hex(word)
