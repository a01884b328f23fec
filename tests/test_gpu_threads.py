"""Several host threads using the library at once, each on its own CUDA
stream: the per-device caches (error word, occupancy counts, shared-memory
attributes) are shared, and every result must equal bit for bit the same
call made alone."""
import threading

import pytest
import torch

import moe_grouped_gemm_fp8_gb300 as dg
from moe_grouped_gemm_fp8_gb300 import workloads

# shapes the tile chooser sends to different kernels (dg.plan_fp8_gemm_nt):
# split-K 4 with 64-row A slots, split-K 2, 128 x 224 tiles, a 128 x 256
# single-accumulator tile and 256 x 192 tiles
SHAPES = [(64, 1024, 4096), (1024, 1024, 1024), (1024, 4096, 1024), (1536, 3072, 1024),
          (1536, 4096, 4096)]


@pytest.mark.gpu
def test_concurrent_host_threads_on_separate_streams():
    cases = []
    for i, (m, n, k) in enumerate(SHAPES):
        w = workloads.dense(m, n, k, seed=60 + i, with_c=True)
        qa, sfa = dg.quantize_fp8(w.a.cuda(), 1)
        qb, sfb = dg.quantize_fp8(w.b.cuda(), 128)
        c = w.c.cuda()
        want = dg.fp8_gemm_nt(qa, sfa, qb, sfb, c=c)
        cases.append((qa, sfa, qb, sfb, c, want))
    torch.cuda.synchronize()

    errors = []

    def worker(t):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for it in range(6):
                    qa, sfa, qb, sfb, c, want = cases[(t + it) % len(cases)]
                    got = dg.fp8_gemm_nt(qa, sfa, qb, sfb, c=c)
                    stream.synchronize()
                    if not torch.equal(got.view(torch.int16), want.view(torch.int16)):
                        errors.append("thread %d iteration %d differs" % (t, it))
        except Exception as e:  # reported below, on the test's thread
            errors.append("thread %d: %r" % (t, e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    st, word = dg.get_device_error()
    assert st == 0, "device error word 0x%x" % word
