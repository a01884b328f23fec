#!/usr/bin/env python
"""Throughput of the FP8 fine-grained-scaled GEMM path on GB300.

Headline workload (one step): the dense NT prefill-like shapes, M=4096 and
(N, K) in {(2112,7168), (24576,1536), (7168,16384), (4096,7168), (7168,2048)}.
Per shape a step quantises the FP32 activations A (1x128 groups, packed UE8M0
scales) and runs D = A @ B.T and D2 = C + A @ B.T.  The weights B are
quantised (128x128 blocks) once at setup.  Inputs are seeded N(0, 1); the
per-step working set (~2 GB) is larger than L2.  `value` is the step's GEMM
FLOPs over the device time of exactly --steps steps.

The same run then measures, GEMM only, the four other workloads of the benchmark spec
(dense small, dense decode-like, contiguous MoE, masked MoE) and reports each
under "configs" with its own roofline and CPU-oracle baseline; a sustained
prefill figure over >= 1.5 s of back-to-back steps is reported beside the
headline, and the clocks are sampled over the whole measured window.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle
instead, on a bounded row sample of the headline workload.  `--workload X`
measures one other workload alone and prints its own line.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "FP8 TFLOPS (and % of GB300 FP8 peak / HBM roofline) per shape at 1 GPU"
FP8_OVER_BF16 = 2.0  # nominal dense FP8 : BF16 tensor throughput (4.5 : 2.25 PFLOP/s)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
OTHER_CONFIGS = ("small", "decode", "contiguous", "masked")
SUSTAINED_SECONDS = 1.5


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="prefill",
                   choices=["prefill", "decode", "contiguous", "masked", "kgrouped", "fp32scales", "small"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-configs", action="store_true",
                   help="headline workload only (no per-config entries)")
    p.add_argument("--pdl", action="store_true",
                   help="launch the library's kernels with programmatic dependent launch")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--profile-steps", type=int, default=0,
                   help="run this many untimed steps and exit (for an external profiler)")
    p.add_argument("--shape", type=int, default=-1,
                   help="restrict the run to this shape index (profiling of one shape)")
    return p.parse_args()


# --------------------------------------------------------------------------- ranks


class Ranks:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")  # timing barrier / max only, no data-path traffic
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------- clocks


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [line.strip().split(", ") for line in self.file if line.strip()]
        self.file.close()
        os.unlink(self.file.name)
        return summarise_clocks(rows)


def summarise_clocks(rows):
    """Median SM clock over the samples taken under load (power above half of
    the largest draw seen), the max clock and the throttle reasons seen."""
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    samples = []
    for r in rows:
        if len(r) < 9:
            continue
        try:
            samples.append((float(r[1]), float(r[2]), float(r[3]),
                            [n for n, v in zip(names, r[5:9]) if v.strip().lower() == "active"]))
        except ValueError:
            continue
    if not samples:
        return None
    pmax = max(s[2] for s in samples)
    loaded = [s for s in samples if s[2] >= 0.5 * pmax] or samples
    reasons = sorted({n for s in loaded for n in s[3]})
    return {"sm_mhz": statistics.median(s[0] for s in loaded), "sm_max_mhz": max(s[1] for s in samples),
            "samples": len(samples), "samples_under_load": len(loaded),
            "power_w_max": pmax, "reasons": reasons}


# --------------------------------------------------------------------------- byte counts


def algorithmic_bytes_gemm(m, n, k, with_c):
    """Bytes a dense NT GEMM must move: A, B, their packed UE8M0 scale words
    (one 32-bit word per row per 4 K blocks), D, and C when present."""
    kb = k // 128
    return (m * k + n * k + m * ((kb + 3) // 4) * 4 + n * ((kb + 3) // 4) * 4 + 2 * m * n +
            (2 * m * n if with_c else 0))


def algorithmic_bytes_contiguous(valid_rows, groups, n, k):
    """Valid rows of A and D, every expert's B, and the scale words."""
    kp = (k // 128 + 3) // 4
    return valid_rows * k + groups * n * k + 2 * valid_rows * n + 4 * kp * (valid_rows + groups * n)


def algorithmic_bytes_masked(valid_rows, used_groups, n, k):
    """Valid rows of A and D, B of the experts with at least one row, and the
    scale words."""
    kp = (k // 128 + 3) // 4
    return valid_rows * k + used_groups * n * k + 2 * valid_rows * n + 4 * kp * (valid_rows + used_groups * n)


# --------------------------------------------------------------------------- headline workload


def prefill_setup(dg, workloads, dev, only=-1):
    shapes = []
    for i, cfg in enumerate(workloads.PREFILL):
        if only >= 0 and i != only:
            continue
        m, n, k = cfg["m"], cfg["n"], cfg["k"]
        w = workloads.dense(m, n, k, cfg["seed"], with_c=True)
        a = w.a.to(dev)
        qb, sfb = dg.quantize_fp8(w.b.to(dev), 128)
        qa = torch.empty(m, k, dtype=torch.float8_e4m3fn, device=dev)
        sfa = torch.empty(dg.sf_packed_shape(m, k), dtype=torch.int32, device=dev)
        shapes.append(dict(m=m, n=n, k=k, a=a, qa=qa, sfa=sfa, qb=qb, sfb=sfb, c=w.c.to(dev),
                           d=torch.empty(m, n, dtype=torch.bfloat16, device=dev),
                           d2=torch.empty(m, n, dtype=torch.bfloat16, device=dev),
                           host=w))
    return shapes


def prefill_step(dg, shapes, events=None):
    """One step; if `events` is a list, appends (start, end, flops) per GEMM."""
    for s in shapes:
        dg.quantize_fp8(s["a"], 1, out=(s["qa"], s["sfa"]))
        for c, d in ((None, s["d"]), (s["c"], s["d2"])):
            if events is not None:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
            dg.fp8_gemm_nt(s["qa"], s["sfa"], s["qb"], s["sfb"], d=d, c=c)
            if events is not None:
                e1.record()
                events.append((e0, e1, 2.0 * s["m"] * s["n"] * s["k"], s))


def step_flops(shapes):
    return sum(2 * 2.0 * s["m"] * s["n"] * s["k"] for s in shapes)


# DRAM bytes (read + write) of one launch of the step's largest GEMM, from an
# ncu capture of that launch, keyed by the shape and the tile configuration
# the library chose for it at capture time: (m, n, k, with C, block_m,
# block_n, split_k, cta_pair, multicast).  A launch whose configuration is not
# listed has no traffic figure (the counters would be stale).
CAPTURED_TRAFFIC = {
    # 256 x 192 tiles, eight epilogue warps, 2048-row raster band, one CTA per
    # tile: 367.5 MB read + 47.3 MB written
    (4096, 7168, 16384, False, 256, 192, 1, 0, 0): 367509760 + 47258112,
    # the same tiles in clusters of two sharing B by TMA multicast:
    # 393.4 MB read + 47.9 MB written
    (4096, 7168, 16384, False, 256, 192, 1, 0, 1): 393375232 + 47889408,
}


def captured_traffic(dg, m, n, k, with_c, num_sms):
    plan = dg.plan_fp8_gemm_nt_ws(m, n, k, has_c=with_c, num_sms=num_sms)
    key = (m, n, k, bool(with_c), plan["block_m"], plan["block_n"], plan["split_k"], int(plan["cta_pair"]),
           int(plan["multicast"]))
    return CAPTURED_TRAFFIC.get(key), plan


def prefill_roofline(res, fp8_peak, peak_source, traffic=None, plan=None):
    """Roofline of the dominant kernel: the D = A @ B.T launch (no C) with the
    largest share of the step (per-launch CUDA-event times of the timed
    region; its D = C + A @ B.T twin runs the same kernel), plus the same
    figure over every GEMM launch of the step."""
    dom = dominant_launch(res["per_shape"])
    r = {"bound": "tensor", "achieved": dom["tflops"], "peak": fp8_peak, "unit": "TFLOP/s",
         "frac": dom["tflops"] / fp8_peak, "traffic": traffic,
         "traffic_unit": "bytes per launch (dram read + write)",
         "kernel": "fp8_gemm_kernel, D%s = A@B.T, M=%d N=%d K=%d (largest GEMM of the step)" %
                   (" = C +" if dom["c"] else "", dom["m"], dom["n"], dom["k"]),
         "all_gemms": {"achieved": res["achieved"], "frac": res["achieved"] / fp8_peak},
         "peak_source": peak_source}
    if plan is not None:
        r["tile"] = plan
    return r


def dominant_launch(per_shape):
    return max((e for e in per_shape if not e["c"]), key=lambda e: e["us"])


def run_prefill(args, ranks, dg, workloads, dev, clocks):
    dg.set_pdl(bool(args.pdl))
    shapes = prefill_setup(dg, workloads, dev, args.shape)
    if args.profile_steps:
        for _ in range(args.profile_steps):
            prefill_step(dg, shapes)
        torch.cuda.synchronize()
        return None
    t_warm = time.perf_counter()
    while True:
        for _ in range(max(3, args.warmup)):
            prefill_step(dg, shapes)
        torch.cuda.synchronize()
        if time.perf_counter() - t_warm > 0.5:
            break
    st, word = dg.get_device_error()
    if st != 0:
        raise RuntimeError("device error after warm-up: 0x%x" % word)

    # device-timed region: exactly --steps steps, inputs resident in HBM
    events = []
    ranks.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        prefill_step(dg, shapes, events)
    t1.record()
    torch.cuda.synchronize()
    ranks.barrier()
    ms = t0.elapsed_time(t1) / args.steps
    ms_max = ranks.max(ms)
    flops_step = step_flops(shapes)
    value = ranks.sum(flops_step) / (ms_max * 1e-3) / 1e12

    gemm_ms = [e0.elapsed_time(e1) for e0, e1, _, _ in events]
    gemm_flops = [f for _, _, f, _ in events]
    achieved = sum(gemm_flops) / (sum(gemm_ms) * 1e-3) / 1e12
    per_shape = []
    for i, s in enumerate(shapes):
        for j, with_c in enumerate((False, True)):
            ts = [gemm_ms[q] for q in range(2 * i + j, len(events), 2 * len(shapes))]
            t = statistics.median(ts)
            f = 2.0 * s["m"] * s["n"] * s["k"]
            byt = algorithmic_bytes_gemm(s["m"], s["n"], s["k"], with_c)
            per_shape.append({"m": s["m"], "n": s["n"], "k": s["k"], "c": with_c, "us": t * 1e3,
                              "tflops": f / (t * 1e-3) / 1e12, "gbs": byt / (t * 1e-3) / 1e9})

    # sustained: the same step back to back for >= SUSTAINED_SECONDS (clocks
    # settle under the power cap; the short headline region cannot show that)
    n_sus = max(args.steps, int(math.ceil(SUSTAINED_SECONDS / max(ms * 1e-3, 1e-6))))
    ranks.barrier()
    torch.cuda.synchronize()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(n_sus):
        prefill_step(dg, shapes)
    s1.record()
    torch.cuda.synchronize()
    ms_sus = ranks.max(s0.elapsed_time(s1) / n_sus)
    sustained = {"value": ranks.sum(flops_step) / (ms_sus * 1e-3) / 1e12, "unit": "TFLOPS",
                 "steps": n_sus, "ms_per_step": ms_sus, "seconds": ms_sus * n_sus * 1e-3}

    st, word = dg.get_device_error()
    if st != 0:
        raise RuntimeError("device error in timed region: 0x%x" % word)

    e2e = None
    if not args.no_e2e:
        e2e = run_prefill_e2e(args, ranks, dg, shapes, dev)
    ws = sum(s["a"].numel() * 4 + s["qa"].numel() + s["qb"].numel() + 3 * 2 * s["m"] * s["n"] for s in shapes)
    res = dict(value=value, ms=ms_max, achieved=achieved, per_shape=per_shape, e2e=e2e,
               sustained=sustained, launches=args.steps * len(shapes) * 3, flops_step=flops_step,
               working_set_gb=ws / 1e9)
    del shapes
    torch.cuda.empty_cache()
    return res


def run_prefill_e2e(args, ranks, dg, shapes, dev):
    host = []
    h2d = d2h = 0
    for s in shapes:
        hb = {"a": s["host"].a.pin_memory(), "c": s["host"].c.pin_memory(),
              "qb": s["qb"].cpu().pin_memory(), "sfb": s["sfb"].cpu().pin_memory(),
              "d": torch.empty(s["m"], s["n"], dtype=torch.bfloat16).pin_memory(),
              "d2": torch.empty(s["m"], s["n"], dtype=torch.bfloat16).pin_memory()}
        dv = {k: torch.empty_like(v, device=dev) for k, v in hb.items() if k in ("a", "c", "qb", "sfb")}
        host.append((hb, dv))
        h2d += sum(hb[k].numel() * hb[k].element_size() for k in ("a", "c", "qb", "sfb"))
        d2h += 2 * s["m"] * s["n"] * 2

    # Three streams: the host-to-device copies of shape i+1 and the
    # device-to-host copies of shape i-1 run while shape i computes.  Events
    # order every reuse of a device buffer across steps (a copy into an input
    # waits for the previous step's kernels that read it; a GEMM writing D
    # waits for the previous step's copy of D to the host).
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    n_sh = len(shapes)
    used = [None] * n_sh     # compute done with shape i's inputs (previous step)
    drained = [None] * n_sh  # D of shape i copied to the host (previous step)

    def step():
        for i, (s, (hb, dv)) in enumerate(zip(shapes, host)):
            with torch.cuda.stream(s_in):
                if used[i] is not None:
                    s_in.wait_event(used[i])
                for k in ("a", "c", "qb", "sfb"):
                    dv[k].copy_(hb[k], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            comp.wait_event(ready)
            if drained[i] is not None:
                comp.wait_event(drained[i])
            dg.quantize_fp8(dv["a"], 1, out=(s["qa"], s["sfa"]))
            dg.fp8_gemm_nt(s["qa"], s["sfa"], dv["qb"], dv["sfb"], d=s["d"])
            dg.fp8_gemm_nt(s["qa"], s["sfa"], dv["qb"], dv["sfb"], d=s["d2"], c=dv["c"])
            done = torch.cuda.Event()
            done.record(comp)
            used[i] = done
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                hb["d"].copy_(s["d"], non_blocking=True)
                hb["d2"].copy_(s["d2"], non_blocking=True)
                out = torch.cuda.Event()
                out.record(s_out)
            drained[i] = out

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    ranks.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    dt = ranks.max((time.perf_counter() - t0) / args.steps)
    return {"value": ranks.sum(step_flops(shapes)) / dt / 1e12, "unit": "TFLOPS",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3}


# --------------------------------------------------------------------------- CPU oracle timing


def calibrate(run, probe, seconds, limit):
    """Sample size (rows) that keeps one call of run(size) near `seconds` of
    wall time on this host: time run(probe), then scale linearly (at most
    `limit`)."""
    t0 = time.perf_counter()
    run(probe)
    dt = max(time.perf_counter() - t0, 1e-3)
    return int(min(limit, max(probe, probe * seconds / dt)))


def timed_baseline(run, size, what):
    import oracle
    t0 = time.perf_counter()
    flops = run(size)
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOPS", "cores": oracle.get_threads(), "kind": "oracle",
            "sample": what % size + ", FP64, %.1f s" % dt}


def oracle_sample(workloads, rows_per_shape, seed=0):
    """Bounded sample of the prefill workload for the CPU oracle: per shape,
    `rows_per_shape` randomly chosen rows of A (quantised 1x128 by the oracle)
    against the oracle-quantised B, computing D and D2 = C + D for those rows.
    `take(items, r)` keeps the first r of them (still a random subset)."""
    import oracle
    rng = np.random.default_rng(seed)
    items = []
    for cfg in workloads.PREFILL:
        m, n, k = cfg["m"], cfg["n"], cfg["k"]
        w = workloads.dense(m, n, k, cfg["seed"], with_c=True)
        qb, _, sb = oracle.quantize(w.b.numpy(), 128)
        rows = rng.choice(m, size=min(m, rows_per_shape), replace=False)
        a_rows = np.ascontiguousarray(w.a.numpy()[rows])
        c_rows = np.ascontiguousarray(w.c[torch.from_numpy(rows)].view(torch.int16).numpy().view(np.uint16))
        items.append(dict(n=n, k=k, a=a_rows, c=c_rows, qb=qb, sb=sb))
    return items


def take(items, rows):
    return [dict(it, a=np.ascontiguousarray(it["a"][:rows]), c=np.ascontiguousarray(it["c"][:rows]))
            for it in items]


def oracle_run(items):
    import oracle
    flops = 0.0
    for it in items:
        qa, _, sa = oracle.quantize(it["a"], 1)
        idx = np.arange(qa.shape[0], dtype=np.int64)
        oracle.gemm_nt_rows(qa, sa, it["qb"], it["sb"], idx)
        oracle.gemm_nt_rows(qa, sa, it["qb"], it["sb"], idx, it["c"])
        flops += 2 * 2.0 * qa.shape[0] * it["qb"].shape[0] * it["k"]
    return flops


def calibrated_rows(items, seconds, probe_rows=16):
    return calibrate(lambda r: oracle_run(take(items, r)), probe_rows, seconds, len(items[0]["a"]))


def cpu_baseline(workloads, seconds=8.0):
    items = oracle_sample(workloads, 2048)
    rows = calibrated_rows(items, seconds)
    return timed_baseline(lambda r: oracle_run(take(items, r)), rows,
                          "%d random rows of A per prefill shape (quantise + D and C + D rows)")


def cpu_baseline_config(name, workloads, seconds=3.0):
    """The oracle on a bounded sample of one of the other workloads: the rows
    of A quantised by the oracle and their output rows computed against the
    oracle-quantised B (B is quantised once, outside the timed part, as the
    GPU side's weights are)."""
    import oracle
    rng = np.random.default_rng(1)
    if name == "small":
        cfg = workloads.SMALL
        w = workloads.dense(cfg["m"], cfg["n"], cfg["k"], cfg["seed"])
        a, b = w.a.numpy(), w.b.numpy()

        def run(reps):
            f = 0.0
            for _ in range(reps):
                qa, _, sa = oracle.quantize(a, 1)
                qb, _, sb = oracle.quantize(b, 128)
                oracle.gemm_nt(qa, sa, qb, sb)
                f += 2.0 * cfg["m"] * cfg["n"] * cfg["k"]
            return f
        reps = calibrate(run, 2, seconds, 100000)
        return timed_baseline(run, reps, "%d repetitions of the whole workload (quantise A and B + GEMM)")
    if name == "decode":
        items = []
        for cfg in workloads.DECODE:
            w = workloads.dense(cfg["m"], cfg["n"], cfg["k"], cfg["seed"])
            qb, _, sb = oracle.quantize(w.b.numpy(), 128)
            rows = rng.choice(cfg["m"], size=cfg["m"], replace=False)
            items.append(dict(a=np.ascontiguousarray(w.a.numpy()[rows]), qb=qb, sb=sb, k=cfg["k"]))

        def run(r):
            f = 0.0
            for it in items:
                qa, _, sa = oracle.quantize(it["a"][:r], 1)
                oracle.gemm_nt_rows(qa, sa, it["qb"], it["sb"], np.arange(qa.shape[0], dtype=np.int64))
                f += 2.0 * qa.shape[0] * it["qb"].shape[0] * it["k"]
            return f
        r = calibrate(run, 1, seconds, 64)
        return timed_baseline(run, r, "%d random rows of A per decode shape (quantise + D rows)")
    if name == "contiguous":
        cfg = workloads.CONTIG
        w = workloads.contiguous(cfg["num_groups"], cfg["n"], cfg["k"], cfg["seed"])
        G, n, k = cfg["num_groups"], cfg["n"], cfg["k"]
        qbs = [oracle.quantize(w.b[g].numpy(), 128) for g in range(G)]
        qb, sb = np.stack([x[0] for x in qbs]), np.stack([x[2] for x in qbs])
        mi = w.m_indices.numpy()
        per = [rng.permutation(np.nonzero(mi == g)[0]) for g in range(G)]
        a = w.a.numpy()

        def run(r):
            rows = np.concatenate([p[:r] for p in per])
            qa, _, sa = oracle.quantize(np.ascontiguousarray(a[rows]), 1)
            oracle.gemm_contiguous(qa, sa, qb, sb, mi[rows])
            return 2.0 * rows.size * n * k
        r = calibrate(run, 1, seconds, min(p.size for p in per))
        return timed_baseline(run, r, "%d random valid rows of A per expert (quantise + D rows)")
    if name == "masked":
        cfg = workloads.MASKED
        G, cap, n, k = cfg["num_groups"], cfg["cap"], cfg["n"], cfg["k"]
        w = workloads.masked(G, cap, n, k, cfg["seed"])
        qbs = [oracle.quantize(w.b[g].numpy(), 128) for g in range(G)]
        qb, sb = np.stack([x[0] for x in qbs]), np.stack([x[2] for x in qbs])
        mm = w.masked_m.numpy()
        a = w.a.numpy()

        def run(r):
            take_m = np.minimum(mm, r).astype(np.int32)
            qa = np.zeros((G, r, k), dtype=np.uint8)
            sa = np.ones((G, r, k // 128))
            for g in range(G):
                if take_m[g]:
                    q, _, s = oracle.quantize(np.ascontiguousarray(a[g, :take_m[g]]), 1)
                    qa[g, :take_m[g]], sa[g, :take_m[g]] = q, s
            oracle.gemm_masked(qa, sa, qb, sb, take_m)
            return 2.0 * float(take_m.sum()) * n * k
        r = calibrate(run, 1, seconds, cap)
        return timed_baseline(run, r, "the first min(masked_m, %d) rows of A per expert (quantise + D rows)")
    raise ValueError(name)


def run_reference(args, ranks):
    from moe_grouped_gemm_fp8_gb300 import workloads
    import oracle
    if ranks.rank != 0:
        return 0
    items = oracle_sample(workloads, 2048)
    rows = calibrated_rows(items, 0.5)
    items = take(items, rows)
    for _ in range(args.warmup):
        oracle_run(items)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        flops += oracle_run(items)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = "%d rows of A per prefill shape per step (quantise + D and C + D rows), FP64" % rows
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "dense NT prefill-like M=4096, (N,K) in %s, with and without C; CPU oracle row sample" %
                   workloads.PREFILL_NK},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": oracle.get_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- other workloads


def _flush_l2(buf):
    # reads more bytes than L2 holds; a read leaves clean lines, so the timed
    # launch does not pay for writing back the flush's own data
    torch.sum(buf, dtype=torch.float32)


def _time_gemm(fn, iters, flush):
    """Median device time (ms) of fn() over iters launches, L2 flushed before each."""
    ts = []
    for _ in range(iters):
        _flush_l2(flush)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


L2_BYTES = 129 * 1024 * 1024


def _copies_for(nbytes: int) -> int:
    """How many copies of a launch's inputs to rotate through so that, between
    two uses of one copy, the others stream well over twice L2's capacity."""
    return int(min(64, max(3, math.ceil(2.5 * L2_BYTES / max(nbytes, 1)) + 1)))


def _time_graph(fns, replays):
    """Per-launch device time (ms): the launches in fns (one per input copy)
    are captured back to back in one CUDA graph; each replay is timed with
    events on the capturing stream and the median replay time is divided by
    the number of launches."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for f in fns:
            f()
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(replays):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / len(fns))
    return statistics.median(ts)


_FLOOR_LIB = None


def _floor_lib():
    """libdg_floor.so (built by build_floor()): the streaming-read kernel."""
    global _FLOOR_LIB
    if _FLOOR_LIB is None:
        import ctypes
        from moe_grouped_gemm_fp8_gb300 import build as dg_build
        lib = ctypes.CDLL(dg_build.build_floor())
        lib.dg_hbm_read_floor.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int,
                                          ctypes.c_void_p]
        lib.dg_hbm_read_floor.restype = ctypes.c_int
        _FLOOR_LIB = lib
    return _FLOOR_LIB


def _stream_floor_us(nbytes, dev, replays):
    """Per-launch device time (us) of a plain streaming read of nbytes (a
    hand-written kernel: 4 CTAs of 512 threads per SM, eight 16-byte
    non-caching loads in flight per thread), timed like the GEMMs: one launch
    per buffer copy, copies totalling > 2.5x L2, in one CUDA graph.  The
    per-launch floor of any kernel that reads that many bytes from HBM once
    (launch gap, ramp-up and drain included), reported next to the
    memory-bound GEMMs."""
    lib = _floor_lib()
    grid = 4 * torch.cuda.get_device_properties(dev).multi_processor_count
    n = max(16, (nbytes + 15) // 16 * 16)
    bufs = [torch.ones(n // 4, dtype=torch.int32, device=dev) for _ in range(_copies_for(nbytes))]
    sink = torch.zeros(1, dtype=torch.int32, device=dev)

    def read(b):
        rc = lib.dg_hbm_read_floor(b.data_ptr(), n, sink.data_ptr(), grid, torch.cuda.current_stream(dev).cuda_stream)
        if rc != 0:
            raise RuntimeError("streaming-read floor kernel: CUDA error %d" % rc)

    fns = [(lambda b=b: read(b)) for b in bufs]
    for f in fns:
        f()
    t = _time_graph(fns, replays)
    del bufs, fns
    return t * 1e3


def build_cases(name, dg, workloads, dev):
    """GEMM-only launch closures of one workload.  Each case owns enough
    copies of its inputs and outputs that the copies together exceed L2
    several times over (B of the decode shapes alone would fit)."""
    cases = []

    def rotate(tensors, nbytes):
        r = _copies_for(nbytes)
        return [tensors] + [tuple(t.clone() for t in tensors) for _ in range(r - 1)]

    if name in ("decode", "small"):
        cfgs = workloads.DECODE if name == "decode" else [workloads.SMALL]
        for cfg in cfgs:
            m, n, k = cfg["m"], cfg["n"], cfg["k"]
            w = workloads.dense(m, n, k, cfg["seed"])
            qa, sfa = dg.quantize_fp8(w.a.to(dev), 1)
            qb, sfb = dg.quantize_fp8(w.b.to(dev), 128)
            d = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
            byt = algorithmic_bytes_gemm(m, n, k, False)
            fns = [(lambda t=t: dg.fp8_gemm_nt(t[0], t[1], t[2], t[3], d=t[4]))
                   for t in rotate((qa, sfa, qb, sfb, d), byt)]
            cases.append(dict(name="dense m=%d n=%d k=%d" % (m, n, k), fns=fns, flops=2.0 * m * n * k,
                              bytes=byt, shape=(m, n, k)))
    elif name == "contiguous":
        cfg = workloads.CONTIG
        w = workloads.contiguous(cfg["num_groups"], cfg["n"], cfg["k"], cfg["seed"])
        qa, sfa = dg.quantize_fp8(w.a.to(dev), 1)
        qb, sfb = dg.quantize_fp8(w.b.to(dev), 128)
        mi = w.m_indices.to(dev)
        d = torch.empty(w.a.shape[0], cfg["n"], dtype=torch.bfloat16, device=dev)
        valid = int(w.counts.sum())
        n, k, G = cfg["n"], cfg["k"], cfg["num_groups"]
        byt = algorithmic_bytes_contiguous(valid, G, n, k)
        fns = [(lambda t=t: dg.m_grouped_fp8_gemm_nt_contiguous(t[0], t[1], t[2], t[3], t[4], d=t[5]))
               for t in rotate((qa, sfa, qb, sfb, mi, d), byt)]
        cases.append(dict(name="contiguous G=%d valid_rows=%d padded_rows=%d n=%d k=%d" %
                          (G, valid, w.a.shape[0], n, k), fns=fns, flops=2.0 * valid * n * k, bytes=byt))
    elif name == "fp32scales":
        # the prefill shapes through the FP32-scale (promotion) kernel; the
        # scales are the quantiser's (powers of two), passed as FP32
        for cfg in workloads.PREFILL:
            m, n, k = cfg["m"], cfg["n"], cfg["k"]
            w = workloads.dense(m, n, k, cfg["seed"])
            qa, sa = dg.quantize_fp8(w.a.to(dev), 1, packed=False)
            qb, sb = dg.quantize_fp8(w.b.to(dev), 128, packed=False)
            fa = torch.zeros(k // 128, dg.get_tma_aligned_size(m, 4), dtype=torch.float32, device=dev)
            fa[:, :m] = sa.t()
            fb = sb.contiguous()
            d = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
            byt = algorithmic_bytes_gemm(m, n, k, False)
            fns = [(lambda t=t: dg.fp8_gemm_nt_fp32_sf(t[0], t[1], t[2], t[3], d=t[4]))
                   for t in rotate((qa, fa, qb, fb, d), byt)]
            cases.append(dict(name="fp32-scale dense m=%d n=%d k=%d" % (m, n, k), fns=fns,
                              flops=2.0 * m * n * k, bytes=byt))
    elif name == "kgrouped":
        cfg = workloads.KGROUPED
        w = workloads.k_grouped(cfg["num_groups"], cfg["m"], cfg["n"], cfg["seed"])
        qa, sfa = dg.quantize_fp8_cols(w.a.to(dev))
        qb, sfb = dg.quantize_fp8_cols(w.b.to(dev))
        ks = w.ks.to(dev)
        G, m, n = cfg["num_groups"], cfg["m"], cfg["n"]
        d = torch.empty(G, m, n, dtype=torch.float32, device=dev)
        valid = int(w.counts.sum())
        sum_k = int(w.ks.sum())
        byt = valid * (m + n) + 4 * G * m * n + (sum_k // 128) * (m + n)
        fns = [(lambda t=t: dg.k_grouped_fp8_gemm_tn_contiguous(t[0], t[1], t[2], t[3], t[4], d=t[5]))
               for t in rotate((qa, sfa, qb, sfb, ks, d), byt)]
        cases.append(dict(name="k-grouped G=%d valid_k=%d padded_k=%d m=%d n=%d" % (G, valid, sum_k, m, n),
                          fns=fns, flops=2.0 * valid * m * n, bytes=byt))
    elif name == "masked":
        cfg = workloads.MASKED
        G, cap, n, k = cfg["num_groups"], cfg["cap"], cfg["n"], cfg["k"]
        w = workloads.masked(G, cap, n, k, cfg["seed"])
        qa, sfa = dg.quantize_fp8(w.a.to(dev), 1)
        qb, sfb = dg.quantize_fp8(w.b.to(dev), 128)
        mm = w.masked_m.to(dev)
        d = torch.empty(G, cap, n, dtype=torch.bfloat16, device=dev)
        valid = int(w.masked_m.sum())
        used = int((w.masked_m > 0).sum())
        byt = algorithmic_bytes_masked(valid, used, n, k)
        exp_m = int(w.masked_m.float().mean())
        fns = [(lambda t=t: dg.m_grouped_fp8_gemm_nt_masked(t[0], t[1], t[2], t[3], t[4], exp_m, d=t[5]))
               for t in rotate((qa, sfa, qb, sfb, mm, d), byt)]
        cases.append(dict(name="masked G=%d cap=%d valid_rows=%d n=%d k=%d" % (G, cap, valid, n, k),
                          fns=fns, flops=2.0 * valid * n * k, bytes=byt))
    return cases


# which roofline bounds each workload (the tensor-core rate for the
# compute-bound ones, HBM for the memory-bound ones)
CONFIG_BOUND = {"small": "tensor", "decode": "hbm", "contiguous": "tensor", "masked": "hbm",
                "kgrouped": "tensor", "fp32scales": "tensor"}
CONFIG_DESC = {
    "small": "dense NT M=128 N=256 K=512, no C",
    "decode": "dense NT decode-like M in {64,128}, (N,K) in the five prefill pairs, no C",
    "contiguous": "M-grouped contiguous MoE: 8 experts, B [8,4096,7168], per-expert rows U[256,8192] "
                  "padded to 128 (padding rows tagged -1)",
    "masked": "M-grouped masked MoE decode: 16 experts x capacity 256, B [16,7168,2048], masked_m U[0,256]",
    "kgrouped": "K-grouped MoE weight gradient: 8 experts, M=4096, N=7168, token rows U[256,8192] padded to 128",
    "fp32scales": "dense NT prefill shapes through the FP32-scale (promotion) kernel",
}


def measure_config(name, args, dg, workloads, dev, peaks, peak_src, flush):
    """GEMM-only device timing of one workload (CUDA-graph replays over input
    copies exceeding L2, and one isolated launch after an L2 flush) with its
    roofline."""
    cases = build_cases(name, dg, workloads, dev)
    if args.shape >= 0 and name == args.workload:
        cases = [cases[args.shape]]
    for c in cases:
        for _ in range(max(3, args.warmup)):
            for f in c["fns"]:
                f()
    torch.cuda.synchronize()
    st, word = dg.get_device_error()
    if st != 0:
        raise RuntimeError("device error: 0x%x" % word)
    if args.profile_steps:
        for _ in range(args.profile_steps):
            for c in cases:
                c["fns"][0]()
        torch.cuda.synchronize()
        return None
    hbm = peaks["hbm_gbs"]
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    replays = max(args.steps, 20)
    res = []
    for c in cases:
        t = _time_graph(c["fns"], replays)
        t1 = _time_gemm(c["fns"][0], max(3, replays // 3), flush)
        r = {"case": c["name"], "us": t * 1e3, "copies": len(c["fns"]),
             "tflops": c["flops"] / (t * 1e-3) / 1e12,
             "gbs": c["bytes"] / (t * 1e-3) / 1e9,
             "frac_fp8_peak": c["flops"] / (t * 1e-3) / 1e12 / fp8_peak,
             "frac_hbm": c["bytes"] / (t * 1e-3) / 1e9 / hbm,
             "us_isolated_after_flush": t1 * 1e3}
        if CONFIG_BOUND[name] == "hbm":
            fl = _stream_floor_us(c["bytes"], dev, replays)
            r["stream_floor_us"] = fl
            r["floor_over_gemm"] = fl / r["us"]
        res.append(r)
    st, word = dg.get_device_error()
    if st != 0:
        raise RuntimeError("device error: 0x%x" % word)
    tot_t = sum(r["us"] for r in res) * 1e-6
    tot_f = sum(c["flops"] for c in cases)
    tot_b = sum(c["bytes"] for c in cases)
    bound = CONFIG_BOUND[name]
    achieved = (tot_b / tot_t / 1e9) if bound == "hbm" else (tot_f / tot_t / 1e12)
    peak = hbm if bound == "hbm" else fp8_peak
    roof = {"bound": bound, "achieved": achieved, "peak": peak,
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s", "frac": achieved / peak, "traffic": None,
            "peak_source": peak_src if bound == "hbm" else
            "%s bf16 burst %.1f TFLOP/s x %.1f nominal FP8:BF16 ratio" % (peak_src, peaks["bf16_tflops"],
                                                                         FP8_OVER_BF16)}
    if name == "small":
        roof["limited_by"] = "launch latency (0.03 GFLOP per launch)"
    entry = {"workload": CONFIG_DESC[name], "value": tot_f / tot_t / 1e12, "unit": "TFLOPS",
             "us": tot_t * 1e6, "gbs": tot_b / tot_t / 1e9, "roofline": roof, "cases": res,
             "gpu_launches": sum(len(c["fns"]) for c in cases) * (replays + 1)
                             + len(cases) * max(3, replays // 3),
             "timing": "CUDA-graph replays of one launch per input copy (copies totalling > 2.5x L2), "
                       "median replay time / launches; us_isolated_after_flush: one launch after an L2 flush"}
    if CONFIG_BOUND[name] == "hbm":
        entry["stream_floor"] = ("stream_floor_us: a hand-written streaming read (libdg_floor.so) of the case's "
                                 "algorithmic bytes, timed the same way (one launch per copy in a CUDA graph); "
                                 "floor_over_gemm: its time over the GEMM's (1 = the GEMM runs at the time of "
                                 "a plain read of its bytes)")
    if name == "decode":
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        entry["plans"] = [dict(shape=list(c["shape"]), **dg.plan_fp8_gemm_nt_ws(*c["shape"], num_sms=sms))
                          for c in cases]
    del cases
    torch.cuda.empty_cache()
    return entry


def main():
    args = parse_args()
    ranks = Ranks()
    if args.impl == "reference":
        rc = run_reference(args, ranks)
        ranks.close()
        return rc
    import moe_grouped_gemm_fp8_gb300 as dg
    from moe_grouped_gemm_fp8_gb300 import workloads

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(ranks.local)
    dev = torch.device("cuda", ranks.local)
    peaks, peak_src = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    flush = torch.zeros(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    clocks = ClockSampler(torch.cuda.current_device())
    if args.workload != "prefill":
        dg.set_pdl(bool(args.pdl))
        ranks.barrier()
        clocks.start()
        entry = measure_config(args.workload, args, dg, workloads, dev, peaks, peak_src, flush)
        clk = clocks.stop()
        ranks.barrier()
        if entry is None:
            ranks.close()
            return 0
        t = ranks.max(entry["us"] * 1e-6)
        f = ranks.sum(entry["value"] * 1e12 * entry["us"] * 1e-6)
        line = {
            "metric": METRIC, "value": f / t / 1e12, "unit": "TFLOPS", "n_gpus": ranks.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3",
            "data": "synthetic",
            "config": {"workload": entry["workload"], "pdl": bool(args.pdl),
                       "l2": "inputs larger than L2: each case rotates over input copies totalling "
                             ">2.5x L2, launched back to back in a CUDA graph"},
            "roofline": entry["roofline"], "gpu_launches": entry["gpu_launches"], "cases": entry["cases"],
            "impl": "ours",
        }
        if "plans" in entry:
            line["plans"] = entry["plans"]
        if clk:
            line["clocks"] = clk
        if ranks.rank == 0 and ranks.world == 1 and not args.no_cpu_baseline and args.workload in OTHER_CONFIGS:
            line["cpu_baseline"] = cpu_baseline_config(args.workload, workloads)
        if ranks.rank == 0:
            print(json.dumps(line), flush=True)
        ranks.close()
        return 0

    # clocks are sampled from the first warm-up step to the end of the last
    # measurement (the sampler needs a few hundred ms to start reporting)
    clocks.start()
    res = run_prefill(args, ranks, dg, workloads, dev, clocks)
    if res is None:
        clocks.stop()
        ranks.close()
        return 0
    configs = {}
    if not args.no_configs:
        dg.set_pdl(bool(args.pdl))
        for name in OTHER_CONFIGS:
            configs[name] = measure_config(name, args, dg, workloads, dev, peaks, peak_src, flush)
    clk = clocks.stop()
    dom = dominant_launch(res["per_shape"])
    traffic, plan = captured_traffic(dg, dom["m"], dom["n"], dom["k"], dom["c"], num_sms)
    line = {
        "metric": METRIC, "value": res["value"], "unit": "TFLOPS", "n_gpus": ranks.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3",
        "data": "synthetic",
        "config": {"workload": "dense NT prefill-like M=4096, (N,K) in %s; per step: quantise A "
                               "(1x128, packed UE8M0), D = A@B.T and D2 = C + A@B.T per shape; B "
                               "quantised (128x128) once at setup" % (workloads.PREFILL_NK,),
                   "l2": "inputs larger than L2 (per-step working set %.2f GB)" % res["working_set_gb"],
                   "replicas": ranks.world, "pdl": bool(args.pdl)},
        "roofline": prefill_roofline(res, fp8_peak, "%s bf16 burst %.1f TFLOP/s x %.1f nominal FP8:BF16 ratio" %
                                     (peak_src, peaks["bf16_tflops"], FP8_OVER_BF16), traffic, plan),
        "gpu_launches": res["launches"],
        "shapes": res["per_shape"],
        "sustained": res["sustained"],
        "impl": "ours",
    }
    if clk:
        line["clocks"] = clk
    if res["e2e"]:
        line["e2e"] = res["e2e"]
    if configs:
        line["configs"] = configs
    if ranks.rank == 0 and ranks.world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(workloads)
        for name, entry in configs.items():
            entry["cpu_baseline"] = cpu_baseline_config(name, workloads)
    if ranks.rank == 0:
        print(json.dumps(line), flush=True)
    ranks.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
