#!/usr/bin/env python3
"""Benchmark of the Groth16 quotient-evaluation (H) path over BN254 Fr on GB300.

One step = one whole H computation (gather, three inverse NTTs with 1/n, coset shift,
three forward NTTs, join in both encodings) on the proving-key-shaped 2^18 workload
(140296 constraints, 262144 wires, CSR A/B with the GATHER_CU page's row statistics),
inputs resident in HBM. The working set (~90 MB) fits in L2, so L2 is flushed (a
256 MiB write) between timed steps, outside the timed events.

Prints ONE JSON line. Under torchrun every rank runs its own replica (independent
proofs, no data exchange); value = steps x ranks / max-over-ranks time.

--impl reference times the CPU oracle (plain C, one thread) on the same workload: the
only reference implementation this path has.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Groth16 H computations/s at 2^18"
UNIT = "H/s"
LOG_N = 18
WORKLOAD = "groth16_h_bn254_2^18"
# Integer multiply-add work in 32-bit IMAD results: a 256-bit Montgomery multiply takes
# 64 + 64 full 32x32 -> 64-bit products (two IMAD results each: the low and the high
# word) and 8 low-only products; a Montgomery reduction (from_mont) 64 full and 8 low.
OPS_PER_MM = 2 * 128 + 8
OPS_PER_FROM_MONT = 2 * 64 + 8
IMAD_PER_CLK_PER_SM = 64  # 32-bit integer multiply-add results per clock per SM
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None,
                   help="timed steps (default 1000; 10 for --impl reference)")
    p.add_argument("--warmup", type=int, default=None,
                   help="untimed warm-up steps (default 20; 1 for --impl reference)")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-extra", action="store_true", help="skip the 2^22 secondary lines")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    p.add_argument("--msm-only", action="store_true",
                   help="time only the 2^18 H multiexp over G1 (the extra line's "
                        "measurement; for profiler captures of its kernels)")
    p.add_argument("--stress-only", action="store_true",
                   help="time only the 2^22 stress H on given a, b, c and one 2^22 coset "
                        "NTT (the extra line's measurements; for profiler captures of "
                        "their kernels)")
    p.add_argument("--serialize", action="store_true",
                   help="headline pass too with the three vectors in one launch per phase "
                        "on one stream (for profiler captures of the kernels as the "
                        "roofline pass times them)")
    args = p.parse_args()
    ref = args.impl == "reference"
    if args.steps is None:
        args.steps = 10 if ref else 1000
    if args.warmup is None:
        args.warmup = 1 if ref else 20
    return args


# A reference step is one whole 2^18 H by the CPU oracle (about 1.5 s on one core); when
# the requested steps would run longer than this, the arm stops after the steps that fit
# and reports how many it timed.
REFERENCE_BUDGET_S = 240.0


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def combine_ranks(local_seconds, units_per_rank, dist=None, device=None):
    """Whole-job throughput over replicas: every rank processed units_per_rank units; the
    job took the slowest rank's time (max over ranks). Returns (units / s, max seconds)."""
    world = 1
    slowest = float(local_seconds)
    if dist is not None and dist.is_initialized():
        import torch

        world = dist.get_world_size()
        t = torch.tensor([slowest], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        slowest = float(t.item())
    return world * units_per_rank / slowest, slowest


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


_SM_COUNT = None


def sm_count():
    """The device's SM count (cudaDevAttrMultiProcessorCount, through torch)."""
    global _SM_COUNT
    if _SM_COUNT is None:
        import torch

        _SM_COUNT = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return _SM_COUNT


def imad_peak():
    """The derived IMAD peak, results per second: SMs x 32-bit IMAD results per clock per
    SM x the maximum SM clock (MEASURED_PEAKS.json's, else 2070 MHz)."""
    return sm_count() * IMAD_PER_CLK_PER_SM * float(measured_peaks().get("sm_max_mhz", 2070.0)) * 1e6


def plan_for(k):
    """Slice levels of the launch plan (mirrors the library): (kk per level)."""
    if k <= 22:
        lo = (k + 1) // 2
        return [lo, k - lo]
    lo = (k + 2) // 3
    rest = k - lo
    mid = (rest + 1) // 2
    return [lo, mid, rest - mid]


def kernel_counts_per_h(k, nnz_a, nnz_b, from_witness=True):
    """The method's Montgomery multiplies and reductions (from_mont) of one whole H on 2^k
    (every multiply of the algorithm, skipped by the kernels or not), charged to the kernel
    that does them, as {name: (multiplies, reductions)}. gather_a / gather_b: one multiply
    per term of A / of B; ntt_dif: the
    butterflies of the inverse's top slice levels (3 vectors) and, from a witness, the n
    products c = a * b formed at its load; ntt_mid: the low levels of both transforms, the
    1/n scale and the coset shift (3 vectors); ntt_dit: the forward's top levels; prejoin:
    the join's n products a * b; join: the n reductions of h_std."""
    n = 1 << k
    kk = plan_for(k)
    top = sum(kk[1:])
    c = {}
    if from_witness:
        c["gather_a"] = (nnz_a, 0)
        c["gather_b"] = (nnz_b, 0)
    c["ntt_dif"] = (3 * top * (n // 2) + (n if from_witness else 0), 0)
    c["ntt_mid"] = (3 * (kk[0] * n + 2 * n), 0)
    c["ntt_dit"] = (3 * top * (n // 2), 0)
    c["prejoin"] = (n, 0)
    c["join"] = (0, n)
    return c


def kernel_ops_per_h(k, nnz_a, nnz_b, from_witness=True, mm_ops=None, red_ops=None):
    """Algorithmic 32-bit IMAD results of one whole H per kernel name: the counts above at
    mm_ops per multiply and red_ops per reduction (default: 264 and 136, a full 32 x 32
    product counted as two results). Their sum is h_ops."""
    mm_ops = OPS_PER_MM if mm_ops is None else mm_ops
    red_ops = OPS_PER_FROM_MONT if red_ops is None else red_ops
    return {name: mm * mm_ops + red * red_ops
            for name, (mm, red) in kernel_counts_per_h(k, nnz_a, nnz_b, from_witness).items()}


def launches_per_h(k, from_witness=True):
    """Launches per kernel name of one H with G3H_SERIALIZE (three vectors per launch)."""
    levels = len(plan_for(k))
    out = {"ntt_dif": levels - 1, "ntt_mid": 1, "ntt_dit": levels - 1, "prejoin": 1, "join": 1}
    if from_witness:
        out.update({"gather_a": 1, "gather_b": 1})
    return out


def algorithmic_ops(kernel, k, nnz_a, nnz_b, from_witness=True):
    """Algorithmic 32-bit IMAD results of one launch of `kernel` (serialized H)."""
    ops = kernel_ops_per_h(k, nnz_a, nnz_b, from_witness)
    if not ops.get(kernel):
        return 0
    return ops[kernel] // launches_per_h(k, from_witness)[kernel]


def h_ops(k, nnz_a, nnz_b, from_witness=True):
    """Algorithmic IMAD results of one whole H on 2^k, the method's count: 6 (n/2) k + 7n
    multiplies (butterflies, 1/n, shift, join), with a witness nnz_A + nnz_B + n more (the
    gather and c = a * b), and n reductions."""
    n = 1 << k
    mm = 3 * n * k + 7 * n + ((nnz_a + nnz_b + n) if from_witness else 0)
    return OPS_PER_MM * mm + OPS_PER_FROM_MONT * n


def hbm_floor_bytes(k, nnz_a, nnz_b, n_wires):
    """The bytes one H must move at least: the CSR matrices (row pointers, columns, values)
    and the witness read once, h_mont and h_std written once."""
    n = 1 << k
    return 2 * (n + 1) * 4 + (nnz_a + nnz_b) * (4 + 32) + n_wires * 32 + 2 * n * 32


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                self.samples.append((time.monotonic(), float(parts[0]), float(parts[1]),
                                     parts[3:7]))
            except ValueError:
                continue

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        used = inside
        if not used and self.samples:  # region shorter than the sampling period
            used = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({self.NAMES[i] for s in used for i, v in enumerate(s[3])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(s[1] for s in used),
                "sm_max_mhz": max(s[2] for s in used), "reasons": reasons,
                "samples": len(inside)}


def cpu_baseline(A, B, w, budget_s=12.0, max_runs=20):
    """The oracle as it stands, one thread, on whole 2^18 H computations."""
    import oracle

    oracle.build()
    runs, total = 0, 0.0
    while runs < max_runs and (total < budget_s or runs == 0):
        t = time.perf_counter()
        oracle.compute_h(LOG_N, A, B, w)
        total += time.perf_counter() - t
        runs += 1
    out = {"value": runs / total, "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": "%d whole 2^18 H computations (%.1f s), C oracle, one thread" % (
               runs, total)}
    # the same oracle on every host core: independent H computations on host threads (the
    # C calls release the interpreter lock), the aggregate rate
    from concurrent.futures import ThreadPoolExecutor

    cores = max(1, os.cpu_count() or 1)
    per = max(1, int(round(budget_s / 2 / max(total / runs, 1e-3))))
    t = time.perf_counter()
    with ThreadPoolExecutor(cores) as ex:
        list(ex.map(lambda _: oracle.compute_h(LOG_N, A, B, w), range(cores * per)))
    dt = time.perf_counter() - t
    out["all_cores_value"] = cores * per / dt
    out["all_cores"] = cores
    out["all_cores_sample"] = "%d whole 2^18 H computations on %d threads (%.1f s)" % (
        cores * per, cores, dt)
    # the H multiexp's oracle (double-and-add per point) on a sample of the 2^18 bases,
    # as points per second, beside the GPU's msm_2^18_per_s * 2^18
    from bn254_scalar_field_gb300 import synth_g1

    pts = synth_g1.points(512, seed=synth_g1.default_seed(LOG_N))
    sc = synth_g1.scalars(512, seed=synth_g1.default_seed(LOG_N) + 1)
    t = time.perf_counter()
    oracle.g1_msm(pts, sc)
    dt = time.perf_counter() - t
    out["msm_points_per_s"] = 512 / dt
    out["msm_sample"] = "512 of the 2^18 bases and scalars (%.2f s), C oracle, one thread" % dt
    # the other proving-key domains, one thread, median of 5 runs (3 for 2^17); the 2^22
    # stress H (some 25 s a run on one core) is not timed
    from bn254_scalar_field_gb300 import synth

    per = {"2^18": out["value"]}
    for k, reps in ((12, 5), (14, 5), (17, 3)):
        Ak, Bk, wk = synth.problem(k)
        ts = []
        for _ in range(reps):
            t = time.perf_counter()
            oracle.compute_h(k, Ak, Bk, wk)
            ts.append(time.perf_counter() - t)
        per["2^%d" % k] = 1.0 / statistics.median(ts)
    out["per_config_h_per_s"] = per
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return
    from bn254_scalar_field_gb300 import synth
    import oracle

    oracle.build()
    A, B, w = synth.problem(LOG_N)
    for _ in range(args.warmup):
        oracle.compute_h(LOG_N, A, B, w)
    t0 = time.perf_counter()
    done = 0
    while done < args.steps:
        oracle.compute_h(LOG_N, A, B, w)
        done += 1
        if time.perf_counter() - t0 > REFERENCE_BUDGET_S:
            break
    dt = time.perf_counter() - t0
    value = done / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "steps_timed": done, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / done,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "impl": "CPU oracle (plain C, 4x64-bit limbs)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "%d whole 2^18 H computations, one thread" % done},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch

    from bn254_scalar_field_gb300 import build, g3h, synth

    torch.cuda.set_device(local)
    if args.stress_only:
        build.build()
        dev = torch.device("cuda", local)
        r = stress_2_22(torch, dev, g3h, synth, reps=args.steps, warmup=args.warmup,
                        flags=g3h.G3H_SERIALIZE if args.serialize else 0, extra=False)
        if rank == 0:
            print(json.dumps({"metric": "Groth16 H computations/s, 2^22 stress vectors",
                              "value": r["h_2^22_per_s"], "unit": "H/s", "steps": args.steps,
                              "warmup": args.warmup, "higher_is_better": True,
                              "data": "synthetic", "extra": r}))
        return
    if args.msm_only:
        build.build()
        dev = torch.device("cuda", local)
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        r = h_msm(torch, dev, g3h, flush, steps=args.steps, warmup=args.warmup)
        r.update(g2_msm(torch, dev, g3h, flush, steps=args.steps))
        if rank == 0:
            print(json.dumps({"metric": "G1 multiexp (the H MSM) at 2^18", "value": r["msm_2^18_per_s"],
                              "unit": "MSM/s", "steps": args.steps, "warmup": args.warmup,
                              "higher_is_better": True, "data": "synthetic", "extra": r}))
        return
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    build.build()
    dev = torch.device("cuda", local)
    n = 1 << LOG_N
    A, B, w = synth.problem(LOG_N)
    nnz_a, nnz_b = int(A[0][-1]), int(B[0][-1])
    ctx = g3h.Context(LOG_N, w.shape[0], A, B, device=local)
    wd = torch.from_numpy(w.view(np.int32)).to(dev)
    hm = torch.empty((n, 8), dtype=torch.int32, device=dev)
    hs = torch.empty((n, 8), dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(args.warmup, 3)):
        ctx.compute_h(wd, hm, hs)
        flush.fill_(1)
    ctx.sync()

    def timed_steps(per_kernel):
        """K steps, each bracketed by CUDA events on the launching stream, L2 flushed
        between steps outside the events. With per_kernel the library also records an
        event pair around each of its launches (a few microseconds per launch, so the
        step times of that pass are not used for the headline), and runs the three
        vectors as one launch per phase on one stream (G3H_SERIALIZE), so that each
        kernel's events bracket that kernel alone; by default the vectors run on three
        streams whose kernels overlap."""
        flags = g3h.G3H_SERIALIZE if (per_kernel or args.serialize) else 0
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        if per_kernel:
            ctx.timing_enable(True)
        t_start = time.monotonic()
        for i in range(args.steps):
            evs[i][0].record(stream)
            ctx.compute_h(wd, hm, hs, flags=flags)
            evs[i][1].record(stream)
            flush.fill_(i & 0xFF)
        torch.cuda.synchronize(dev)
        t_end = time.monotonic()
        if dist:
            dist.barrier()
        ctx.sync()
        kt = None
        if per_kernel:
            kt = ctx.timing_read()
            ctx.timing_enable(False)
        return sum(a.elapsed_time(b) for a, b in evs) / 1e3, kt, t_start, t_end

    sampler = ClockSampler(local)
    time.sleep(0.1)
    local_s, _, t0, t1 = timed_steps(False)
    sampler.stop()
    value, step_s = combine_ranks(local_s, args.steps, dist, dev)
    step_ms = step_s * 1e3
    # second pass of the same K steps: per-kernel device times for the roofline
    serial_s, kt, _, _ = timed_steps(True)
    # launches per headline step (three streams): counted on one step
    ctx.timing_enable(True)
    ctx.compute_h(wd, hm, hs)
    launches = args.steps * sum(v[0] for v in ctx.timing_read().values())
    ctx.timing_enable(False)

    # roofline of the dominant kernel: algorithmic IMAD results per launch / mean time
    top = max(kt, key=lambda k: kt[k][1])
    top_launches, top_ms = kt[top]
    per_launch_ms = top_ms / top_launches
    per_h = launches_per_h(LOG_N)
    census = {k: v[0] / args.steps for k, v in kt.items()}
    ops = algorithmic_ops(top, LOG_N, nnz_a, nnz_b)
    peaks = measured_peaks()
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    sms = sm_count()
    peak_tops = sms * IMAD_PER_CLK_PER_SM * sm_max * 1e6 / 1e12
    achieved = ops / (per_launch_ms * 1e-3) / 1e12
    traffic = None
    heavy_pct = None
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f)
        from bn254_scalar_field_gb300.build import kernel_digest

        ent = rec.get(top)
        if ent and ent.get("kernel_digest") == kernel_digest(top) and ent.get("log_n") == LOG_N:
            traffic = ent["bytes_per_launch"]
            heavy_pct = ent.get("pipe_fma_heavy_pct")
    except (OSError, ValueError, ImportError):
        pass
    per_h_ops = h_ops(LOG_N, nnz_a, nnz_b)
    step_s_1 = step_ms / args.steps * 1e-3
    kernel_ms_sum = sum(v[1] for v in kt.values()) / args.steps
    # the multiply pipe measured on this GPU by the library's probes (independent chains of
    # mad.lo, mad.hi and mad.wide on every SM), outside the timed regions
    p_lo = ctx.measure_int_mul(g3h.G3H_MUL_LO) / 1e12
    p_hi = ctx.measure_int_mul(g3h.G3H_MUL_HI) / 1e12
    p_wide = ctx.measure_int_mul(g3h.G3H_MUL_WIDE) / 1e12
    # the cost of a full 32 x 32 -> 64 product in 32-bit IMAD slots, as measured: a
    # Montgomery multiply then costs 128 such products and 8 low words
    wide_slots = p_lo / p_wide
    mm_measured = 128 * wide_slots + 8
    red_measured = 64 * wide_slots + 8
    top_measured = kernel_ops_per_h(LOG_N, nnz_a, nnz_b, mm_ops=mm_measured,
                                    red_ops=red_measured)[top] / per_h[top]
    h_measured = sum(kernel_ops_per_h(LOG_N, nnz_a, nnz_b, mm_ops=mm_measured,
                                      red_ops=red_measured).values())
    roofline = {
        "bound": "alu", "kernel": top, "achieved": achieved, "peak": peak_tops,
        "unit": "T IMAD/s", "frac": achieved / peak_tops, "traffic": traffic,
        "peak_source": "derived: %d SMs x %d 32-bit IMAD results/clk/SM x %.0f MHz; a "
                       "32x32->64 product counts two" % (sms, IMAD_PER_CLK_PER_SM, sm_max),
        "whole_step_frac": per_h_ops / step_s_1 / 1e12 / peak_tops,
        "peak_measured": p_lo,
        "peak_measured_hi": p_hi,
        "peak_measured_wide": p_wide,
        "frac_of_measured": achieved / p_lo,
        "whole_step_frac_of_measured": per_h_ops / step_s_1 / 1e12 / p_lo,
        "wide_product_slots_measured": wide_slots,
        "ops_per_mm_measured_slots": mm_measured,
        "frac_of_measured_in_measured_slots": top_measured / (per_launch_ms * 1e-3) / 1e12 / p_lo,
        "whole_step_frac_of_measured_in_measured_slots": h_measured / step_s_1 / 1e12 / p_lo,
        "ncu_heavy_fma_pipe_pct": heavy_pct,
        "h_ops": per_h_ops,
        "launch_census_per_h": census,
        "launch_census_ok": census == {k: float(v) for k, v in per_h.items()},
        "timing": "step times from a pass without per-kernel events (vectors on three "
                  "streams); kernel times from a second pass of the same K steps with the "
                  "library's per-launch events and the three vectors in one launch per "
                  "phase on one stream (G3H_SERIALIZE), so each kernel runs alone",
        "serialized_ms_per_step": serial_s * 1e3 / args.steps,
        "kernels_ms_per_step_sum": kernel_ms_sum,
        "kernels_ms_per_step": {k: v[1] / args.steps for k, v in kt.items()},
    }

    # end to end through the public API with host (pinned) buffers, copies included
    wp = torch.from_numpy(w.view(np.int32)).pin_memory()
    hmp = torch.empty((n, 8), dtype=torch.int32).pin_memory()
    hsp = torch.empty((n, 8), dtype=torch.int32).pin_memory()
    e2e_steps = max(3, min(args.steps, 200))
    for _ in range(3):
        ctx.compute_h(wp, hmp, hsp)
    e2e_s = 0.0
    for _ in range(e2e_steps):
        flush.fill_(3)
        torch.cuda.synchronize(dev)
        t = time.perf_counter()
        ctx.compute_h(wp, hmp, hsp)
        e2e_s += time.perf_counter() - t
    e2e_value, e2e_s = combine_ranks(e2e_s, e2e_steps, dist, dev)
    e2e = {"value": e2e_value, "unit": UNIT, "steps": e2e_steps,
           "h2d_bytes_per_step": int(w.nbytes), "d2h_bytes_per_step": int(2 * n * 32)}

    extra = {"ntt_gelem_s_2^18_in_h": 6 * n / (step_ms / args.steps * 1e-3) / 1e9}
    # HBM as the secondary roof: the bytes an H must move at least, per step time
    floor = hbm_floor_bytes(LOG_N, nnz_a, nnz_b, int(w.shape[0]))
    floor_gbs = floor / (step_ms / args.steps * 1e-3) / 1e9
    hbm_peak = float(measured_peaks().get("hbm_gbs", 0.0)) or None
    extra.update({"hbm_floor_bytes_per_h_2^18": floor, "hbm_floor_gb_s_2^18": floor_gbs,
                  "hbm_floor_frac_of_measured_2^18": floor_gbs / hbm_peak if hbm_peak else None})
    extra.update(batched(torch, dev, ctx, w, n, flush))
    if not args.no_extra and rank == 0:
        extra.update(h_msm(torch, dev, g3h, flush))
        extra.update(g2_msm(torch, dev, g3h, flush))
        extra.update(other_domains(torch, dev, g3h, synth, flush))
        extra.update(stress_2_22(torch, dev, g3h, synth))
    ctx.close()

    if rank == 0:
        cpu = None if args.no_cpu else cpu_baseline(A, B, w)
        clocks = sampler.summary(t0, t1)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "constraints": 140296, "wires": int(w.shape[0]),
                       "nnz_a": nnz_a, "nnz_b": nnz_b, "parallelism": "replicas x%d" % world,
                       "l2": "flushed between timed steps (256 MiB write)"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clocks, "extra": extra,
        }
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


def batched(torch, dev, ctx, w, n, flush, count=8, reps=20):
    """Batched H (several witnesses per call, on overlapping lanes): H/s with inputs in
    HBM, and end to end with pinned host buffers. Same witness repeated: the work is
    data-independent."""
    stream = torch.cuda.current_stream(dev)
    wd = torch.from_numpy(w.view(np.int32)).to(dev).unsqueeze(0).repeat(count, 1, 1).contiguous()
    hm = torch.empty((count, n, 8), dtype=torch.int32, device=dev)
    hs = torch.empty_like(hm)
    for _ in range(3):
        ctx.compute_h_batch(wd, hm, hs)
    ms = 0.0
    for _ in range(reps):
        flush.fill_(5)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ctx.compute_h_batch(wd, hm, hs)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms += e0.elapsed_time(e1)
    wp = wd.cpu().pin_memory()
    hmp = torch.empty((count, n, 8), dtype=torch.int32).pin_memory()
    hsp = torch.empty_like(hmp).pin_memory()
    ctx.compute_h_batch(wp, hmp, hsp)
    e2e_s = 0.0
    for _ in range(reps // 2):
        flush.fill_(6)
        torch.cuda.synchronize(dev)
        t = time.perf_counter()
        ctx.compute_h_batch(wp, hmp, hsp)
        e2e_s += time.perf_counter() - t
    return {"batch_count": count, "batch_h_per_s": count * reps / (ms * 1e-3),
            "batch_e2e_h_per_s": count * (reps // 2) / e2e_s}


MSM_OPS_PER_MADD = (8 + 2) * OPS_PER_MM  # madd-2008-s: 8 multiplies + 2 squarings


def h_msm(torch, dev, g3h, flush, steps=50, warmup=3):
    """The H multiexp at 2^18 (sum of h_i P_i over G1, h uniform in [0, r), bases sampled
    on the curve): device buffers, bases prepared once (untimed), L2 flushed between
    steps. Roofline of the bucket accumulation: one mixed addition per nonzero window
    digit (16 per scalar), 10 Montgomery multiplies each."""
    from bn254_scalar_field_gb300 import synth_g1

    k = LOG_N
    n = 1 << k
    pts = synth_g1.points(n, seed=synth_g1.default_seed(k))
    sc = synth_g1.scalars(n, seed=synth_g1.default_seed(k) + 1)
    ctx = g3h.Context(0, device=dev.index)
    ctx.msm_prepare(torch.from_numpy(pts.view(np.int32)).to(dev))
    sd = torch.from_numpy(sc.view(np.int32)).to(dev)
    res = torch.zeros(24, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(warmup, 1)):
        ctx.msm(sd, res)
    evs = []
    for i in range(steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.fill_(i & 0xFF)
        e0.record(stream)
        ctx.msm(sd, res)
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize(dev)
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    ctx.timing_enable(True)
    for i in range(10):
        flush.fill_(i & 0xFF)
        ctx.msm(sd, res)
    kt = ctx.timing_read()
    ctx.timing_enable(False)
    ctx.sync()
    # a witness multiexp on the same bases: the 2^18 proving-key witness (99 % of wires 0
    # or 1) in standard form, made on the device
    from bn254_scalar_field_gb300 import synth

    _, _, w = synth.problem(k)
    wd = torch.from_numpy(w.view(np.int32)).to(dev)
    ws = torch.empty_like(wd)
    ctx.mont_to_std(wd, ws)
    for _ in range(3):
        ctx.msm(ws, res)
    wevs = []
    for i in range(steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.fill_(i & 0xFF)
        e0.record(stream)
        ctx.msm(ws, res)
        e1.record(stream)
        wevs.append((e0, e1))
    torch.cuda.synchronize(dev)
    wit_ms = statistics.median(a.elapsed_time(b) for a, b in wevs)
    ctx.timing_enable(True)
    for i in range(10):
        flush.fill_(i & 0xFF)
        ctx.msm(ws, res)
    wkt = ctx.timing_read()
    ctx.timing_enable(False)
    ctx.sync()
    ctx.close()
    entries = 16 * n  # nonzero digits: all but about 2^-16 of them
    acc_ms = kt["msm_accumulate"][1] / kt["msm_accumulate"][0]
    peak = imad_peak()
    achieved = entries * MSM_OPS_PER_MADD / (acc_ms * 1e-3)
    return {"msm_2^18_ms": ms, "msm_2^18_per_s": 1e3 / ms,
            "witness_msm_2^18_ms": wit_ms,
            "witness_msm_2^18_kernels_ms": {k2: v[1] / v[0] for k2, v in wkt.items()},
            "msm_2^18_points_per_s": n * 1e3 / ms,
            "msm_2^18_kernels_ms": {k2: v[1] / v[0] for k2, v in kt.items()},
            "msm_accumulate_t_imad_s": achieved / 1e12,
            "msm_accumulate_frac_of_derived_imad_peak": achieved / peak}


MSM_G2_OPS_PER_MADD = (8 * 3 + 2 * 2) * OPS_PER_MM  # F_q2: 3 F_q multiplies, 2 per square


def g2_msm(torch, dev, g3h, flush, k=16, steps=20):
    """The multiexp over the twist (G2, the B query's) on 2^16 sampled twist points, with
    uniform scalars and with a witness (99 % of the values 0 or 1) as scalars: device
    buffers, bases prepared once, L2 flushed between steps."""
    from bn254_scalar_field_gb300 import synth_g1, synth_g2

    n = 1 << k
    pts = synth_g2.points(n, seed=synth_g2.default_seed(k))
    sc = synth_g1.scalars(n, seed=synth_g2.default_seed(k) + 1)
    ctx = g3h.Context(0, device=dev.index)
    ctx.msm_g2_prepare(torch.from_numpy(pts.view(np.int32)).to(dev))
    sd = torch.from_numpy(sc.view(np.int32)).to(dev)
    res = torch.zeros(48, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        ctx.msm_g2(sd, res)
    evs = []
    for i in range(steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.fill_(i & 0xFF)
        e0.record(stream)
        ctx.msm_g2(sd, res)
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize(dev)
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    ctx.timing_enable(True)
    for i in range(5):
        flush.fill_(i & 0xFF)
        ctx.msm_g2(sd, res)
    kt = ctx.timing_read()
    ctx.timing_enable(False)
    # the B query's multiexp proper takes the witness as scalars: 99 % of the wires 0 or 1
    # (the 2^17 and 2^18 proving keys' share), in standard form, made on the device
    from bn254_scalar_field_gb300 import synth

    w = synth.witness(synth.SplitMix64(synth.default_seed(k) + 7), n, 0.99)
    wd = torch.from_numpy(w.view(np.int32)).to(dev)
    ws = torch.empty_like(wd)
    ctx.mont_to_std(wd, ws)
    for _ in range(3):
        ctx.msm_g2(ws, res)
    wevs = []
    for i in range(steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.fill_(i & 0xFF)
        e0.record(stream)
        ctx.msm_g2(ws, res)
        e1.record(stream)
        wevs.append((e0, e1))
    torch.cuda.synchronize(dev)
    ctx.sync()
    wit_ms = statistics.median(a.elapsed_time(b) for a, b in wevs)
    ctx.close()
    acc_ms = kt["msm_accumulate"][1] / kt["msm_accumulate"][0]
    peak = imad_peak()
    achieved = 16 * n * MSM_G2_OPS_PER_MADD / (acc_ms * 1e-3)
    return {"msm_g2_2^%d_ms" % k: ms,
            "witness_msm_g2_2^%d_ms" % k: wit_ms,
            "msm_g2_2^%d_kernels_ms" % k: {k2: v[1] / v[0] for k2, v in kt.items()},
            "msm_g2_accumulate_frac_of_derived_imad_peak": achieved / peak}


def other_domains(torch, dev, g3h, synth, flush, steps=200):
    """H/s on the other three proving-key-shaped domains (2^12, 2^14, 2^17), timed like
    the headline: device buffers, L2 flushed between steps outside the events."""
    out = {}
    stream = torch.cuda.current_stream(dev)
    for k in (12, 14, 17):
        A, B, w = synth.problem(k)
        n = 1 << k
        ctx = g3h.Context(k, w.shape[0], A, B, device=dev.index)
        wd = torch.from_numpy(w.view(np.int32)).to(dev)
        hm = torch.empty((n, 8), dtype=torch.int32, device=dev)
        hs = torch.empty_like(hm)
        for _ in range(5):
            ctx.compute_h(wd, hm, hs)
        evs = []
        for i in range(steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ctx.compute_h(wd, hm, hs)
            e1.record(stream)
            evs.append((e0, e1))
            flush.fill_(i & 0xFF)
        torch.cuda.synchronize(dev)
        ms = sum(a.elapsed_time(b) for a, b in evs) / steps
        ops = h_ops(k, int(A[0][-1]), int(B[0][-1]))
        out["h_per_s_2^%d" % k] = 1e3 / ms
        out["ms_per_h_2^%d" % k] = ms
        out["h_2^%d_frac_of_derived_imad_peak" % k] = ops / (ms * 1e-3) / imad_peak()
        # batched: many witnesses per call (device buffers), one launch per phase per
        # chunk of witnesses on these domains
        count = 256 if k <= 14 else 32
        wb = wd.unsqueeze(0).repeat(count, 1, 1).contiguous()
        hmb = torch.empty((count, n, 8), dtype=torch.int32, device=dev)
        hsb = torch.empty_like(hmb)
        for _ in range(2):
            ctx.compute_h_batch(wb, hmb, hsb)
        bms = []
        for i in range(10):
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ctx.compute_h_batch(wb, hmb, hsb)
            e1.record(stream)
            bms.append((e0, e1))
        torch.cuda.synchronize(dev)
        bms = statistics.median(a.elapsed_time(b) for a, b in bms)
        out["batch_h_per_s_2^%d" % k] = count * 1e3 / bms
        out["batch_count_2^%d" % k] = count
        out["batch_h_2^%d_frac_of_derived_imad_peak" % k] = count * ops / (bms * 1e-3) / imad_peak()
        ctx.close()
        del wb, hmb, hsb
    return out


def stress_2_22(torch, dev, g3h, synth, reps=10, warmup=2, flags=0, extra=True):
    """Secondary figures on the 2^22 stress vectors (inputs larger than L2): one forward
    coset NTT (Fr NTT Gelem/s) and the H path on given a, b, c = a*b; with `extra` also the
    witness copy to standard form on 2^24 elements."""
    k = synth.STRESS_LOG_N
    n = 1 << k
    a, b = synth.stress_ab(k)
    ctx = g3h.Context(k, device=dev.index)
    ad = torch.from_numpy(a.view(np.int32)).to(dev)
    bd = torch.from_numpy(b.view(np.int32)).to(dev)
    cd = torch.empty_like(ad)
    ctx.mul(ad, bd, cd)
    hm = torch.empty_like(ad)
    hs = torch.empty_like(ad)
    x = ad.clone()
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(warmup):
            fn()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ts.append((e0, e1))
        torch.cuda.synchronize(dev)
        return statistics.median(a.elapsed_time(b) for a, b in ts)

    h_ms = timed(lambda: ctx.compute_h_abc(ad, bd, cd, hm, hs, flags=flags))
    ntt_ms = timed(lambda: ctx.ntt(x, coset=True))
    if not extra:
        ctx.sync()
        ctx.close()
        ops = h_ops(k, 0, 0, from_witness=False)
        return {"h_2^22_abc_ms": h_ms, "h_2^22_per_s": 1e3 / h_ms,
                "h_2^22_frac_of_derived_imad_peak": ops / (h_ms * 1e-3) / imad_peak(),
                "ntt_2^22_coset_fwd_ms": ntt_ms, "ntt_2^22_gelem_s": n / (ntt_ms * 1e-3) / 1e9}
    # the witness copy to standard form (HBM-bound: 32 bytes read + 32 written per
    # element) on 2^24 elements, 4x the L2 each way
    del x, hm, hs
    big = torch.cat([ad, bd, cd, ad])
    big_out = torch.empty_like(big)
    m2s_ms = timed(lambda: ctx.mont_to_std(big, big_out))
    m2s_gbs = 64 * big.shape[0] / (m2s_ms * 1e-3) / 1e9
    ctx.sync()
    ctx.close()
    peak = float(measured_peaks().get("hbm_gbs", 0.0)) or None
    ops = h_ops(k, 0, 0, from_witness=False)
    peak_imad = imad_peak()
    return {"h_2^22_frac_of_derived_imad_peak": ops / (h_ms * 1e-3) / peak_imad,
            "ntt_2^22_coset_fwd_ms": ntt_ms, "ntt_2^22_gelem_s": n / (ntt_ms * 1e-3) / 1e9,
            "h_2^22_abc_ms": h_ms, "h_2^22_per_s": 1e3 / h_ms,
            "ntt_gelem_s_2^22_in_h": 6 * n / (h_ms * 1e-3) / 1e9,
            "mont_to_std_2^24_ms": m2s_ms, "mont_to_std_2^24_gb_s": m2s_gbs,
            "mont_to_std_2^24_frac_of_measured_hbm": m2s_gbs / peak if peak else None}


if __name__ == "__main__":
    main()
