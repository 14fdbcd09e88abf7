"""Benchmark: effective GB/s of random BMMC permutations at n = 28, int32.

Workload (one step): the 1 GiB array in[i] = i (2^28 int32) permuted by the
32 random invertible BMMCs of seeds 0..31 (splitmix64 rejection sampling,
c drawn after acceptance), one single-pass launch each, inputs resident in
HBM.  Effective bandwidth = (read + write bytes) / time = 2 * 2^28 * 4 bytes
per permutation ("A kernel that is correct", "One number").  The array is
8x the L2, so no L2 flush is needed between launches.

Also reported: the copy kernel on the same bytes (the practical ceiling),
the worst-case matrix (low 10 bits mapped entirely to high bits), the other
benchmark configurations, the end-to-end figure through the host-buffer C
entry point, the roofline of the dominant kernel, SM clocks sampled during
the timed region, and the CPU oracle on a bounded sample (the baseline).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (under torchrun) every rank runs the same workload on its own GPU
(replicas: the permutation needs no exchange at one array per GPU) and the
time is the maximum over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective GB/s (read+write) for random BMMC at n=28 int32; % of copy & HBM peak"
UNIT = "GB/s"
N_BITS = 28
ELEM = 4
SEEDS = 32
WORST_LOW = 10
HBM_NOMINAL_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["bmmc_index_transforms_gb300/csrc/kernels.cu",
                  "bmmc_index_transforms_gb300/csrc/kernel_params.h",
                  "bmmc_index_transforms_gb300/csrc/planner.cpp"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "bmmc_tiled_kernel_n28_int32_random.md")


def workload_name() -> str:
    return (f"random invertible BMMC n={N_BITS} int32 (in[i]=i, 1 GiB), seeds 0..{SEEDS - 1}, "
            "one single-pass permutation per seed")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic():
    """Bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (null otherwise)."""
    try:
        text = open(TRAFFIC_FILE).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return int(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", self.gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # samples under load: power above the midpoint of idle and peak draw
        thr = (min(power) + max(power)) / 2 if power else 0
        loaded = [s for s, p in zip(sm, power) if p >= thr] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


def gpu_id_for_smi(torch, dev_index: int) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev_index] if vis else str(dev_index)


# ---------------------------------------------------------------------------
# CPU oracle (the baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample_gbs(sample_log2: int, seed: int, threads: int, x_offset: int = 0, n_bits: int = N_BITS):
    """Time the CPU oracle (as it stands) scattering a contiguous sample of
    2^sample_log2 source indices of the n = 28 workload for one seed."""
    import numpy as np

    import oracle
    from oracle import reference as ref
    from bmmc_index_transforms_gb300 import synth

    rows, c, _ = synth.draw_bmmc(seed, n_bits, lambda r: ref.f2_rank(n_bits, r) == n_bits)
    global _ORACLE_BUFS
    try:
        inp, out = _ORACLE_BUFS
        assert inp.shape[0] == 1 << n_bits
    except NameError:
        inp = np.arange(1 << n_bits, dtype=np.uint32)
        out = np.empty_like(inp)
        out.fill(0)  # touch every page now, so the timed scatter takes no first-touch faults
        _ORACLE_BUFS = (inp, out)
    lo = x_offset % (1 << n_bits)
    hi = min(1 << n_bits, lo + (1 << sample_log2))
    t0 = time.perf_counter()
    oracle.scatter(n_bits, rows, c, inp, out, threads=threads, x_range=(lo, hi))
    dt = time.perf_counter() - t0
    return 2.0 * (hi - lo) * ELEM / dt / 1e9, dt, hi - lo


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle

    threads = oracle.host_threads()
    total = args.warmup + args.steps
    sample_log2 = args.ref_sample_log2 or (23 if total <= 60 else 22 if total <= 200 else 20)
    vals = []
    t_all = 0.0
    for s in range(total):
        gbs, dt, cnt = oracle_sample_gbs(sample_log2, s % SEEDS, threads, x_offset=s << sample_log2,
                                         n_bits=args.ref_n)
        if s >= args.warmup:
            vals.append((cnt, dt))
            t_all += dt
    moved = sum(2.0 * cnt * ELEM for cnt, _ in vals)
    value = moved / t_all / 1e9
    sample = (f"per step 2^{sample_log2} consecutive source indices of one seed's n={args.ref_n} int32 "
              f"permutation (seed = step mod 32), plain C oracle loop split over {threads} host threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_all / max(1, args.steps) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic", "config": {"workload": workload_name(), "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def median(xs):
    return statistics.median(xs) if xs else float("nan")


def max_over_ranks(torch, value: float, dist=None, device=None) -> float:
    """The slowest rank's time (MAX all-reduce); the value itself at N = 1."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput_gbs(world: int, launches_per_rank: int, bytes_per_launch: float, elapsed_ms: float) -> float:
    """Whole-job effective GB/s: the bytes all replicas moved over the
    slowest rank's time."""
    return world * launches_per_rank * bytes_per_launch / (elapsed_ms / 1e3) / 1e9


def time_launches(torch, fn, reps: int, warm: int = 2):
    """Mean milliseconds per call of fn() over `reps` back-to-back calls
    between two CUDA events on the current stream (the queue stays full, so
    no host launch latency is counted).  For arrays larger than the L2 this
    is the cold-cache time of one launch.  Returns (mean, mean, mean) for the
    (median, min, mean) interface."""
    for _ in range(warm):
        fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    return ms, ms, ms


def time_small(torch, fn, flush_buf, reps: int = 30):
    """Two figures for arrays that fit in the L2: `flushed` - before each
    timed launch a write of a buffer larger than the L2 both evicts the
    array and keeps the GPU busy, so the event pair brackets only the
    kernel; `warm` - the median of back-to-back launches with the array
    resident in the L2."""
    for _ in range(3):
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda.synchronize()
    for a, b in ev:
        flush_buf.zero_()
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    flushed = median([a.elapsed_time(b) for a, b in ev])
    warm, _, _ = time_launches(torch, fn, reps, warm=1)
    return flushed, warm


def run_ours(args):
    import torch

    import bmmc_index_transforms_gb300 as bm
    from bmmc_index_transforms_gb300 import _build, synth

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        dist = None
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    if rank == 0:
        _build.build()
    if dist:
        dist.barrier()
    _build.build()  # no-op when fresh

    N = 1 << N_BITS
    nbytes = N * ELEM
    alg_bytes = 2.0 * nbytes  # one read + one write of the array per permutation

    def planner_accepts(rows):
        try:
            h = bm.bmmc_plan(N_BITS, rows, 0, ELEM)
        except bm.BmmcError as e:
            if e.status == 2:
                return False
            raise
        bm.bmmc_plan_destroy(h)
        return True

    plans, mats = [], []
    for s in range(SEEDS):
        rows, c, _ = synth.draw_bmmc(s, N_BITS, planner_accepts)
        plans.append(bm.Plan(rows, c, ELEM))
        mats.append((rows, c))
    wrows, wc, _ = synth.draw_bmmc(0, N_BITS, planner_accepts, low_to_high=WORST_LOW)
    worst = bm.Plan(wrows, wc, ELEM)

    d_in = torch.arange(N, dtype=torch.int32, device=dev)
    d_out = torch.empty_like(d_in)
    stream = torch.cuda.current_stream(dev)

    def step(record=None):
        for k, p in enumerate(plans):
            if record is not None:
                record[k][0].record(stream)
            p.permute(d_in, d_out, stream)
            if record is not None:
                record[k][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # Timed region: back-to-back launches with one event at every step
    # boundary (K + 1 events; nothing else on the stream, so the events add
    # no gaps).  The headline is the median step time; the roofline's mean
    # launch duration is the whole region's time over its launches.
    sampler = ClockSampler(gpu_id_for_smi(torch, dev.index)) if rank == 0 else None
    if sampler:
        sampler.start()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    marks[0].record(stream)
    for k in range(args.steps):
        step()
        marks[k + 1].record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    step_ms = [marks[k].elapsed_time(marks[k + 1]) for k in range(args.steps)]
    elapsed_ms = max_over_ranks(torch, marks[0].elapsed_time(marks[-1]), dist, dev)
    median_step_ms = max_over_ranks(torch, median(step_ms), dist, dev)
    launches = args.steps * len(plans)
    value = job_throughput_gbs(world, len(plans), alg_bytes, median_step_ms)
    value_region = job_throughput_gbs(world, launches, alg_bytes, elapsed_ms)
    mean_launch_ms = elapsed_ms / launches

    # Per-seed figures from a short separate pass with an event pair around
    # every launch (after the timed region).
    probe_steps = 5
    per_launch = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
                   for _ in plans] for _ in range(probe_steps)]
    for k in range(probe_steps):
        step(per_launch[k])
    torch.cuda.synchronize(dev)
    launch_ms = [[a.elapsed_time(b) for a, b in per_launch[k]] for k in range(probe_steps)]
    per_seed_gbs = [alg_bytes / (median([launch_ms[k][s] for k in range(probe_steps)]) / 1e3) / 1e9
                    for s in range(len(plans))]

    # --- extras (outside the timed region) ---
    copy_med, copy_min, _ = time_launches(torch, lambda: bm.bmmc_copy(d_in, d_out, nbytes, stream), 30)
    copy_gbs = alg_bytes / (copy_med / 1e3) / 1e9
    torch_copy_med, _, _ = time_launches(torch, lambda: d_out.copy_(d_in), 20)
    torch_copy_gbs = alg_bytes / (torch_copy_med / 1e3) / 1e9
    w_med, w_min, w_mean = time_launches(torch, lambda: worst.permute(d_in, d_out, stream), 30)
    worst_gbs = alg_bytes / (w_med / 1e3) / 1e9
    configs = other_configs(torch, bm, synth, dev, stream) if not args.quick else {}
    e2e = end_to_end(torch, bm, plans, dev, stream, nbytes, alg_bytes)

    peak, peak_kind = measured_peak()
    achieved = alg_bytes / (mean_launch_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": committed_traffic(),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "kernel": "bmmc_tiled_kernel<elem=4, threads=%d, chunks_per_thread=%d>" % (
                    plans[0].info["threads"], plans[0].info["chunks_per_thread"]),
                "algorithmic_bytes_per_launch": int(alg_bytes)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle

        threads = oracle.host_threads()
        gbs, dt, cnt = oracle_sample_gbs(24, 0, threads)
        # scale the sample so that it holds roughly 10-30 s of CPU work
        target_cpu_s = 20.0
        log2 = 24
        while dt * threads < target_cpu_s / 2 and log2 < 27:
            log2 += 1
            gbs, dt, cnt = oracle_sample_gbs(log2, 0, threads)
        cpu = {"value": round(gbs, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"2^{log2} consecutive source indices of the seed-0 n=28 int32 permutation "
                         f"({dt:.2f} s wall on {threads} host threads; plain C oracle loop)"}
        # the same loop on one host thread (a 2^22-index sample, about a second)
        g1, dt1, _ = oracle_sample_gbs(22, 0, 1, x_offset=1 << 26)
        cpu["single_thread"] = {"value": round(g1, 4), "unit": UNIT, "cores": 1,
                                "sample": f"2^22 source indices of the same permutation ({dt1:.2f} s)"}

    if rank == 0:
        seed_mean = sum(per_seed_gbs) / len(per_seed_gbs)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(median_step_ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
            "data": "synthetic",
            "config": {"workload": workload_name(), "n": N_BITS, "elem_bytes": ELEM,
                       "matrices_per_step": len(plans), "mode": "single pass",
                       "statistic": "value = the step's algorithmic bytes / median CUDA-event step time "
                                    "(one event at every step boundary, max over ranks)",
                       "l2": "inputs larger than L2 (1 GiB array, 126 MB L2): no flush",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "value_region_mean": round(value_region, 2),
            "ms_per_step_region_mean": round(elapsed_ms / args.steps, 4),
            "per_seed_median_gbs_mean": round(seed_mean, 1),
            "per_seed_median_gbs_min": round(min(per_seed_gbs), 1),
            "per_seed_median_pct_of_copy_min": round(min(per_seed_gbs) / copy_gbs, 4),
            "pct_of_copy": round(value / world / copy_gbs, 4),
            "pct_of_hbm_8tbs": round(value / world / HBM_NOMINAL_GBS, 4),
            "copy_kernel_gbs": round(copy_gbs, 1),
            "torch_copy_gbs": round(torch_copy_gbs, 1),
            "per_seed_median_gbs": {"mean": round(seed_mean, 1),
                                    "median": round(median(per_seed_gbs), 1),
                                    "min": round(min(per_seed_gbs), 1),
                                    "max": round(max(per_seed_gbs), 1),
                                    "all": [round(v, 1) for v in per_seed_gbs]},
            "worst_case_gbs": round(worst_gbs, 1),
            "configs": configs,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    for p in plans:
        p.close()
    worst.close()
    if dist:
        dist.destroy_process_group()
    return 0


# Times per copy the Futhark copy post prints ("Impact", with the stride
# sorting) on an AMD RX 7900 XT, in microseconds: context, not a target.
PAGE_US_RX7900XT = {
    ("slice_2d", (8192, 8193)): 971, ("slice_2d", (65536, 1025)): 992,
    ("slice_2d", (1048576, 65)): 990, ("slice_2d", (16777216, 5)): 1010,
    ("slice_3d", (256, 256, 1025)): 1366, ("slice_3d", (65536, 32, 33)): 1364,
    ("reversed_rows", (8192, 8192)): 996, ("reversed_rows", (16777216, 4)): 999,
}


def axes_lmad(synth, shape, perm):
    """x.permute(perm) made contiguous, as a copy between two LMADs."""
    out_rm = synth.row_major_strides([shape[p] for p in perm])
    out_strides = [0] * len(shape)
    for pos, p in enumerate(perm):
        out_strides[p] = out_rm[pos]
    total = 1
    for v in shape:
        total *= v
    return dict(sizes=list(shape), in_offset=0, in_strides=synth.row_major_strides(shape), in_elems=total,
                out_offset=0, out_strides=out_strides, out_elems=total)


def lmad_case(torch, bm, w, a32, b32, stream, page_us=None, elem=4):
    """One general LMAD copy (elements of `elem` bytes, buffers viewed as
    bytes): mean of 30 back-to-back launches; effective bytes = one read and
    one write of the destination."""
    src = a32.view(torch.uint8)[: w["in_elems"] * elem]
    dst = b32.view(torch.uint8)[: w["out_elems"] * elem]
    args = (w["sizes"], w["in_offset"], w["in_strides"], w["out_offset"], w["out_strides"], elem)
    kind = bm.lmad_copy_query(*args, src, dst)["kind"]
    ms, _, _ = time_launches(torch, lambda: bm.lmad_copy(*args, src, dst, stream), 30)
    r = {"kind": kind, "us": round(ms * 1e3, 1), "gbs": round(2.0 * w["out_elems"] * elem / (ms / 1e3) / 1e9, 1)}
    if page_us:
        r["page_us_rx7900xt"] = page_us
    return r


def other_configs(torch, bm, synth, dev, stream):
    """Effective GB/s of the other benchmark configurations.  Arrays larger
    than the L2: mean of 30 back-to-back launches.  Arrays that fit in it:
    L2-flushed median and warm back-to-back mean."""
    from bmmc_index_transforms_gb300.maps import axes_rows, bitrev_rows, rotate_rows

    out = {}
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def big(n, elem, fn):
        ms, _, _ = time_launches(torch, fn, 30)
        return {"gbs": round(2.0 * (1 << n) * elem / (ms / 1e3) / 1e9, 1), "ms": round(ms, 4)}

    def small(n, elem, fn):
        fl, warm = time_small(torch, fn, flush_buf)
        b = 2.0 * (1 << n) * elem
        return {"gbs_l2_flushed": round(b / (fl / 1e3) / 1e9, 1), "ms_l2_flushed": round(fl, 4),
                "gbs_warm": round(b / (warm / 1e3) / 1e9, 1), "ms_warm": round(warm, 4)}

    def accept(n):
        def f(rows):
            try:
                bm.bmmc_plan_destroy(bm.bmmc_plan(n, rows, 0, 4))
                return True
            except bm.BmmcError:
                return False
        return f

    # C1: n=16 random int32, seed 0 (512 KiB moved: launch latency and L2)
    rows, c, _ = synth.draw_bmmc(0, 16, accept(16))
    a = torch.arange(1 << 16, dtype=torch.int32, device=dev)
    b = torch.empty_like(a)
    with bm.Plan(rows, c, 4) as p:
        out["n16_random_int32"] = small(16, 4, lambda: p.permute(a, b, stream))
    out["n16_copy"] = small(16, 4, lambda: bm.bmmc_copy(a, b, 1 << 18, stream))
    # C2: 4096^2 fp32 transpose (n=24, 128 MiB moved: the L2's size)
    a = torch.arange(1 << 24, dtype=torch.float32, device=dev)
    b = torch.empty_like(a)
    with bm.Plan(rotate_rows(24, 12), 0, 4) as p:
        out["transpose_4096_fp32"] = small(24, 4, lambda: p.permute(a, b, stream))
    out["transpose_4096_copy"] = small(24, 4, lambda: bm.bmmc_copy(a, b, 1 << 26, stream))
    del a, b
    # C3: bit reversal n=28 int32 / int64
    a = torch.arange(1 << 28, dtype=torch.int64, device=dev)
    b = torch.empty_like(a)
    with bm.Plan(bitrev_rows(28), 0, 8) as p:
        out["bitrev_n28_int64"] = big(28, 8, lambda: p.permute(a, b, stream))
    a32 = a[: 1 << 27].view(torch.int32)
    b32 = b[: 1 << 27].view(torch.int32)
    with bm.Plan(bitrev_rows(28), 0, 4) as p:
        out["bitrev_n28_int32"] = big(28, 4, lambda: p.permute(a32, b32, stream))
    # C5: 5-D [32,64,64,64,32] fp32 perm (4,2,0,3,1), and the float4 view
    with bm.Plan(axes_rows((5, 6, 6, 6, 5), synth.FIVE_D_AXES), 0, 4) as p:
        out["dims5_fp32"] = big(28, 4, lambda: p.permute(a32, b32, stream))
    with bm.Plan(axes_rows((5, 6, 6, 6, 3), synth.FIVE_D_AXES), 0, 16) as p:
        out["dims5_float4"] = big(26, 16, lambda: p.permute(a32, b32, stream))
    # two-factor mode on seed 0 (the paper's two-kernel scheme), same algorithmic bytes
    rows, c, _ = synth.draw_bmmc(0, 28, accept(28))
    scratch = torch.empty(1 << 28, dtype=torch.int32, device=dev)
    with bm.Plan(rows, c, 4, mode=1) as p:
        out["random_n28_int32_two_factor"] = big(28, 4, lambda: p.permute_scratch(a32, b32, scratch, stream))
    # the per-element (naive) kernel of the paper's comparison: reads
    # coalesced, every write scattered (seed 0 and bit reversal)
    with bm.Plan(rows, c, 4, naive=True) as p:
        out["random_n28_int32_naive"] = big(28, 4, lambda: p.permute(a32, b32, stream))
    with bm.Plan(bitrev_rows(28), 0, 4, naive=True) as p:
        out["bitrev_n28_int32_naive"] = big(28, 4, lambda: p.permute(a32, b32, stream))
    # the n=16 random map on 4096 arrays at once (batch_log2 = 12: 1 GiB in one launch)
    rows16, c16, _ = synth.draw_bmmc(0, 16, accept(16))
    with bm.Plan(rows16, c16, 4, batch_log2=12) as p:
        out["n16_random_int32_batch4096"] = big(28, 4, lambda: p.permute(a32, b32, stream))
    # parm lowering at n=28 int32: P_A, f (here the identity), P_(A^-1): two passes,
    # algorithmic bytes of one permutation each
    mask = 0x9ABCDEF & ((1 << 28) - 1)
    A = bm.bmmc_parm_rows(28, mask)
    with bm.Plan(A, 0, 4) as pa, bm.Plan(bm.bmmc_inverse_rows(A), 0, 4) as pb:
        def parm_pass():
            pa.permute(a32, b32, stream)
            pb.permute(b32, a32, stream)
        r = big(28, 4, parm_pass)
        out["parm_lowering_n28_int32_two_permutes"] = {"gbs_per_permute": round(2 * r["gbs"], 1),
                                                        "ms_both": r["ms"]}
    # general LMAD copies: the "Impact" workloads of the Futhark copy post
    # (copy xss[:, 1:], copy xsss[:, :, 1:], copy (map reverse xss) on i32),
    # beside the page's own times with stride sorting on an AMD RX 7900 XT
    # (context, another machine), and two transposes of odd sizes
    for kind, shape in synth.LMAD_PAGE_WORKLOADS:
        w = synth.page_lmad_workload(kind, shape)
        out["lmad_" + kind + "_" + "x".join(map(str, shape)) + "_int32"] = lmad_case(
            torch, bm, w, a32, b32, stream, PAGE_US_RX7900XT[(kind, tuple(shape))])
    for name, shape, perm in (("t2d_8191x8193", (8191, 8193), (1, 0)),
                              ("batched_64x1000x1000", (64, 1000, 1000), (0, 2, 1))):
        out["lmad_" + name + "_int32"] = lmad_case(torch, bm, axes_lmad(synth, shape, perm), a32, b32, stream)
    # image layout conversions, 1- and 2-byte transposes (narrow and tile
    # kernels, the register path, a ragged last tile) and permutations of
    # 4-byte pixels and 16-byte vectors (moved as words)
    for name, shape, perm, elem in (("nhwc2nchw_32x1024x1024x3_uint8", (32, 1024, 1024, 3), (0, 3, 1, 2), 1),
                                    ("nhwc2nchw_8x512x512x64_fp16", (8, 512, 512, 64), (0, 3, 1, 2), 2),
                                    ("nhwc2nchw_8x512x512x48_fp16", (8, 512, 512, 48), (0, 3, 1, 2), 2),
                                    ("nhwc2nchw_4x512x512x100_uint8", (4, 512, 512, 100), (0, 3, 1, 2), 1),
                                    ("reverse_axes_8x512x512x48_fp16", (8, 512, 512, 48), (3, 2, 1, 0), 2),
                                    ("t2d_8192x8192_bf16", (8192, 8192), (1, 0), 2),
                                    ("t2d_16384x16384_uint8", (16384, 16384), (1, 0), 1),
                                    ("t2d_16384x16400_uint8", (16384, 16400), (1, 0), 1),
                                    ("t2d_16383x16385_uint8", (16383, 16385), (1, 0), 1),
                                    ("t2d_11585x11587_fp16", (11585, 11587), (1, 0), 2),
                                    ("swap_hw_8000x6000x4_uint8", (8000, 6000, 4), (1, 0, 2), 1),
                                    ("swap_4000x4096x16_uint8", (4000, 4096, 16), (1, 0, 2), 1),
                                    # the blocked copy: batches of small transposes, a tiny
                                    # group A, 3-byte pixels
                                    ("batched_1000000x4x5_int32", (1000000, 4, 5), (0, 2, 1), 4),
                                    ("batched_100000x12x20_int32", (100000, 12, 20), (0, 2, 1), 4),
                                    ("perm_384x4096x2x12x2_uint8", (384, 4096, 2, 12, 2), (4, 0, 2, 1, 3), 1),
                                    ("swap_hw_8000x6000x3_uint8", (8000, 6000, 3), (1, 0, 2), 1)):
        out["lmad_" + name] = lmad_case(torch, bm, axes_lmad(synth, shape, perm), a32, b32, stream, elem=elem)
    # the same slice on 1- and 2-byte elements (uint8 crop, fp16 slice: the rows kernel)
    out["lmad_slice_2d_16384x16385_uint8"] = lmad_case(
        torch, bm, synth.page_lmad_workload("slice_2d", (16384, 16385)), a32, b32, stream, elem=1)
    out["lmad_slice_2d_16384x8193_fp16"] = lmad_case(
        torch, bm, synth.page_lmad_workload("slice_2d", (16384, 8193)), a32, b32, stream, elem=2)
    del a, b, scratch, flush_buf
    torch.cuda.empty_cache()
    return out


def end_to_end(torch, bm, plans, dev, stream, nbytes, alg_bytes, steps: int = 4):
    """Same metric with the array in pinned host memory, every step (one seed
    per step) reading the host input and leaving the result in host memory.

    Two paths through the public API are timed: bmmc_permute on the host
    buffers themselves (the kernel reads and writes host memory over
    NVLink-C2C; reported as e2e) and bmmc_permute_host (cudaMemcpyAsync to
    device staging buffers, permute, copy back; reported as e2e.staged).
    Beside them, the ceiling of the direct path: bmmc_copy between the same
    two pinned host buffers (e2e.ceiling, and e2e.frac = e2e / ceiling)."""
    h_in = torch.arange(nbytes // ELEM, dtype=torch.int32).pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    d_in = torch.empty(nbytes // ELEM, dtype=torch.int32, device=dev)
    d_out = torch.empty_like(d_in)

    def timed(fn):
        fn(plans[0])
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for k in range(steps):
            fn(plans[k % len(plans)])
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / steps

    ms_direct = timed(lambda p: p.permute(h_in, h_out, stream))
    ms_staged = timed(lambda p: p.permute_host(h_in, h_out, d_in, d_out, stream))
    # the ceiling of the direct path: the copy kernel reading the same pinned
    # host input and writing the same pinned host output
    ms_ceiling = timed(lambda p: bm.bmmc_copy(h_in, h_out, nbytes, stream))
    del h_in, h_out, d_in, d_out
    direct = alg_bytes / (ms_direct / 1e3) / 1e9
    ceiling = alg_bytes / (ms_ceiling / 1e3) / 1e9
    staged = {"value": round(alg_bytes / (ms_staged / 1e3) / 1e9, 2), "unit": UNIT,
              "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes, "ms_per_step": round(ms_staged, 3),
              "path": "bmmc_permute_host (cudaMemcpyAsync pinned host -> device, permute, device -> host)"}
    return {"value": round(direct, 2), "unit": UNIT, "h2d_bytes_per_step": nbytes,
            "d2h_bytes_per_step": nbytes, "ms_per_step": round(ms_direct, 3),
            "path": "bmmc_permute on pinned host buffers: the kernel reads the host input and writes the "
                    "host output directly over NVLink-C2C",
            "ceiling": {"value": round(ceiling, 2), "unit": UNIT, "ms_per_step": round(ms_ceiling, 3),
                        "path": "bmmc_copy between the same pinned host buffers (same bytes each way)"},
            "frac": round(direct / ceiling, 4),
            "staged": staged}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=150)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="skip the other configurations")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--ref-n", type=int, default=N_BITS,
                    help="reference arm: n of the workload (default the benchmark's 28; smaller only for smoke tests)")
    ap.add_argument("--ref-sample-log2", type=int, default=0,
                    help="reference arm: log2 source indices per step (0 = sized to the step count)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
