"""Benchmark of the embedding similarity scan on GB300.

One step = one full pass of the hot path over one batch of synthetic input:
for the diversity workload, one ``dseq_run`` of B sequences x L iterations
(every iteration: contraction, min-fold, masked argmax, commit) on a table
already resident in HBM; for the BMU workload, one ``bmu_search`` of n
samples against M neurons; for the SOM epoch workload, one ``som_epoch``
(the BMU search, then the neighbourhood update of the map in place).

Prints ONE JSON line (rank 0).  ``value`` is whole-job throughput
(sequence-iterations/s, or samples/s) from CUDA events on the launching
stream around each timed step, with the L2 flushed (a 512 MB write) between
steps; ``e2e`` is the same metric through the C ABI with host buffers (the
table upload, start/pick copies inside the timed region); ``roofline`` is the
dominant kernel's algorithmic FLOP rate against the measured tensor peak;
``cpu_baseline`` is the CPU oracle timed on a bounded sample on this host.
The default line (page-1 diversity, no options) also carries ``bmu``: the
SOM 256 x 256 best-matching-unit search timed in the same run, with its own
value, roofline, end-to-end number and CPU baseline.  ``--opt
isolate_epilogue=1`` times the epilogue-isolated diversity kernel (the
contraction compiled out) and reports its running-minimum stream against
HBM.

``--impl reference`` times the CPU oracle itself as the reference arm.
Multi-GPU (torchrun): every rank runs the full workload on its own GPU
(independent replicas, weak scaling); with ``--shard`` the ranks split one
workload's sequences (or samples) and rank 0 gathers the results (strong
scaling).  Time is the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
PROFILES = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = {
    "tc_dseq_kernel": ["tc_dseq.cu", "common.cuh", "internal.h", "numeric.cuh"],
    "tc_bmu_kernel": ["tc_bmu.cu", "common.cuh", "internal.h"],
    "tc_bmu_resident_kernel": ["tc_bmu.cu", "common.cuh", "internal.h"],
    "gram_walk_kernel": ["gram.cu", "common.cuh", "internal.h"],
    "gram_walk_cluster_kernel": ["gram.cu", "common.cuh", "internal.h"],
    "gram_walk_kernel_regs": ["gram.cu", "common.cuh", "internal.h"],
}
# the longest row of running minima the one-CTA walk holds in registers
WALK_REGS_MAX_N = 17 * 128 * 4


def _walk_kernel_name(place: int, N: int) -> str:
    """The Gram walk kernel the library launches for a run whose running
    minima sat at `place` (the "walk" statistic): one CTA per sequence keeps
    rows of up to 8704 candidates in registers, longer ones in shared
    memory; place 2 is the cluster walk, place 3 the one-CTA kernel over
    global memory."""
    if place == 2:
        return "gram_walk_cluster_kernel"
    if place == 1 and N <= WALK_REGS_MAX_N:
        return "gram_walk_kernel_regs"
    return "gram_walk_kernel"


def _bmu_kernel_name(D: int, opts) -> str:
    """The BMU kernel the library launches: the resident-sample CTA-pair
    kernel for D <= 256, else the streaming one."""
    return "tc_bmu_resident_kernel" if D <= 256 and "pair=0" not in opts else "tc_bmu_kernel"


FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def _peaks():
    """(bf16 burst TF/s, bf16 sustained TF/s, HBM GB/s, source)."""
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        burst = float(p["bf16_tflops"])
        return (burst, float(p.get("bf16_tflops_sustained", burst)), float(p["hbm_gbs"]),
                "measured")
    except Exception:
        return (FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED, FALLBACK_HBM_GBS,
                "fallback")


def _kernel_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "embedding_similarity_scan_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profiled_traffic(kernel: str, workload: str, variant: str = ""):
    """DRAM bytes per launch from the committed ncu summary of this kernel,
    variant and workload, taken from the section whose source hash is the
    current kernel source's; None if there is none.  The variant ("" for the
    default launch, "_pair0" for single-CTA tensor kernels) keys the line, so
    one variant's counters never stand in for another's."""
    path = os.path.join(PROFILES, f"{kernel}.{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    current = _kernel_hash(kernel)
    marks = list(re.finditer(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text))
    for k, m in enumerate(marks):
        if m.group(1) != current:
            continue
        end = marks[k + 1].start() if k + 1 < len(marks) else len(text)
        t = re.search(rf"traffic_bytes_per_launch{variant}:\s*([0-9.eE+]+)", text[m.end():end])
        if t:
            return float(t.group(1))
    return None


def _traffic_variant(opts) -> str:
    """Key of a launch variant's traffic line: "_pair0" for the single-CTA
    tensor kernels, "_centroid" / "_f16" for the centroid criterion and
    fp16 storage (their DRAM traffic differs from the default's)."""
    v = "_pair0" if "pair=0" in opts else ""
    if "criterion=1" in opts:
        v += "_centroid"
    if "storage=1" in opts:
        v += "_f16"
    return v


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms (a page-1
    timed region of 40 steps lasts about 0.11 s)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = [r.split(", ") for r in (self.out or "").strip().splitlines() if r.strip()]
        sm, mx, reasons, watts = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                try:
                    watts.append(float(r[3]))
                except ValueError:
                    pass
                for name, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w": statistics.median(watts) if watts else None,
                "power_w_max": max(watts) if watts else None}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import oracle

    cores = os.cpu_count() or 1
    threads = oracle.threads(cores)
    if args.workload in workloads.DIVERSITY:
        cfg = workloads.DIVERSITY[args.workload]
        E = cfg.table(seed=0)
        starts = cfg.starts(seed=0)
        nseq = args.ref_sample or max(1, min(cfg.B, threads))
        sample = f"{nseq} of {cfg.B} sequences x the full L={cfg.L} per step"
        unit = "sequence-iterations/s"
        metric = "sequence-iterations/s"

        def step(i):
            sel = starts[(np.arange(nseq) + i * nseq) % cfg.B]
            oracle.dseq(E, sel, cfg.L, threads=threads)
            return nseq * cfg.L
    elif args.workload in workloads.BMU:
        cfg = workloads.BMU[args.workload]
        X = cfg.samples(seed=0)
        W = cfg.codebook(seed=0)
        # batches of 16 x threads: the oracle deals samples out in chunks of 16
        nsamp = args.ref_sample or 16 * threads
        sample = f"{nsamp} of {cfg.n} samples per step"
        unit = "samples/s"
        metric = "BMU samples/s"

        def step(i):
            lo = (i * nsamp) % cfg.n
            oracle.bmu(X[lo:lo + nsamp], W, threads=threads)
            return nsamp
    else:
        name = workloads.SOM_EPOCH[args.workload]
        cfg = workloads.BMU[name]
        sx, sy = workloads.SOM_SIDES[name]
        X = cfg.samples(seed=0)
        W = cfg.codebook(seed=0)
        bmu = np.random.default_rng(0).integers(0, cfg.M, cfg.n).astype(np.int32)
        nsamp = args.ref_sample or 16 * threads
        nneur = 16 * threads
        sample = (f"per step: BMU of {nsamp} of {cfg.n} samples and the update of {nneur} of "
                  f"{cfg.M} neurons, scaled to one epoch")
        unit = "samples/s"
        metric = "SOM epoch samples/s"

        def step(i):
            lo = (i * nsamp) % cfg.n
            t0 = time.perf_counter()
            oracle.bmu(X[lo:lo + nsamp], W, threads=threads)
            t1 = time.perf_counter()
            neur = (np.arange(nneur) * 7919 + i) % cfg.M
            oracle.som_update(X, bmu, W, sx, sy, workloads.SOM_SIGMA, workloads.SOM_RADIUS,
                              neurons=neur, threads=threads)
            t2 = time.perf_counter()
            epoch_s = (t1 - t0) / nsamp * cfg.n + (t2 - t1) / nneur * cfg.M
            # samples processed at the epoch rate during this step's wall time
            return cfg.n * (t2 - t0) / epoch_s

    for i in range(args.warmup):
        step(i)
    work = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        work += step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = work / dt
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "sample": sample},
        "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm


def _cpu_baseline(args, cfg, epoch_of=None):
    """The oracle as it stands, on all host cores, on a bounded sample.

    BMU samples are timed in batches of 16 x threads per call: the oracle
    hands samples to its threads in chunks of 16, so a smaller batch leaves
    threads idle and understates its rate."""
    import oracle

    cores = os.cpu_count() or 1
    threads = oracle.threads(cores)
    t_target = args.cpu_seconds
    if isinstance(cfg, workloads.DiversityConfig):
        E = cfg.table(seed=0)
        starts = cfg.starts(seed=0)
        # calibrate on one sequence per thread, then size the sample
        n = threads
        t0 = time.perf_counter()
        oracle.dseq(E, starts[:n], cfg.L, threads=threads)
        dt = time.perf_counter() - t0
        reps = max(1, int(t_target / max(dt, 1e-3)) - 1)
        n_total = n
        t0 = time.perf_counter()
        for r in range(reps):
            sel = starts[(np.arange(n) + (r + 1) * n) % cfg.B]
            oracle.dseq(E, sel, cfg.L, threads=threads)
            n_total += n
        dt2 = time.perf_counter() - t0
        total_t, total_n = dt + dt2, n_total
        return {"value": total_n * cfg.L / total_t, "unit": "sequence-iterations/s",
                "cores": threads, "kind": "oracle",
                "sample": f"{total_n} of {cfg.B} sequences x L={cfg.L} "
                          f"({total_t:.1f} s of CPU work)"}
    X = cfg.samples(seed=0)
    W = cfg.codebook(seed=0)
    batch = 16 * threads

    def time_bmu(budget):
        done, total = 0, 0.0
        while (total < budget or done == 0) and done + batch <= cfg.n:
            t0 = time.perf_counter()
            oracle.bmu(X[done:done + batch], W, threads=threads)
            total += time.perf_counter() - t0
            done += batch
        return done, total

    if epoch_of is not None:
        # one epoch = the BMU of every sample + the update of every neuron; time
        # a bounded sample of each and scale both to the whole epoch
        sx, sy = workloads.SOM_SIDES[epoch_of]
        bmu = np.random.default_rng(0).integers(0, cfg.M, cfg.n).astype(np.int32)
        nb, tb = time_bmu(t_target / 2)
        nu, tu, k = 0, 0.0, batch
        while (tu < t_target / 2 or nu == 0) and nu + k <= cfg.M:
            t0 = time.perf_counter()
            oracle.som_update(X, bmu, W, sx, sy, workloads.SOM_SIGMA, workloads.SOM_RADIUS,
                              neurons=np.arange(nu, nu + k), threads=threads)
            tu += time.perf_counter() - t0
            nu += k
        epoch_s = tb / nb * cfg.n + tu / nu * cfg.M
        return {"value": cfg.n / epoch_s, "unit": "samples/s", "cores": threads,
                "kind": "oracle", "bmu_samples_per_s": nb / tb,
                "sample": (f"BMU of {nb} of {cfg.n} samples in batches of {batch} ({tb:.1f} s) "
                           f"and update of {nu} of {cfg.M} neurons ({tu:.1f} s), scaled to one "
                           f"epoch ({epoch_s:.0f} s)")}
    done, total_t = time_bmu(t_target)
    return {"value": done / total_t, "unit": "samples/s", "cores": threads, "kind": "oracle",
            "sample": (f"{done} of {cfg.n} samples in batches of {batch} "
                       f"({total_t:.1f} s of CPU work)")}


@dataclasses.dataclass
class _Workload:
    """One workload as the timed loop sees it."""
    name: str
    cfg: object
    is_div: bool
    epoch_of: object
    units: int
    flop: float
    stream_bytes: object
    stream_note: str
    update_bytes: object
    kernel_name: str
    metric: str
    unit: str
    config: dict
    step: object
    e2e_step: object
    close: object
    update_ns: list
    result: object = None  # host copy of the last step's picks (or BMU indices)


def _workload(args, name, es, dev, rank, opts) -> _Workload:
    import torch

    from embedding_similarity_scan_gb300.shard import shard_range

    world = int(os.environ.get("WORLD_SIZE", "1"))
    # --shard: the ranks split one workload (its sequences or samples) with
    # no exchange on the data path; otherwise each rank runs a whole replica
    shard = args.shard and world > 1
    update_ns = []
    if name in workloads.DIVERSITY:
        cfg = workloads.DIVERSITY[name]
        if args.iters > 0:
            cfg = dataclasses.replace(cfg, L=args.iters)
        E_host = torch.from_numpy(cfg.table(seed=0)).pin_memory()
        if shard:
            lo, hi = shard_range(cfg.B, rank, world)
            starts_np = cfg.starts(seed=0)[lo:hi]
            cfg = dataclasses.replace(cfg, B=hi - lo)
        else:
            # each rank runs its own replica: the same table, its own sequences
            starts_np = cfg.starts(seed=rank)
        starts_host = torch.from_numpy(starts_np).pin_memory()
        ctx = es.dseq_create(E_host.to(dev))
        starts_dev = starts_host.to(dev)
        picks_dev = torch.empty((cfg.B, cfg.L), dtype=torch.int32, device=dev)
        if "criterion=1" in opts:
            # centroid: one held-candidate bit read per (sequence, candidate)
            stream_bytes = cfg.N * cfg.B * cfg.L / 8.0
            stream_note = "held-candidate bits read (B*N/8 bytes per iteration)"
        else:
            stream_bytes = 8.0 * cfg.N * cfg.B * cfg.L  # running-minimum read + write
            stream_note = "running-minimum read+write bytes (8*B*N per iteration)"

        def step():
            es.dseq_run(ctx, starts_dev, cfg.L, picks=picks_dev)
            return {k: es.dseq_last_stat(k)
                    for k in ("kernel_ns", "launches", "gram", "gram_ns", "walk_ns", "walk")}

        # the end-to-end leg's result buffer: pinned host memory, allocated
        # once (a caller's output array, not part of the call)
        picks_host = torch.empty((cfg.B, cfg.L), dtype=torch.int32).pin_memory()

        def e2e_step():
            c = es.dseq_create(E_host)
            try:
                es.dseq_run(c, starts_host, cfg.L, picks=picks_host)
            finally:
                c.close()
            return E_host.numel() * 4 + starts_host.numel() * 4, picks_host.numel() * 4

        return _Workload(
            name, cfg, True, None, cfg.B * cfg.L, 2.0 * cfg.N * cfg.D * cfg.B * cfg.L,
            stream_bytes, stream_note, None, "tc_dseq_kernel", "sequence-iterations/s",
            "sequence-iterations/s",
            {"workload": name, "N": cfg.N, "D": cfg.D, "B": cfg.B, "L": cfg.L,
             "l2": "flushed between steps (512 MB write)"},
            step, e2e_step, ctx.close, update_ns, lambda: picks_dev.cpu().numpy())
    if name in workloads.SOM_EPOCH:
        if shard:
            raise SystemExit("--shard: a sharded SOM epoch would need the per-neuron sums "
                             "reduced across ranks before the update; not provided")
        epoch_of = workloads.SOM_EPOCH[name]
        cfg = workloads.BMU[epoch_of]
        sx, sy = workloads.SOM_SIDES[epoch_of]
        sigma, radius = workloads.SOM_SIGMA, workloads.SOM_RADIUS
        # each rank runs its own shard: the same codebook, its own samples
        X_host = torch.from_numpy(cfg.samples(seed=rank)).pin_memory()
        W_host = torch.from_numpy(cfg.codebook(seed=0)).pin_memory()
        X_dev, W_dev = X_host.to(dev), W_host.to(dev)
        idx_dev = torch.empty(cfg.n, dtype=torch.int32, device=dev)
        dist_dev = torch.empty(cfg.n, dtype=torch.float32, device=dev)

        def step():
            # each step is the next epoch of training on the same map
            es.som_epoch(X_dev, W_dev, sx, sy, sigma, radius, bmu=idx_dev, dist=dist_dev)
            update_ns.append(es.dseq_last_stat("update_ns"))
            return {k: es.dseq_last_stat(k) for k in ("kernel_ns", "launches")}

        # the end-to-end leg trains a host copy of the same map in place, as
        # the device leg trains W_dev: pinned host buffers allocated once
        W_h = W_host.clone().pin_memory()
        idx_h = torch.empty(cfg.n, dtype=torch.int32).pin_memory()
        dist_h = torch.empty(cfg.n, dtype=torch.float32).pin_memory()

        def e2e_step():
            es.som_epoch(X_host, W_h, sx, sy, sigma, radius, bmu=idx_h, dist=dist_h)
            return (X_host.numel() + W_h.numel()) * 4, W_h.numel() * 4 + cfg.n * 8

        # the update's algorithmic bytes: read the samples and their BMUs,
        # read and write the codebook
        return _Workload(
            name, cfg, False, epoch_of, cfg.n, 2.0 * cfg.n * cfg.M * cfg.D, None, "",
            4.0 * cfg.n * cfg.D + 4.0 * cfg.n + 8.0 * cfg.M * cfg.D,
            _bmu_kernel_name(cfg.D, opts), "SOM epoch samples/s", "samples/s",
            {"workload": name, "n": cfg.n, "M": cfg.M, "D": cfg.D, "map": f"{sx}x{sy}",
             "sigma": sigma, "radius": radius, "l2": "flushed between steps (512 MB write)"},
            step, e2e_step, lambda: None, update_ns, lambda: idx_dev.cpu().numpy())
    cfg = workloads.BMU[name]
    if args.samples > 0:
        cfg = dataclasses.replace(cfg, n=args.samples)
    if shard:
        lo, hi = shard_range(cfg.n, rank, world)
        X_np = cfg.samples(seed=0)[lo:hi]
        cfg = dataclasses.replace(cfg, n=hi - lo)
    else:
        # each rank runs its own replica: the same codebook, its own samples
        X_np = cfg.samples(seed=rank)
    X_host = torch.from_numpy(np.ascontiguousarray(X_np)).pin_memory()
    W_host = torch.from_numpy(cfg.codebook(seed=0)).pin_memory()
    X_dev, W_dev = X_host.to(dev), W_host.to(dev)
    idx_dev = torch.empty(cfg.n, dtype=torch.int32, device=dev)
    dist_dev = torch.empty(cfg.n, dtype=torch.float32, device=dev)

    def step():
        es.bmu_search(X_dev, W_dev, idx=idx_dev, dist=dist_dev)
        return {k: es.dseq_last_stat(k) for k in ("kernel_ns", "launches")}

    idx_h = torch.empty(cfg.n, dtype=torch.int32).pin_memory()
    dist_h = torch.empty(cfg.n, dtype=torch.float32).pin_memory()

    def e2e_step():
        es.bmu_search(X_host, W_host, idx=idx_h, dist=dist_h)
        return (X_host.numel() + W_host.numel()) * 4, cfg.n * 8

    return _Workload(
        name, cfg, False, None, cfg.n, 2.0 * cfg.n * cfg.M * cfg.D, None, "", None,
        _bmu_kernel_name(cfg.D, opts), "BMU samples/s", "samples/s",
        {"workload": name, "n": cfg.n, "M": cfg.M, "D": cfg.D,
         "l2": "flushed between steps (512 MB write)"},
        step, e2e_step, lambda: None, update_ns, lambda: idx_dev.cpu().numpy())


def _measure(args, wl, opts, dev, local, pg, ws, flush):
    """Warm up, time args.steps steps with CUDA events (L2 flushed between
    them), then the end-to-end leg; returns the JSON line (no cpu_baseline)."""
    import torch

    stream = torch.cuda.current_stream()
    bf16_burst, bf16_sustained, hbm_peak, peak_src = _peaks()
    isolate = "isolate_epilogue=1" in opts
    config = dict(wl.config)
    if opts:
        config["options"] = list(opts)
    shrunk = args.iters > 0 or args.samples > 0
    if shrunk:
        config["reduced"] = "smaller than the workload (--iters / --samples): a profiling case"
    if isolate:
        config["isolated_epilogue"] = ("contraction compiled out (picks meaningless): measures "
                                       "the running-minimum stream of the fused epilogue alone")

    def barrier():
        torch.cuda.synchronize()
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        wl.step()
        flush.zero_()
    barrier()
    wl.update_ns.clear()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    stats = []
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            ev[i][0].record(stream)
            stats.append(wl.step())
            ev[i][1].record(stream)
            flush.zero_()
        barrier()
        t_wall = time.perf_counter() - t_wall
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = sum(step_ms)
    if pg is not None:
        t = torch.tensor([total_ms], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        total_ms = float(t.item())
    units_all = ws * wl.units
    if pg is not None and args.shard:
        # strong scaling: the ranks' shares of one workload add up
        t = torch.tensor([float(wl.units)], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.SUM)
        units_all = float(t.item())
    value = units_all * args.steps / (total_ms / 1e3)

    # end to end through the C ABI with host buffers
    e2e_steps = max(1, min(args.steps, 3))
    wl.e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        h2d, d2h = wl.e2e_step()
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    if pg is not None:
        t = torch.tensor([e2e_s], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        e2e_s = float(t.item())
    e2e_value = units_all * e2e_steps / e2e_s

    kernel_ns = [st["kernel_ns"] for st in stats]
    launches = sum(st["launches"] for st in stats)
    k_avg_s = statistics.mean(kernel_ns) / 1e9 if kernel_ns and min(kernel_ns) > 0 else None
    gram = bool(stats) and all(st.get("gram", 0) == 1 for st in stats)
    achieved = wl.flop / k_avg_s / 1e12 if k_avg_s else None
    clocks = clk.summary()
    # a run held at the power cap is compared with the sustained tensor peak
    # (cuBLAS run back to back under the cap), otherwise with the burst peak
    capped = "sw_power_cap" in clocks["reasons"]
    bf16_peak = bf16_sustained if capped else bf16_burst
    peak_kind = "sustained" if capped else "burst"
    # fp32-equivalent tensor peak of the split contraction: three fp16 MMAs per
    # fp32 multiply-add (fp16 and bf16 run at the same nominal rate)
    split_peak = bf16_peak / 3.0
    fp16_storage = wl.is_div and "storage=1" in opts
    if fp16_storage:
        # one fp16 product per multiply-add: the plain fp16 (= bf16 nominal)
        # peak; the centroid query keeps two parts (hi*2^12, lo), two products
        nprod = 2 if "criterion=1" in opts else 1
        tensor_peak = bf16_peak / nprod
        burst_peak = bf16_burst / nprod
        peak_note = (f"peak = {peak_src} bf16 {peak_kind} {bf16_peak:.1f} TFLOP/s"
                     + (f" / {nprod} ({nprod} fp16 MMAs" if nprod > 1 else " (one fp16 MMA")
                     + " per multiply-add)")
    else:
        tensor_peak = split_peak
        burst_peak = bf16_burst / 3.0
        peak_note = (f"peak = {peak_src} bf16 {peak_kind} {bf16_peak:.1f} TFLOP/s / 3 (three "
                     f"fp16 MMAs per fp32 multiply-add); {peak_kind} because the clock "
                     f"sampler {'saw' if capped else 'did not see'} sw_power_cap")
    roof = {"bound": "tensor", "achieved": achieved, "peak": tensor_peak, "unit": "TFLOP/s",
            "frac": (achieved / tensor_peak) if achieved else None,
            "peak_kind": peak_kind,
            "frac_of_burst": (achieved / burst_peak) if achieved else None,
            "traffic": None if (shrunk or isolate) else _profiled_traffic(
                wl.kernel_name, wl.epoch_of or wl.name, _traffic_variant(opts)),
            "kernel": wl.kernel_name,
            "note": (f"achieved = algorithmic FLOP (2*{'N*D*B*L' if wl.is_div else 'n*M*D'})"
                     f" / kernel time (CUDA events on the launching stream); {peak_note}")}
    if "engine=1" in opts:
        # the plain fp32 SIMT variant: bound by the FP32 pipe, 128 fp32 FMA
        # lanes per SM, 2 FLOP each, at the maximum SM clock
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = clocks.get("sm_max_mhz") or 2070.0
        alu_peak = sms * 128 * 2 * mhz * 1e6 / 1e12
        roof.update({"bound": "alu", "peak": alu_peak,
                     "frac": (achieved / alu_peak) if achieved else None,
                     "peak_kind": "fp32 pipe, derived", "frac_of_burst": None, "traffic": None,
                     "kernel": "ffma_dseq_fold_kernel" if wl.is_div else "ffma_bmu_kernel",
                     "note": (f"achieved = algorithmic FLOP / kernel time "
                              f"({'fold + commit launches' if wl.is_div else 'one launch'}, "
                              f"CUDA events); peak = {sms} SMs x 128 FP32 lanes x 2 FLOP x "
                              f"{mhz:.0f} MHz (derived, not measured)")})
    if wl.stream_bytes is not None and k_avg_s:
        hbm_achieved = wl.stream_bytes / k_avg_s / 1e9
        if isolate or hbm_achieved / hbm_peak > (roof["frac"] or 0.0):
            # the min-distance stream binds (or is all the isolated kernel
            # does): report the HBM roofline instead
            roof.update({"bound": "hbm", "achieved": hbm_achieved, "peak": hbm_peak,
                         "unit": "GB/s", "frac": hbm_achieved / hbm_peak, "peak_kind": "copy",
                         "frac_of_burst": None,
                         "tensor_frac": None if isolate else roof["frac"],
                         "note": (f"achieved = {wl.stream_note} / kernel time; peak = "
                                  f"{peak_src} copy bandwidth {hbm_peak:.1f} GB/s")})
    gram_product = None
    if gram:
        # the Gram engine: the walk streams one row of G per sequence-iteration
        # (plus the running minima when they live in global memory, not on
        # chip in one CTA or a cluster); the Gram product is
        # tensor-bound and reported beside it
        cfg = wl.cfg
        place = stats[0]["walk"]
        m_global = place == 3
        walk_kernel = _walk_kernel_name(place, cfg.N)
        # reads only: a running minimum is written back only where it fell
        walk_bytes = cfg.B * cfg.L * cfg.N * (4.0 + (4.0 if m_global else 0.0))
        walk_s = statistics.mean(st["walk_ns"] for st in stats) / 1e9
        gram_s = statistics.mean(st["gram_ns"] for st in stats) / 1e9
        # the distinct dot products of the symmetric product: N (N + 1) / 2
        gflop = 1.0 * cfg.N * (cfg.N + 1) * cfg.D
        roof = {"bound": "hbm", "achieved": walk_bytes / walk_s / 1e9, "peak": hbm_peak,
                "unit": "GB/s", "frac": walk_bytes / walk_s / 1e9 / hbm_peak, "peak_kind": "copy",
                "traffic": None if shrunk else _profiled_traffic(walk_kernel, wl.name),
                "kernel": walk_kernel,
                "note": (f"achieved = algorithmic bytes of the walk (one row of G, 4*N bytes, per "
                         f"sequence-iteration{' + the running minima read, 4*N; writes of the minima that fell are not counted' if m_global else ''})"
                         f" / walk kernel time (CUDA events); peak = {peak_src} copy bandwidth "
                         f"{hbm_peak:.1f} GB/s; L2 serves the rows that many sequences read in "
                         f"the same stretch of iterations, so frac can exceed 1 where G is not far "
                         f"above L2 (traffic = the DRAM bytes of one launch, from ncu)")}
        gram_product = {"bound": "tensor", "achieved": gflop / gram_s / 1e12, "peak": tensor_peak,
                        "unit": "TFLOP/s", "frac": gflop / gram_s / 1e12 / tensor_peak,
                        "peak_kind": peak_kind, "frac_of_burst": gflop / gram_s / 1e12 / burst_peak,
                        "ms": gram_s * 1e3, "share_of_step": gram_s * 1e3 / (total_ms / args.steps),
                        "kernel": "tc_bmu_kernel (Gram store epilogue)",
                        "note": ("achieved = N*(N+1)*D (2*D FLOP for each of the N*(N+1)/2 "
                                 "distinct entries of the symmetric G) / time of the operand split "
                                 f"and the Gram product (CUDA events); {peak_note}")}
    line = {
        "metric": wl.metric, "value": value, "unit": wl.unit, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "strong" if (pg is not None and args.shard) else "weak", "vs_baseline": None,
        "dtype": ("f32 (FFMA)" if "engine=1" in opts
                  else "f16 storage, f32 accumulate" if fp16_storage
                  else "fp16x3-split (fp32-accurate), f32 accumulate"),
        "data": "synthetic", "config": config, "roofline": roof,
        "e2e": {"value": e2e_value, "unit": wl.unit, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": int(launches), "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    if gram_product is not None:
        line["engine"] = "gram"
        line["gram_product"] = gram_product
        line["dtype"] = "fp16x3-split Gram product (fp32-accurate), f32 walk"
    if wl.stream_bytes is not None and k_avg_s and not gram:
        line["min_distance_stream"] = {
            "achieved_gbs": wl.stream_bytes / k_avg_s / 1e9, "peak_gbs": hbm_peak,
            "frac": wl.stream_bytes / k_avg_s / 1e9 / hbm_peak,
            "note": f"{wl.stream_note} / kernel time"
                    + (" (epilogue-isolated kernel)" if isolate else " (fused kernel)")}
    if wl.epoch_of is not None and wl.update_ns and min(wl.update_ns) > 0:
        u_s = statistics.mean(wl.update_ns) / 1e9
        line["som_update"] = {
            "achieved_gbs": wl.update_bytes / u_s / 1e9, "peak_gbs": hbm_peak,
            "frac": wl.update_bytes / u_s / 1e9 / hbm_peak, "ms": u_s * 1e3,
            "share_of_step": u_s * 1e3 / (total_ms / args.steps),
            "note": ("neighbourhood update kernels: algorithmic bytes (samples + BMUs read, "
                     "codebook read + write) / their CUDA-event time")}
    return line


# the BMU half of the metric, measured beside the default diversity line
BMU_BESIDE = "som256"


def run_ours(args):
    import torch

    opts = list(args.opt)
    if any(o.split("=")[0] in ("isolate_epilogue", "fault_skip_arrive", "fault_skip_copy")
           for o in opts):
        # the library accepts its measurement options only when opted in
        os.environ["DSEQ_ENABLE_TEST_OPTIONS"] = "1"
    import embedding_similarity_scan_gb300 as es

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    es.load()
    for kv in opts:
        k, v = kv.split("=")
        es.dseq_set_option(k, int(v))
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    wl = _workload(args, args.workload, es, dev, rank, opts)
    line = _measure(args, wl, opts, dev, local, pg, ws, flush)
    if pg is not None and args.shard:
        # the host-side gather that completes a sharded run (outside the
        # timed region): every rank's picks (or BMU indices) in rank order
        from embedding_similarity_scan_gb300.shard import gather_rows

        rows = gather_rows(wl.result())
        line["shard"] = {"ranks": ws, "gathered_rows": int(rows.shape[0]),
                         "note": "contiguous shares of one workload, results gathered on the host"}
    wl.close()
    default_line = not opts and args.workload == "page1" and args.iters == 0
    if default_line and line.get("engine") == "gram" and args.with_scan:
        # the per-iteration contraction kernel on the same workload, timed in
        # the same run (the library picks the Gram engine for this shape)
        es.dseq_set_option("gram", 0)
        sw = _workload(args, args.workload, es, dev, rank, opts)
        sc = _measure(args, sw, opts, dev, local, pg, ws, flush)
        sw.close()
        es.dseq_set_option("gram", 2)
        keep = ("value", "unit", "ms_per_step", "dtype", "roofline", "min_distance_stream",
                "gpu_launches", "clocks", "wall_s_timed_region")
        line["scan"] = {k: sc[k] for k in keep if k in sc}
        line["scan"]["note"] = ("the per-iteration contraction kernel (option gram=0) on the "
                                "same workload and sequences")
    with_cpu = rank == 0 and ws == 1 and not args.no_cpu_baseline
    if with_cpu and "isolate_epilogue=1" not in opts:
        line["cpu_baseline"] = _cpu_baseline(args, wl.cfg, wl.epoch_of)
    # the default line also carries the BMU half of the metric: the SOM
    # 256 x 256 search timed in the same run, with its own roofline and CPU
    # baseline
    if args.with_bmu and default_line:
        bw = _workload(args, BMU_BESIDE, es, dev, rank, opts)
        b = _measure(args, bw, opts, dev, local, pg, ws, flush)
        bw.close()
        keep = ("metric", "value", "unit", "ms_per_step", "steps", "warmup", "dtype", "config",
                "roofline", "e2e", "gpu_launches", "clocks", "wall_s_timed_region")
        line["bmu"] = {k: b[k] for k in keep}
        if with_cpu:
            line["bmu"]["cpu_baseline"] = _cpu_baseline(args, bw.cfg, None)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="page1",
                    choices=sorted(workloads.DIVERSITY) + sorted(workloads.BMU)
                    + sorted(workloads.SOM_EPOCH))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--iters", type=int, default=0,
                    help="diversity workloads: L iterations instead of the workload's (small "
                         "cases for profiling; the line is then not the workload's)")
    ap.add_argument("--samples", type=int, default=0,
                    help="BMU workloads: this many samples instead of the workload's (as --iters)")
    ap.add_argument("--ref-sample", type=int, default=0)
    ap.add_argument("--opt", action="append", default=[],
                    help="library option name=value, e.g. storage=1 (process-wide)")
    ap.add_argument("--shard", action="store_true",
                    help="under torchrun: split one workload's sequences (or samples) across "
                         "the ranks (strong scaling) instead of a replica per rank")
    ap.add_argument("--no-scan", dest="with_scan", action="store_false",
                    help="leave out the per-iteration kernel's measurement that the default "
                         "page-1 line carries beside the Gram engine's")
    ap.add_argument("--no-bmu", dest="with_bmu", action="store_false",
                    help="leave out the BMU search (som256) that the default page-1 line "
                         "carries beside the diversity number")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
