#!/usr/bin/env python3
"""Benchmark of the quaternion cumulative-product scan, forward + backward.

One step = one forward scan (``quat_cumprod_fwd``) and one backward
(``quat_cumprod_bwd``) over one batch of seeded synthetic inputs, through the C
ABI.  Metric: elements per second, elements = B*S*H*J, with inputs resident in
HBM when the timed region starts; ``e2e`` is the same metric with the inputs
copied from pinned host memory and the outputs copied back inside each step.

``--impl reference`` times the fp64 CPU oracle (the only reference
implementation of this scan) on the host cores, on a bounded lane sample of the
same workload.

Multi-GPU (torchrun): every rank runs its own independent batch (lanes are
independent; no collective on the data path), timing is the max over ranks,
``value`` is the total over ranks (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from quaternion_cumulative_product_gb300 import workloads  # noqa: E402

METRIC = "quat-scan fwd+bwd elements/s (B*S*H*J)"
UNIT = "elements/s"
DEFAULT_WORKLOAD = "mamba3"
FWD_BYTES_PER_ELEMENT = 32      # read q, write cum
BWD_BYTES_PER_ELEMENT = 48      # read q and d_cum, write d_q
STEP_BYTES = FWD_BYTES_PER_ELEMENT + BWD_BYTES_PER_ELEMENT
L2_BYTES = 126 * (1 << 20)
# Every timed loop starts right after a synchronize, on an idle GPU. A device-side
# spin of about 300 us (at 2.07 GHz; longer at lower clocks) goes ahead of its
# first event, so that the first step's interval does not also hold the host's
# time to enqueue the first call. The spin touches no memory: L2 still holds
# what the previous kernel left, as it does before every later step.
LEAD_SPIN_CYCLES = 600_000
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
TRAFFIC_NOTE = ("dram__bytes_read.sum + dram__bytes_write.sum of one launch of the call's kernels, each captured "
                "alone by ncu (profiles/dram_traffic.txt, null unless the kernel sources hash to the captured "
                "source); inside the step the backward also writes back the lines the forward left dirty in L2")
KERNEL_SOURCES = [os.path.join(ROOT, "quaternion_cumulative_product_gb300", "csrc", f)
                  for f in ("quat_scan.cu", "quat_device.cuh", "quat_common.cuh", "quat_tiles.cuh",
                            "quat_chain.cuh", "quat_walk.cuh", "quat_segwalk.cuh", "quat_segwalk_ws.cuh", "quat_segwalk_bwd.cuh",
                            "quat_segwalk_tab.cuh", "quat_short.cuh")]


# Forward configurations of the segmented chained walk in the library's table.
SEGWALK_FWD_VARIANTS = (9, 10, 11, 12, 13, 14, 15, 16, 17, 18, 19, 20, 21, 22, 23, 24)


# Backward configurations of the segmented walk (after its carries-only pass
# when the carries are recomputed).
SEGWALK_BWD_VARIANTS = tuple(range(11, 25)) + (30, 31, 32, 33)
SHORT_FWD_VARIANTS = SHORT_BWD_VARIANTS = (25, 26, 27, 28, 29)


def design_name(call: str, kernels: int, variant: int = -1) -> str:
    if variant in (SHORT_BWD_VARIANTS if call.startswith("quat_cumprod_bwd") else SHORT_FWD_VARIANTS):
        return f"{call} (short-sequence kernel: the whole sequence of a few lanes in one CTA)"
    if call == "quat_cumprod_fwd" and variant in SEGWALK_FWD_VARIANTS:
        return f"{call} (segmented chained walk kernel)"
    if call == "quat_cumprod_bwd" and variant in SEGWALK_BWD_VARIANTS:
        return f"{call} (carries pass + segmented walk kernels)" if kernels == 2 else f"{call} (segmented walk kernel)"
    if kernels != 1:
        return f"{call} (aggregate + carry + apply kernels)"
    return f"{call} (walk kernel)"


def _code_only(text: str) -> str:
    """The source without comments and blank lines (a comment edit changes no kernel)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current source."""
    try:
        with open(TRAFFIC_FILE) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 4 and parts[0] == kernel and parts[1] == workload:
                    fields = dict(p.split("=", 1) for p in parts[2:] if "=" in p)
                    if fields.get("source_hash") == kernel_source_hash():
                        return float(fields["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


# ---------------------------------------------------------------------------
# Distributed helpers (host logic; tested with gloo on CPU).
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return world, rank, local


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own independent batch (weak scaling)."""
    return base_seed + 1000 * rank


def lead_spin() -> None:
    """Keeps the current stream busy while the host enqueues a timed loop's first step."""
    import torch
    torch.cuda._sleep(LEAD_SPIN_CYCLES)


def weak_scaling_value(world: int, elements_per_rank: int, step_ms: float) -> float:
    """Whole-job elements/s: every rank processes its own batch in ``step_ms`` (max over ranks)."""
    return world * elements_per_rank / (step_ms * 1e-3)


def reduce_max(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# Clocks sampler (nvidia-smi during the timed region).
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="qs_clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        loaded = [s for s, p in zip(sm, pw) if p is not None and p > 200] or sm
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded lane sample).
# ---------------------------------------------------------------------------
def oracle_sample(w, max_lanes: int, arrays=None):
    """A bounded lane sample of workload ``w`` for the CPU oracle (fp64 arrays)."""
    import numpy as np
    if arrays is None:
        arrays = workloads.make_inputs(w) if w.elements <= (1 << 26) else _sample_inputs(w, max_lanes)
    q, init, d_cum = arrays
    H, J = q.shape[2], q.shape[3]
    avail = q.shape[0] * H * J
    lanes = min(max_lanes, avail)
    rng = np.random.default_rng(0)
    pick = np.sort(rng.choice(avail, lanes, replace=False))
    sq, si, sd = workloads.sample_lanes((q, init, d_cum), pick, H, J)
    return tuple(a.astype(np.float64) for a in (sq, si, sd)), lanes


def time_oracle(sample, target_s: float):
    """Runs oracle fwd+bwd on the sample until ``target_s`` elapsed (at least once).

    Returns (elements/s, threads used, repetitions, seconds).
    """
    import oracle
    sq, si, sd = sample
    cores = os.cpu_count() or 1
    done, elapsed, reps = 0, 0.0, 0
    while elapsed < target_s or reps == 0:
        t0 = time.perf_counter()
        oracle.fwd(sq, si, nthreads=cores)
        oracle.bwd(sq, si, sd, nthreads=cores)
        elapsed += time.perf_counter() - t0
        done += sq.shape[1] * sq.shape[2]
        reps += 1
    return done / elapsed, cores, reps, elapsed


def sample_description(w, lanes, reps, cores):
    return (f"{lanes} of {w.lanes} lanes (full S={w.S}) of {w.describe()}, fwd+bwd, "
            f"{reps} repetition(s), fp64 C oracle, {cores} threads")


def _sample_inputs(w, max_lanes):
    # Workloads too large to draw on the host in full: the same recipe on fewer
    # batch entries (same distributions and seed).
    B = max(1, min(w.B, max_lanes // max(1, w.H * w.J)))
    small = workloads.custom(w.name, B, w.S, w.H, w.J, q_kind=w.q_kind, theta_max=w.theta_max,
                             init_kind=w.init_kind, dcum_sigma=w.dcum_sigma, seed=w.seed)
    return workloads.make_inputs(small)


# ---------------------------------------------------------------------------
# Arms.
# ---------------------------------------------------------------------------
def run_reference(args, w, world, rank):
    if rank != 0:
        return 0
    sample, lanes = oracle_sample(w, args.cpu_lanes)
    for _ in range(args.warmup):
        time_oracle(sample, 0.0)
    rates, t_all, reps_all, cores = [], 0.0, 0, os.cpu_count() or 1
    for _ in range(args.steps):
        rate, cores, reps, secs = time_oracle(sample, 0.0)
        rates.append(rate)
        t_all += secs
        reps_all += reps
    value = sum(rates) / len(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_all / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generator, workloads.py)",
        "config": {"workload": w.describe(), "B": w.B, "S": w.S, "H": w.H, "J": w.J,
                   "elements": w.elements},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample_description(w, lanes, 1, cores) + " per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def time_other_workload(qs, torch, name, dev, stream, steps, warmup, peak):
    """The step, each call alone and the saved-carries step of another workload.

    Inputs are drawn on the device (``workloads.make_inputs_device``: the same
    distributions as the seeded table, torch's generator); L2 is flushed by a
    read before every step and every rep when a tensor is smaller than twice
    the L2 size.
    """
    wl = workloads.WORKLOADS[name]
    E = wl.elements
    q, init, d_cum = workloads.make_inputs_device(wl, dev)
    cum, d_q, d_init = torch.empty_like(q), torch.empty_like(q), torch.empty_like(init)
    carries = torch.empty((wl.B, (wl.S + qs.QS_CARRY_STEPS - 1) // qs.QS_CARRY_STEPS, wl.H, wl.J, 4),
                          dtype=torch.float32, device=dev)
    flush = q.numel() * 4 < 2 * L2_BYTES
    flushbuf = torch.ones(2 * L2_BYTES // 4, device=dev)

    def fwd():
        qs.quat_cumprod_fwd(q, init, cum)

    def bwd():
        qs.quat_cumprod_bwd(q, init, d_cum, d_q, d_init)

    def cfwd():
        qs.quat_cumprod_fwd_carries(q, init, cum, carries)

    def cbwd():
        qs.quat_cumprod_bwd_carries(q, carries, d_cum, d_q, d_init)

    def steps_of(a, b):
        for _ in range(warmup):
            a()
            b()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        torch.cuda.synchronize(dev)
        lead_spin()
        for e0, e1, e2 in ev:
            if flush:
                flushbuf.sum()
            e0.record(stream)
            a()
            e1.record(stream)
            b()
            e2.record(stream)
        torch.cuda.synchronize(dev)
        return (statistics.mean(x.elapsed_time(y) for x, y, _ in ev),
                statistics.mean(y.elapsed_time(z) for _, y, z in ev))

    def alone(calls, reps=20):
        ms = []
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(reps):
            flushbuf.sum()
            a0.record(stream)
            for c in calls:
                c()
            a1.record(stream)
            a1.synchronize()
            ms.append(a0.elapsed_time(a1))
        return statistics.median(ms)

    fwd_ms, bwd_ms = steps_of(fwd, bwd)
    al = {"fwd": alone([fwd]), "bwd": alone([bwd]), "fwd_bwd": alone([fwd, bwd])}
    cf_ms, cb_ms = steps_of(cfwd, cbwd)
    st = qs.quat_cumprod_status(device=dev)
    if st != qs.QS_OK:
        raise RuntimeError(f"device status after workload {name}: {qs.quat_cumprod_strerror(st)}")

    def frac(nbytes, ms):
        return nbytes * E / (ms * 1e-3) / 1e9 / peak

    plans = {c: qs.quat_cumprod_plan(c, wl.B, wl.S, wl.H, wl.J, device=dev)
             for c in ("fwd", "bwd", "fwd_carries", "bwd_carries")}
    return {
        "config": wl.describe(), "elements": E, "steps": steps,
        "l2": "flushed by a read before every step" if flush else "inputs larger than L2, no flush",
        "inputs": "drawn on the device (workloads.make_inputs_device, seed %d)" % wl.seed,
        "step": {"fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "ms": fwd_ms + bwd_ms,
                 "value": E / ((fwd_ms + bwd_ms) * 1e-3), "unit": UNIT,
                 "fwd_frac": frac(FWD_BYTES_PER_ELEMENT, fwd_ms), "bwd_frac": frac(BWD_BYTES_PER_ELEMENT, bwd_ms),
                 "step_frac": frac(STEP_BYTES, fwd_ms + bwd_ms)},
        "alone": {k: {"ms": v, "frac": frac(nb, v)} for k, v, nb in
                  (("fwd", al["fwd"], FWD_BYTES_PER_ELEMENT), ("bwd", al["bwd"], BWD_BYTES_PER_ELEMENT),
                   ("fwd_bwd", al["fwd_bwd"], STEP_BYTES))},
        "saved_carries": {"fwd_ms": cf_ms, "bwd_ms": cb_ms, "value": E / ((cf_ms + cb_ms) * 1e-3),
                          "bwd_frac": frac(BWD_BYTES_PER_ELEMENT, cb_ms)},
        "plan": {c: {"variant": v, "kernels": k} for c, (v, k) in plans.items()},
    }


def run_ours(args, w, world, rank, local):
    import numpy as np
    import torch
    import torch.distributed as dist

    import quaternion_cumulative_product_gb300 as qs

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device (the scan has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=dev)
    qs.load_library()

    wr = workloads.custom(w.name, w.B, w.S, w.H, w.J, q_kind=w.q_kind, theta_max=w.theta_max,
                          init_kind=w.init_kind, dcum_sigma=w.dcum_sigma, seed=rank_seed(w.seed, rank))
    q_np, init_np, dcum_np = workloads.make_inputs(wr)
    q = torch.from_numpy(q_np).to(dev)
    init = torch.from_numpy(init_np).to(dev)
    d_cum = torch.from_numpy(dcum_np).to(dev)
    cum = torch.empty_like(q)
    d_q = torch.empty_like(q)
    d_init = torch.empty_like(init)
    tensor_bytes = q.numel() * 4
    flush = tensor_bytes < 2 * L2_BYTES
    # L2 flush by READING a buffer of twice its size: evicts the inputs without
    # leaving dirty lines for the timed kernels to write back.
    flushbuf = torch.ones(2 * L2_BYTES // 4, device=dev)
    stream = torch.cuda.current_stream(dev)
    launches = [0]
    # The library picks one design per call (a single walk kernel, or the
    # aggregate / carry / apply kernels); count the kernels it launches.
    fwd_variant, fwd_kernels = qs.quat_cumprod_plan(False, w.B, w.S, w.H, w.J, device=dev)
    bwd_variant, bwd_kernels = qs.quat_cumprod_plan(True, w.B, w.S, w.H, w.J, device=dev)
    kernels_per_step = fwd_kernels + bwd_kernels

    def step():
        qs.quat_cumprod_fwd(q, init, cum)
        qs.quat_cumprod_bwd(q, init, d_cum, d_q, d_init)
        launches[0] += kernels_per_step

    for _ in range(args.warmup):
        step()
    st = qs.quat_cumprod_status(device=dev)
    if st != qs.QS_OK:
        raise RuntimeError(f"device status after warm-up: {qs.quat_cumprod_strerror(st)}")
    # Whether a second step on the same inputs gives bitwise the same outputs
    # (outside the timed region).
    first = (cum.clone(), d_q.clone(), d_init.clone())
    step()
    torch.cuda.synchronize(dev)
    repeatable = all(torch.equal(a, b) for a, b in zip(first, (cum, d_q, d_init)))
    del first

    # ---- device-timed region -------------------------------------------------
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    torch.cuda.synchronize(dev)
    barrier(dev)
    sampler.start()
    launches[0] = 0
    torch.cuda.synchronize(dev)
    lead_spin()
    for i in range(args.steps):
        if flush:
            flushbuf.sum()
        e0, e1, e2 = ev[i]
        e0.record(stream)
        qs.quat_cumprod_fwd(q, init, cum)
        e1.record(stream)
        qs.quat_cumprod_bwd(q, init, d_cum, d_q, d_init)
        e2.record(stream)
        launches[0] += kernels_per_step
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    barrier(dev)
    st = qs.quat_cumprod_status(device=dev)
    if st != qs.QS_OK:
        raise RuntimeError(f"device status after timed region: {qs.quat_cumprod_strerror(st)}")
    fwd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    bwd_ms = [b.elapsed_time(c) for _, b, c in ev]
    step_ms_local = sum(f + b for f, b in zip(fwd_ms, bwd_ms)) / args.steps
    step_ms = reduce_max(step_ms_local, dev)
    E = w.elements
    value = weak_scaling_value(world, E, step_ms)

    # ---- each call alone: median over reps, with L2 flushed before every rep
    # by READING a buffer of twice its size, so that no dirty line of earlier
    # work is left for the timed call to write back ---------------------------
    alone_reps = max(20, args.steps)

    def alone(calls):
        ms = []
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        for _ in range(alone_reps):
            flushbuf.sum()
            a0.record(stream)
            for c in calls:
                c()
            a1.record(stream)
            a1.synchronize()
            ms.append(a0.elapsed_time(a1))
        return statistics.median(ms)

    def run_fwd():
        qs.quat_cumprod_fwd(q, init, cum)

    def run_bwd():
        qs.quat_cumprod_bwd(q, init, d_cum, d_q, d_init)

    torch.cuda.synchronize(dev)
    barrier(dev)
    alone_ms = {"fwd": alone([run_fwd]), "bwd": alone([run_bwd]), "fwd_bwd": alone([run_fwd, run_bwd])}
    st = qs.quat_cumprod_status(device=dev)
    if st != qs.QS_OK:
        raise RuntimeError(f"device status after the calls alone: {qs.quat_cumprod_strerror(st)}")
    alone_ms = {k: reduce_max(v, dev) for k, v in alone_ms.items()}

    # ---- the same step with saved chunk carries (forward writes them, the
    # backward starts from them instead of recomputing the forward) ----------
    carries = torch.empty((w.B, (w.S + qs.QS_CARRY_STEPS - 1) // qs.QS_CARRY_STEPS, w.H, w.J, 4),
                          dtype=torch.float32, device=dev)
    cfwd_kernels = qs.quat_cumprod_plan("fwd_carries", w.B, w.S, w.H, w.J, device=dev)[1]
    cbwd_kernels = qs.quat_cumprod_plan("bwd_carries", w.B, w.S, w.H, w.J, device=dev)[1]
    for _ in range(args.warmup):
        qs.quat_cumprod_fwd_carries(q, init, cum, carries)
        qs.quat_cumprod_bwd_carries(q, carries, d_cum, d_q, d_init)
    cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    barrier(dev)
    lead_spin()
    for i in range(args.steps):
        if flush:
            flushbuf.sum()
        e0, e1, e2 = cev[i]
        e0.record(stream)
        qs.quat_cumprod_fwd_carries(q, init, cum, carries)
        e1.record(stream)
        qs.quat_cumprod_bwd_carries(q, carries, d_cum, d_q, d_init)
        e2.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dev)
    st = qs.quat_cumprod_status(device=dev)
    if st != qs.QS_OK:
        raise RuntimeError(f"device status after the saved-carries region: {qs.quat_cumprod_strerror(st)}")
    cfwd_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in cev)
    cbwd_ms = statistics.mean(b.elapsed_time(c) for _, b, c in cev)
    cstep_ms = reduce_max(cfwd_ms + cbwd_ms, dev)
    del carries

    # ---- the same step with bfloat16 tensors (fp32 arithmetic) ---------------
    bq, bi, bd = q.to(torch.bfloat16), init.to(torch.bfloat16), d_cum.to(torch.bfloat16)
    bcum, bdq, bdi = torch.empty_like(bq), torch.empty_like(bq), torch.empty_like(bi)
    even = (w.H * w.J) % 2 == 0
    bf16_kernels = (qs.quat_cumprod_plan("fwd_bf16", w.B, w.S, w.H, w.J, device=dev)[1]
                    + qs.quat_cumprod_plan("bwd_bf16", w.B, w.S, w.H, w.J, device=dev)[1]) if even else 0
    if even:
        for _ in range(args.warmup):
            qs.quat_cumprod_fwd_bf16(bq, bi, bcum)
            qs.quat_cumprod_bwd_bf16(bq, bi, bd, bdq, bdi)
        bev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        torch.cuda.synchronize(dev)
        barrier(dev)
        lead_spin()
        for i in range(args.steps):
            if flush:
                flushbuf.sum()
            e0, e1, e2 = bev[i]
            e0.record(stream)
            qs.quat_cumprod_fwd_bf16(bq, bi, bcum)
            e1.record(stream)
            qs.quat_cumprod_bwd_bf16(bq, bi, bd, bdq, bdi)
            e2.record(stream)
        torch.cuda.synchronize(dev)
        barrier(dev)
        st = qs.quat_cumprod_status(device=dev)
        if st != qs.QS_OK:
            raise RuntimeError(f"device status after the bf16 region: {qs.quat_cumprod_strerror(st)}")
        bfwd_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in bev)
        bbwd_ms = statistics.mean(b.elapsed_time(c) for _, b, c in bev)
        bstep_ms = reduce_max(bfwd_ms + bbwd_ms, dev)
    del bq, bi, bd, bcum, bdq, bdi

    # ---- end to end through the public API with pinned host buffers ---------
    h_q = torch.from_numpy(q_np).pin_memory()
    h_init = torch.from_numpy(init_np).pin_memory()
    h_dcum = torch.from_numpy(dcum_np).pin_memory()
    o_cum = torch.empty(q.shape, dtype=torch.float32).pin_memory()
    o_dq = torch.empty(q.shape, dtype=torch.float32).pin_memory()
    o_di = torch.empty(init.shape, dtype=torch.float32).pin_memory()

    # One call of the C ABI on host buffers per step: the library cuts the
    # batch into slices whose copies in and out overlap the kernels.
    def e2e_step():
        qs.quat_cumprod_fwd_bwd_host(h_q, h_init, h_dcum, o_cum, o_dq, o_di, device=dev, stream=stream,
                                     synchronize=False)

    del cum, d_q
    for _ in range(min(args.warmup, 3)):
        e2e_step()
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    torch.cuda.synchronize(dev)
    barrier(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(a.elapsed_time(b) / e2e_steps, dev)
    st = qs.quat_cumprod_status(device=dev)
    if st != qs.QS_OK:
        raise RuntimeError(f"device status after e2e: {qs.quat_cumprod_strerror(st)}")
    h2d = (h_q.numel() + h_init.numel() + h_dcum.numel()) * 4
    d2h = (o_cum.numel() + o_dq.numel() + o_di.numel()) * 4

    peak, peak_src = measured_peak_hbm()
    # The other roofline-judged workloads, on one GPU only (their figures are
    # per-call fractions, not a job total).
    others = None
    if world == 1 and not args.no_workloads:
        del h_q, h_init, h_dcum, o_cum, o_dq, o_di, q, init, d_cum, d_init, flushbuf
        torch.cuda.empty_cache()
        others = {"note": "each workload's step (forward + backward), each call alone (median of 20, "
                          "L2 flushed by a read before every rep) and the saved-carries step; "
                          "fractions of the measured copy bandwidth at 32 / 48 / 80 B per element"}
        for name in ("small", "large", "long"):
            others[name] = time_other_workload(qs, torch, name, dev, stream, min(args.steps, 10),
                                               args.warmup, peak)
            torch.cuda.empty_cache()
    if rank != 0:
        return 0
    bwd_avg = statistics.mean(bwd_ms)
    fwd_avg = statistics.mean(fwd_ms)
    bwd_gbs = BWD_BYTES_PER_ELEMENT * E / (bwd_avg * 1e-3) / 1e9
    fwd_gbs = FWD_BYTES_PER_ELEMENT * E / (fwd_avg * 1e-3) / 1e9
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        sample, lanes = oracle_sample(w, args.cpu_lanes, (q_np, init_np, dcum_np))
        rate, cores, reps, _ = time_oracle(sample, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": sample_description(w, lanes, reps, cores)}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded generator, workloads.py)",
        "config": {"workload": w.describe(), "B": w.B, "S": w.S, "H": w.H, "J": w.J,
                   "elements": E, "bytes_per_tensor": tensor_bytes,
                   "l2": ("L2 flushed (2x126 MB read) before every step" if flush else
                          f"inputs larger than L2 ({tensor_bytes / 1e6:.0f} MB per tensor > 126 MB), no flush"),
                   "parallelism": ("one independent batch per GPU, no collective" if world > 1
                                   else "single GPU")},
        "roofline": {"bound": "hbm", "kernel": design_name("quat_cumprod_bwd", bwd_kernels, bwd_variant),
                     "variant": bwd_variant,
                     "achieved": bwd_gbs, "peak": peak,
                     "unit": "GB/s", "frac": bwd_gbs / peak, "peak_source": peak_src,
                     "traffic": recorded_traffic("quat_cumprod_bwd", w.name),
                     "traffic_source": TRAFFIC_NOTE,
                     "algorithmic_bytes_per_launch": BWD_BYTES_PER_ELEMENT * E,
                     "avg_launch_ms": bwd_avg},
        "roofline_fwd": {"bound": "hbm", "kernel": design_name("quat_cumprod_fwd", fwd_kernels, fwd_variant),
                         "variant": fwd_variant,
                         "achieved": fwd_gbs, "peak": peak,
                         "unit": "GB/s", "frac": fwd_gbs / peak,
                         "traffic": recorded_traffic("quat_cumprod_fwd", w.name),
                         "algorithmic_bytes_per_launch": FWD_BYTES_PER_ELEMENT * E,
                         "avg_launch_ms": fwd_avg},
        "roofline_step": {"bound": "hbm", "unit": "GB/s", "peak": peak,
                          "achieved": STEP_BYTES * E / (step_ms * 1e-3) / 1e9,
                          "frac": STEP_BYTES * E / (step_ms * 1e-3) / 1e9 / peak,
                          "algorithmic_bytes_per_step": STEP_BYTES * E},
        "alone": {
            "note": f"each call timed by itself: median of {alone_reps} reps, L2 flushed before every rep "
                    "by reading a 2x126 MB buffer (no dirty lines left behind)",
            "reps": alone_reps,
            **{k: {"ms": v, "achieved_gbs": nbytes * E / (v * 1e-3) / 1e9,
                   "frac": nbytes * E / (v * 1e-3) / 1e9 / peak}
               for k, v, nbytes in (("fwd", alone_ms["fwd"], FWD_BYTES_PER_ELEMENT),
                                    ("bwd", alone_ms["bwd"], BWD_BYTES_PER_ELEMENT),
                                    ("fwd_bwd", alone_ms["fwd_bwd"], STEP_BYTES))}},
        "saved_carries": {
            "note": "forward also writes the 64-step chunk carries; backward starts from them "
                    "(the page's node keeps only q and init: this is the measured alternative)",
            "value": weak_scaling_value(world, E, cstep_ms), "unit": UNIT, "ms_per_step": cstep_ms,
            "fwd_ms": cfwd_ms, "bwd_ms": cbwd_ms,
            "bwd_achieved_gbs": BWD_BYTES_PER_ELEMENT * E / (cbwd_ms * 1e-3) / 1e9,
            "bwd_frac": BWD_BYTES_PER_ELEMENT * E / (cbwd_ms * 1e-3) / 1e9 / peak,
            "kernels_per_step": cfwd_kernels + cbwd_kernels},
        "bf16": None if not even else {
            "note": "every tensor bfloat16, fp32 arithmetic; algorithmic bytes 16 (fwd) / 24 (bwd) per element",
            "value": weak_scaling_value(world, E, bstep_ms), "unit": UNIT, "ms_per_step": bstep_ms,
            "fwd_ms": bfwd_ms, "bwd_ms": bbwd_ms,
            "fwd_achieved_gbs": 16 * E / (bfwd_ms * 1e-3) / 1e9,
            "fwd_frac": 16 * E / (bfwd_ms * 1e-3) / 1e9 / peak,
            "bwd_achieved_gbs": 24 * E / (bbwd_ms * 1e-3) / 1e9,
            "bwd_frac": 24 * E / (bbwd_ms * 1e-3) / 1e9 / peak,
            "kernels_per_step": bf16_kernels},
        "cpu_baseline": cpu,
        "e2e": {"value": weak_scaling_value(world, E, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
                "call": "quat_cumprod_fwd_bwd_host (pinned host buffers; batch slices whose copies "
                        "overlap the kernels)"},
        "workloads": others,
        "bitwise_repeatable": repeatable,
        "gpu_launches": launches[0],
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(workloads.WORKLOADS), default=DEFAULT_WORKLOAD)
    p.add_argument("--e2e-steps", type=int, default=5)
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--cpu-lanes", type=int, default=512)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--batch", type=int, default=None,
                   help="the workload's recipe with this many batch entries (a smaller case of a large workload)")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip timing the small, large and long workloads besides the headline one")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.gpus != world and world > 1:
        p.error(f"--gpus {args.gpus} does not match WORLD_SIZE {world}")
    w = workloads.WORKLOADS[args.workload]
    if args.batch is not None:   # the same workload with another batch size
        if args.batch < 1:
            p.error("--batch must be >= 1")
        w = workloads.custom(w.name, args.batch, w.S, w.H, w.J, q_kind=w.q_kind, theta_max=w.theta_max,
                             init_kind=w.init_kind, dcum_sigma=w.dcum_sigma, seed=w.seed)
    if args.impl == "reference":
        return run_reference(args, w, world, rank)
    return run_ours(args, w, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
