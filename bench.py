"""Benchmark of the SCAPE sharded optimizer step on GB300.

One step = the whole hot path over one batch of synthetic per-worker gradients:
scape_step (error-feedback compaction, ordered sparse reduce, sparse AdamS)
plus scape_refresh_mask (the partitioned top-k that the next step uses).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama500m]
    python bench.py --impl reference ...     # the CPU oracle, same metric

Rank 0 prints one JSON line.  With N > 1 (torchrun) the workload's W optimizer
shards are split into N contiguous blocks, one per GPU: each rank holds a
shard-range handle over its parameter slice and steps the slices of all W
workers' gradients (optimizer shards are independent, so no data-path
collective runs), and the value is P over the slowest rank's time (strong
scaling: one problem of fixed size).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SCAPE optimizer-step params/s and achieved HBM GB/s (% of GB300 peak)"
UNIT = "params/s"
PROFILES = os.path.join(ROOT, "profiles")


# --------------------------------------------------------------------- helpers
def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _grad_bytes(wl):
    return 2 if wl.grad_dtype == "bf16" else 4


def mask_churn(prev_bits, bits, k):
    """Fraction of the selected coordinates that changed between two masks:
    |prev XOR new| / (2k), from the two bitmaps (int32 tensors of the same
    length, any device).  0 for identical masks, 1 for disjoint ones."""
    import torch

    x = torch.bitwise_xor(prev_bits, bits).view(torch.uint8).to(torch.int64)
    lut = torch.tensor([bin(v).count("1") for v in range(256)], dtype=torch.int64,
                       device=x.device)
    return float(lut[x].sum().item()) / (2.0 * k) if k else 0.0


FUSION = {"none": 0, "sum": 1, "update": 2}  # scape_set_fusion levels
FUSION_NAME = {v: k for k, v in FUSION.items()}


def apply_fusion(opt, choice):
    """Set the fusion level ("auto": keep the library's default for the
    handle's density) and return the name of the level in force."""
    if choice != "auto":
        opt.set_fusion(FUSION[choice])
    return FUSION_NAME[opt.fusion()]


def algorithmic_bytes(wl, k, fusion="sum", P=None):
    """Bytes the method must move per step, by kernel (see the design notes).
    fusion "sum": the compaction also writes g_bar, so the packed buffers are
    written but never re-read; "update": it also updates w and m at the k
    selected coordinates (no index list or g_bar to read back).  P: the
    parameters one rank's handle covers, when the shards are split."""
    P, W, G = (wl.P if P is None else P), wl.W, _grad_bytes(wl)
    ntiles = (P + 2047) // 2048
    ef = W * P * (G + 8) + P / 8 + 4 * ntiles + 4 * k * W
    # a mask that keeps every coordinate never changes: no refresh after the first
    refresh = 0 if k >= P else 4 * P + P / 8 + P / 8 + 4 * k
    out = {"refresh": refresh}
    if fusion == "update":
        out["ef_compact"] = ef + 4 * k + 16 * k
    elif fusion == "sum":
        out["ef_compact"] = ef + 4 * k
        out["adams_sparse"] = 24 * k
    else:
        out["ef_compact"] = ef
        out["reduce"] = 4 * k * W + 4 * k
        out["adams_sparse"] = 24 * k
    out["total"] = sum(out.values())
    return out


def _kernel_source_hash():
    """Hash of the ef_compact kernel's own source (its section of
    step_kernels.cu) and of the shared header it includes."""
    csrc = os.path.join(ROOT, "sparse_communication_sharded_gb300", "csrc")
    with open(os.path.join(csrc, "step_kernels.cu")) as f:
        src = f.read()
    a = src.index("// ------------------------------------------------------------------ ef_compact")
    b = src.index("// ------------------------------------------------------------------ dense_step")
    h = hashlib.sha256(src[a:b].encode())
    with open(os.path.join(csrc, "scape_internal.cuh"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def _ncu_traffic(workload):
    """DRAM bytes per ef_compact launch from the committed ncu summary, if it
    was taken on the current kernel source; else None."""
    p = os.path.join(PROFILES, f"ef_compact_{workload}.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_sha256_16") != _kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9 and parts[0] == str(self.gpu_index):
                        rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


def _mem_available():
    """Host MemAvailable in bytes (0 if unknown)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def _parse_cpulist(text):
    cpus = set()
    for part in text.strip().split(","):
        if not part:
            continue
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        else:
            cpus.add(int(part))
    return cpus


def _bind_near_gpu(dev):
    """Run this process on the host cores attached to the GPU's socket, so
    that page-locked buffers allocated afterwards sit in that socket's memory
    (first touch) and host<->device copies do not cross the socket link.
    Returns the cores used, or None if the topology is not readable."""
    import torch

    try:
        pr = torch.cuda.get_device_properties(dev)
        path = "/sys/bus/pci/devices/%04x:%02x:%02x.0/local_cpulist" % (
            pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        with open(path) as f:
            cpus = _parse_cpulist(f.read()) & os.sched_getaffinity(0)
        if not cpus:
            return None
        os.sched_setaffinity(0, cpus)
        return sorted(cpus)
    except (AttributeError, OSError, ValueError):
        return None


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# --------------------------------------------------------------------- config
READING = ("paper: only selected coordinates update w and m; the synchronised buffer holds "
           "the mean of the masked error-fed gradients (the first-moment form is "
           "SCAPE_VARIANT_MOMENT_SYNC)")


def k_of(wl):
    """k = sum over shards of ceil(n_s (1 - sparsity)), sparsity in ppm."""
    ppm = round(wl.sparsity * 1e6)
    starts = [s * wl.P // wl.W for s in range(wl.W + 1)]
    return sum(((starts[s + 1] - starts[s]) * (1000000 - ppm) + 999999) // 1000000
               for s in range(wl.W))


def workload_config(wl, args, ws=1):
    """The `config` object of the JSON line; both arms print the same one."""
    return {"workload": wl.name, "P": wl.P, "W": wl.W, "sparsity": wl.sparsity, "k": k_of(wl),
            "grad_dtype": wl.grad_dtype, "state_dtype": "f32", "reading": READING,
            "residuals": args.residuals, "fusion": args.fusion,
            "staging_rows": (0 if args.residuals == "device" else
                             min(wl.W, 12) if args.staging_rows is None else
                             (max(args.staging_rows, 3) if args.staging_rows else 0)),
            "l2": "inputs larger than L2 (gradients + residuals far beyond 129 MB)",
            "parallelism": (f"one problem, its {wl.W} optimizer shards split over {ws} GPUs "
                            f"(contiguous blocks; strong scaling)" if ws > 1 else "1 GPU")}


# --------------------------------------------------------------------- oracle leg
def _local_cores():
    """Host cores this process may run on (those local to the GPU when the
    process was bound to them)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _sample_shards(W, n):
    """n shard indices spread evenly over 0..W-1 (first and last included)."""
    if n >= W:
        return list(range(W))
    if n == 1:
        return [W // 2]
    return sorted({round(j * (W - 1) / (n - 1)) for j in range(n)})


def run_oracle_leg(wl, steps, n_shards, device=None, compare=False, seed=0):
    """The CPU oracle, one process per optimizer shard, on `n_shards` shards of
    the workload: a dense first step, then `steps` lagged sparse steps with
    their mask refreshes.  Shards are independent sub-problems, so each worker
    runs its shard as a one-shard problem of its own (oracle.pool).  Inputs are
    drawn on `device` (the GPU when there is one) with the bench's seed and
    copied into the workers' shared buffers.  With compare, the GPU runs the
    same whole problem from the same inputs and every refresh's mask is
    compared with the oracle's on the sampled shards.

    Returns a dict: params/s of the sampled shards over the sparse steps (the
    sum of their sizes times the steps, over the sum of the per-step times of
    the slowest worker), the per-step wall time of that sample, and, with
    compare, the mask bits compared and flipped."""
    import numpy as np
    import torch

    from oracle import oracle as O
    from oracle.pool import ShardOracles
    from sparse_communication_sharded_gb300 import synth

    P, W = wl.P, wl.W
    hp = O.Hyper()
    start, ks = O.layout(P, W, wl.sparsity)
    shards = _sample_shards(W, n_shards)
    spec = [(int(start[s]), int(start[s + 1]), int(ks[s])) for s in shards]
    gdev = device if device is not None else "cpu"
    w0 = synth.init_params(P, seed=seed, device=gdev)
    if device is not None:
        gen = synth.GradientStream(wl, seed=seed, device=gdev)
        slices = None
    else:
        # no GPU: draw each sampled shard's slices on its own (same recipe)
        gen = None
        slices = [synth.GradientStream(wl, seed=seed + 1 + j, device="cpu", P=hi - lo, offset=lo)
                  for j, (lo, hi, _) in enumerate(spec)]
    opt = None
    if compare:
        import sparse_communication_sharded_gb300 as pkg

        params = w0.clone()
        gdt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
        opt = pkg.Scape(params, W, wl.sparsity, layer_numel=[n for _, n in wl.layers],
                        lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps,
                        weight_decay=hp.weight_decay, grad_dtype=gdt)
    popc = np.array([bin(v).count("1") for v in range(256)], np.int64)
    flips = bits = 0
    step_s = []
    bf16 = wl.grad_dtype == "bf16"
    with ShardOracles(spec, W, wl.grad_dtype, hp, lambda lo, hi: w0[lo:hi].cpu().numpy(),
                      pin=device is not None) as pool:
        del w0
        bufs = gen.alloc() if gen is not None else None
        for t in range(1, steps + 2):
            if gen is not None:
                gen.next_into(bufs)
            for j, (lo, hi, _) in enumerate(spec):
                host = torch.from_numpy(pool.grads(j).view(np.int16 if bf16 else np.float32))
                src_rows = bufs if gen is not None else slices[j].next()
                for w in range(W):
                    src = src_rows[w][lo:hi] if gen is not None else src_rows[w]
                    host[w].copy_(src.view(torch.int16) if bf16 else src, non_blocking=True)
            if opt is not None:
                opt.step(bufs)
                opt.refresh_mask()
            if device is not None:
                torch.cuda.synchronize()
            times = pool.step()
            if t >= 2:
                step_s.append(max(times))
            if opt is not None:
                g = opt.bits().cpu().numpy().view(np.uint32)
                for j, (lo, hi, _) in enumerate(spec):
                    n = hi - lo
                    nw = (n + 31) // 32
                    w0i, sh = lo // 32, lo % 32
                    a = g[w0i:w0i + nw].astype(np.uint64)
                    b = np.zeros(nw, np.uint64)
                    nxt = g[w0i + 1:w0i + 1 + nw].astype(np.uint64)
                    b[:nxt.size] = nxt
                    loc = (((a >> np.uint64(sh)) | (b << np.uint64(32 - sh)))
                           & np.uint64(0xFFFFFFFF)).astype(np.uint32)
                    if n % 32:
                        loc[-1] &= np.uint32((1 << (n % 32)) - 1)
                    x = (loc ^ pool.out(j)["bits"]).view(np.uint8)
                    flips += int(popc[x].sum())
                    bits += n
        del bufs
    if opt is not None:
        opt.close()
        del params
    if device is not None:
        torch.cuda.empty_cache()
    n_sample = sum(hi - lo for lo, hi, _ in spec)
    secs = sum(step_s)
    return {"params_per_s": n_sample * len(step_s) / secs if secs else None,
            "ms_per_step": 1000.0 * secs / max(len(step_s), 1), "steps": len(step_s),
            "shards": shards, "n_sample": n_sample, "processes": len(spec),
            "mask_bits": bits, "mask_flips": flips,
            "mask_flip_fraction": flips / bits if bits else None}


def oracle_sample_text(res, wl):
    return (f"{len(res['shards'])} of {wl.W} optimizer shards ({res['n_sample']} of {wl.P} "
            f"params, {wl.W} workers each), one oracle process per shard in parallel, "
            f"{res['steps']} lagged sparse steps + refreshes after an untimed dense step; "
            f"value = sampled params x steps / sum over steps of the slowest process's time")


# --------------------------------------------------------------------- reference arm
def bench_reference(args, wl):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import torch
    dev = torch.device("cuda:0") if torch.cuda.is_available() else None
    cores = _local_cores()
    if dev is not None:
        near = _bind_near_gpu(dev)
        cores = len(near) if near else cores
    steps = max(1, args.steps)
    t0 = time.perf_counter()
    res = run_oracle_leg(wl, steps, min(cores, wl.W), device=dev)
    wall = time.perf_counter() - t0
    line = {
        "impl": "reference", "metric": METRIC, "value": res["params_per_s"], "unit": UNIT,
        "n_gpus": ws, "steps": res["steps"], "warmup": args.warmup,
        "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(wl, args),
        "cpu_baseline": {"value": res["params_per_s"], "unit": UNIT, "cores": res["processes"],
                         "kind": "oracle", "sample": oracle_sample_text(res, wl)},
        "extrapolated": {"sample_is_whole_problem": res["n_sample"] == wl.P,
                         "shards_timed": len(res["shards"]), "shards_total": wl.W,
                         "ms_per_step_of_sample": res["ms_per_step"],
                         "full_problem_ms_per_step_estimate":
                             res["ms_per_step"] * wl.P / res["n_sample"],
                         "note": "ms_per_step is the measured time of the sampled shards; "
                                 "the full-problem figure scales it by P / sampled params "
                                 "(shards are independent) and is not measured"},
        "wall_s": wall,
        "e2e": {"value": res["params_per_s"], "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------- GPU arm
def time_steps(opt, gen, grads, steps, barrier=lambda: None):
    """Time `steps` whole steps (scape_step + scape_refresh_mask) with CUDA
    events on the current stream; fresh gradients before each, outside the
    timed window.  Returns the per-step milliseconds and wall seconds."""
    import torch

    step_ms, wall = [], []
    st = torch.cuda.current_stream()
    for _ in range(steps):
        gen.next_into(grads)
        barrier()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        ev0.record(st)
        opt.step(grads)
        opt.refresh_mask()
        ev1.record(st)
        torch.cuda.synchronize()
        wall.append(time.perf_counter() - t0)
        barrier()
        step_ms.append(ev0.elapsed_time(ev1))
    return step_ms, wall


def bench_other_workload(name, args, dev, peak):
    """One more shape, timed like the headline one (fewer extras)."""
    import torch

    import sparse_communication_sharded_gb300 as pkg
    from sparse_communication_sharded_gb300 import synth

    wl = synth.WORKLOADS[name]
    gdt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
    params = synth.init_params(wl.P, seed=0, device=dev)
    opt = pkg.Scape(params, wl.W, wl.sparsity, layer_numel=[n for _, n in wl.layers],
                    grad_dtype=gdt)
    fusion = apply_fusion(opt, args.fusion)
    gen = synth.GradientStream(wl, seed=0, device=dev)
    grads = gen.alloc()
    for _ in range(args.warmup):
        gen.next_into(grads)
        opt.step(grads)
        opt.refresh_mask()
    torch.cuda.synchronize()
    opt.profile(True)
    opt.profile_select(["ef_compact"])
    opt.profile_reset()
    step_ms, _ = time_steps(opt, gen, grads, args.other_steps)
    opt.profile_collect()
    ef_ms, ef_n = opt.profile_read()["ef_compact"]
    # per-kernel split from two profiled steps after the timed ones
    opt.profile_select(0xFFFFFFFF)
    opt.profile_reset()
    for _ in range(2):
        gen.next_into(grads)
        opt.step(grads)
        opt.refresh_mask()
    torch.cuda.synchronize()
    opt.profile_collect()
    prof = opt.profile_read()
    opt.profile(False)
    k = opt.k
    opt.close()
    del grads, params, opt
    torch.cuda.empty_cache()
    ms = sum(step_ms) / len(step_ms)
    alg = algorithmic_bytes(wl, k, fusion=fusion)
    ef_avg = ef_ms / max(ef_n, 1)
    step_kernels = ("dense_step", "ef_compact", "reduce", "adams_sparse")
    return {"P": wl.P, "W": wl.W, "sparsity": wl.sparsity, "k": k, "grad_dtype": wl.grad_dtype,
            "fusion": fusion, "steps": args.other_steps, "warmup": args.warmup, "ms_per_step": ms,
            "ms_each": step_ms, "params_per_s": wl.P / (ms / 1000.0),
            "hbm_gbs": alg["total"] / (ms / 1000.0) / 1e9,
            "hbm_frac": alg["total"] / (ms / 1000.0) / 1e9 / peak,
            "alg_bytes_per_step": alg["total"],
            "ef_compact": {"ms_per_launch": ef_avg,
                           "gbs": alg["ef_compact"] / (ef_avg / 1000.0) / 1e9,
                           "frac": alg["ef_compact"] / (ef_avg / 1000.0) / 1e9 / peak},
            "kernels_ms_per_step": {n: m / 2 for n, (m, c) in prof.items() if c},
            "refresh_ms_per_step": sum(m for n, (m, _) in prof.items()
                                       if n not in step_kernels) / 2}


def bench_gpu(args, wl):
    import torch
    import torch.distributed as dist

    import sparse_communication_sharded_gb300 as pkg
    from sparse_communication_sharded_gb300 import multirank, synth

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    pkg.load()

    def barrier():
        if ws > 1:
            dist.barrier()

    P, W = wl.P, wl.W
    gdt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
    seed = 0
    # this rank's block of optimizer shards (all of them on one GPU)
    if W < ws:
        raise SystemExit(f"{W} optimizer shards cannot be split over {ws} GPUs")
    shards = multirank.rank_shards(W, ws, rank)
    lo, hi = multirank.shard_slice(P, W, shards)
    params = synth.init_params(hi - lo, seed=seed + lo, device=dev)
    opt = pkg.Scape(params, W, wl.sparsity, layer_numel=[n for _, n in wl.layers],
                    grad_dtype=gdt, residuals=args.residuals, staging_rows=args.staging_rows,
                    shard_range=(shards.start, shards.stop) if ws > 1 else None)
    fusion = apply_fusion(opt, args.fusion)
    # the slices [lo, hi) of the W workers' gradients
    gen = synth.GradientStream(wl, seed=seed, device=dev, P=hi - lo, offset=lo)
    grads = gen.alloc()

    # warm-up: the dense first step and W - 1 lagged steps
    for _ in range(args.warmup):
        gen.next_into(grads)
        opt.step(grads)
        opt.refresh_mask()
    torch.cuda.synchronize()

    # timed steps: fresh gradients each step (outside the timed window),
    # inputs (~115 GB for llama500m) far larger than the 129 MB L2.  Only the
    # roofline kernel is bracketed by events here: two event records per
    # launch cost about 0.1 ms per step over the ~25 launches; the per-kernel
    # breakdown comes from extra profiled steps after the timed ones.
    opt.profile(True)
    opt.profile_select(["ef_compact"])
    opt.profile_reset()
    n_launch0 = opt.launch_count()
    with ClockSampler(local) as clk:
        step_ms, wall = time_steps(opt, gen, grads, args.steps, barrier=barrier)
    launches = opt.launch_count() - n_launch0
    opt.profile_collect()
    prof_timed = opt.profile_read()
    clocks = clk.summary()
    # per-kernel breakdown: a few more steps with every kernel bracketed
    # (and the mask's step-to-step churn: the temporal stability the lagged
    # mask relies on)
    n_break = 3
    opt.profile_select(0xFFFFFFFF)
    opt.profile_reset()
    churn = []
    for _ in range(n_break):
        prev = opt.bits().clone()
        gen.next_into(grads)
        opt.step(grads)
        opt.refresh_mask()
        churn.append(mask_churn(prev, opt.bits(), opt.k))
    torch.cuda.synchronize()
    opt.profile_collect()
    prof = opt.profile_read()
    # the scattered update's floor on this GPU: its memory accesses alone
    opt.profile_reset()
    for _ in range(3):
        opt.probe_random_access()
    torch.cuda.synchronize()
    opt.profile_collect()
    probe_ms = opt.profile_read()["probe_rmw"][0] / 3
    opt.profile(False)

    my_ms = sum(step_ms) / len(step_ms)
    t_max = my_ms
    if ws > 1:
        tt = torch.tensor([my_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t_max = float(tt.item())
    value = multirank.strong_scaling_value(P, t_max / 1000.0)
    alg = algorithmic_bytes(wl, opt.k, fusion=fusion, P=hi - lo)
    alg_total = multirank.sum_over_ranks(alg["total"], device=dev)
    peak, peak_kind = _peaks()

    ef_ms, ef_n = prof_timed["ef_compact"]
    ef_avg = ef_ms / max(ef_n, 1)
    ef_gbs = alg["ef_compact"] / (ef_avg / 1000.0) / 1e9
    traffic = _ncu_traffic(wl.name)
    kernels = {}
    for name, (ms, n) in prof.items():
        if n:
            kernels[name] = {"launches": n, "ms_per_step": ms / n_break,
                             "share": ms / max(sum(m for m, _ in prof.values()), 1e-9)}
    step_kernels = ("dense_step", "ef_compact", "reduce", "adams_sparse")
    refresh_ms = sum(ms for name, (ms, _) in prof.items() if name not in step_kernels) / n_break
    upd_ms, upd_n = prof["adams_sparse"]
    upd_ms = upd_ms / max(upd_n, 1)
    update_roofline = None
    if upd_n:
        update_roofline = {
            "kernel": "adams_sparse", "bound": "random DRAM accesses",
            "ms_per_launch": upd_ms, "alg_bytes_per_launch": 24 * opt.k,
            "achieved_gbs": 24 * opt.k / (upd_ms / 1000.0) / 1e9,
            "frac_of_hbm_peak": 24 * opt.k / (upd_ms / 1000.0) / 1e9 / peak,
            "probe_ms": probe_ms, "frac_of_probe": probe_ms / upd_ms,
            "note": "probe = the same scattered reads and writes of w and m (and in-order idx "
                    "and g_bar) without the arithmetic, on this GPU: the floor of this kernel"}

    # dense baselines on the same workload and buffers (after the SCAPE timing)
    baselines = None
    if args.baselines and ws == 1:
        baselines = bench_baselines(opt, wl, grads, dev)

    # end to end through the C ABI from pinned host memory
    e2e = None
    if args.e2e_steps > 0:
        e2e = bench_e2e(opt, wl, grads, args.e2e_steps, dev, shared_source=ws > 1)
        if ws > 1:
            # whole job: the ranks' slices make up the P parameters; the
            # slowest rank sets the time
            t_e2e = multirank.max_over_ranks(e2e["ms_per_step"], device=dev)
            e2e["ms_per_step"] = t_e2e
            e2e["value"] = P / (t_e2e / 1000.0)
            e2e["h2d_bytes_per_step"] = int(multirank.sum_over_ranks(e2e["h2d_bytes_per_step"],
                                                                     device=dev))
            e2e["d2h_bytes_per_step"] = int(multirank.sum_over_ranks(e2e["d2h_bytes_per_step"],
                                                                     device=dev))
    opt.close()
    del grads, params, opt, gen
    torch.cuda.empty_cache()

    # the other two shapes of the pages' workloads, timed the same way
    others = {}
    if ws == 1 and args.other_steps > 0:
        for name in ("gpt345m", "llama500m", "llama1p8b"):
            if name != wl.name and args.workload in synth.WORKLOADS:
                others[name] = bench_other_workload(name, args, dev, peak)

    # the CPU oracle on the host cores local to the GPU, one process per
    # shard, on the same inputs as a fresh GPU run of the workload: its rate
    # (the CPU baseline) and the mask bits that differ from the GPU's
    cpu = None
    oracle_leg = None
    if rank == 0 and ws == 1 and args.cpu_steps > 0:
        near = _bind_near_gpu(dev)
        cores = len(near) if near else _local_cores()
        oracle_leg = run_oracle_leg(wl, args.cpu_steps, min(cores, W), device=dev, compare=True)
        cpu = {"value": oracle_leg["params_per_s"], "unit": UNIT,
               "cores": oracle_leg["processes"], "kind": "oracle",
               "sample": oracle_sample_text(oracle_leg, wl),
               "ms_per_step_of_sample": oracle_leg["ms_per_step"],
               "extrapolated": False}

    if rank == 0:
        config = workload_config(wl, args, ws)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_max, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config,
            "hbm_gbs": alg_total / (t_max / 1000.0) / 1e9,
            "hbm_frac": alg_total / (t_max / 1000.0) / 1e9 / (peak * ws),
            "alg_bytes_per_step": alg_total,
            "fusion_level": fusion,
            "rank0_shards": [shards.start, shards.stop],
            "roofline": {"kernel": "ef_compact", "bound": "hbm", "achieved": ef_gbs,
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": ef_gbs / peak, "traffic": traffic,
                         "alg_bytes_per_launch": alg["ef_compact"], "ms_per_launch": ef_avg},
            "kernels": kernels,
            "update_roofline": update_roofline,
            "kernels_measured_over": f"{n_break} profiled steps after the timed ones",
            "refresh_ms_per_step": refresh_ms,
            "mask_churn_per_refresh": churn,
            "mask_flip_fraction": oracle_leg["mask_flip_fraction"] if oracle_leg else None,
            "mask_flips": ({"flipped": oracle_leg["mask_flips"], "compared": oracle_leg["mask_bits"],
                            "over": f"{oracle_leg['steps'] + 1} refreshes of shards "
                                    f"{oracle_leg['shards']} against the oracle on the same "
                                    f"inputs"} if oracle_leg else None),
            "wall_ms_per_step": 1000.0 * sum(wall) / len(wall),
            "gpu_launches": launches,
            "clocks": clocks,
            "e2e": e2e,
            "baselines": baselines,
            "other_workloads": others or None,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# --------------------------------------------------------------------- exchange mode
def bench_exchange(args, wl):
    """The exchange-based multi-rank step (exchange.ScapeDP): each of the N
    ranks owns W/N workers (their full gradients and residuals) and W/N
    optimizer shards; a step is the compaction, the all-to-all of the packed
    values, the owners' update, the sparse parameter all-gather, the owners'
    mask refresh and the mask all-gather (NCCL).  value = P over the slowest
    rank's step time (one problem of fixed size: strong scaling)."""
    import dataclasses

    import torch
    import torch.distributed as dist

    import sparse_communication_sharded_gb300 as pkg
    from sparse_communication_sharded_gb300 import multirank, synth
    from sparse_communication_sharded_gb300.exchange import ScapeDP

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    pkg.load()
    P, W = wl.P, wl.W
    mine = multirank.rank_shards(W, ws, rank)
    lo, hi = multirank.shard_slice(P, W, mine)
    gsz = _grad_bytes(wl)
    wl_ = len(mine)
    need = wl_ * P * (gsz + 4 + 4) + 4 * P + W * (hi - lo) * 4 + 16 * (hi - lo) + (1 << 30)
    free, _ = torch.cuda.mem_get_info()
    if need > 0.92 * free:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "mode": "exchange", "value": None,
                              "unavailable": f"needs ~{need / 2**30:.0f} GiB per GPU at N={ws}, "
                                             f"{free / 2**30:.0f} GiB free"}), flush=True)
        if ws > 1:
            dist.destroy_process_group()
        return 0
    gdt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
    params = synth.init_params(P, seed=0, device=dev)
    opt = ScapeDP(params, W, wl.sparsity, layer_numel=[n for _, n in wl.layers], grad_dtype=gdt)
    gen = synth.GradientStream(dataclasses.replace(wl, W=wl_), seed=1 + rank, device=dev)
    grads = gen.alloc()

    def barrier():
        if ws > 1:
            dist.barrier()

    for _ in range(args.warmup):
        gen.next_into(grads)
        opt.step(grads)
    torch.cuda.synchronize()
    b0, n0 = opt.bytes_sent, opt.launch_count()
    st = torch.cuda.current_stream()
    step_ms = []
    with ClockSampler(local) as clk:
        for _ in range(args.steps):
            gen.next_into(grads)
            barrier()
            torch.cuda.synchronize()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(st)
            opt.step(grads)
            ev1.record(st)
            torch.cuda.synchronize()
            barrier()
            step_ms.append(ev0.elapsed_time(ev1))
    sent = (opt.bytes_sent - b0) / args.steps
    launches = opt.launch_count() - n0
    my_ms = sum(step_ms) / len(step_ms)
    t_max = multirank.max_over_ranks(my_ms, device=dev)
    sent_all = multirank.sum_over_ranks(sent, device=dev)
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "mode": "exchange", "value": P / (t_max / 1000.0), "unit": UNIT,
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": dict(workload_config(wl, args, ws),
                           parallelism=f"{ws} data-parallel ranks, each owning {W // ws} or "
                                       f"{(W + ws - 1) // ws} workers and optimizer shards; "
                                       f"NCCL all-to-all + two all-gathers per step"),
            "exchange_bytes_per_step": sent_all,
            "rank0_ms_each": step_ms, "gpu_launches": launches, "clocks": clk.summary()}),
            flush=True)
    opt.close()
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# --------------------------------------------------------------------- flat sweep
SWEEP_W = (1, 8, 32)
SWEEP_S = (0.0, 0.9, 0.99, 0.999)


def sweep_device_bytes(P, W, k, stride=64):
    """Device memory one flat-sweep point needs: f32 gradients and residuals of
    every worker, w and m, and the library's workspace (the candidate buffer
    of 8 bytes per parameter dominates it), plus the generator's scratch."""
    rows = (P + stride - 1) // stride * stride
    ws = P * 8 + W * k * 4 + 2 * k * 4 + P // 8 + W * 8192 * 4 + (64 << 20)
    return W * P * 4 + W * rows * 4 + 8 * P + ws + 5 * 4 * min(P, 1 << 26) + 4 * P


def bench_sweep(args):
    """The flat sweep: P = 2^e fp32 parameters for the exponents given, W in
    {1, 8, 32}, sparsity in {0, 90, 99, 99.9}%, gradients quantised to 256
    levels (many ties in |m|).  Each point: the dense first step and
    warm-up - 1 lagged steps untimed, then `steps` timed steps (scape_step +
    scape_refresh_mask, CUDA events).  Points whose footprint exceeds 90% of
    the free device memory are reported as skipped."""
    import torch

    import sparse_communication_sharded_gb300 as pkg
    from sparse_communication_sharded_gb300 import synth

    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    pkg.load()
    peak, peak_kind = _peaks()
    points = []
    with ClockSampler(0) as clk:
        for e in args.sweep_exps:
            P = 1 << e
            for W in SWEEP_W:
                for sp in SWEEP_S:
                    wl = synth.flat_workload(P, W, sp, steps=args.steps)
                    k = k_of(wl)
                    need = sweep_device_bytes(P, W, k)
                    torch.cuda.empty_cache()
                    free, _ = torch.cuda.mem_get_info()
                    pt = {"P": P, "log2P": e, "W": W, "sparsity": sp, "k": k,
                          "device_bytes": need}
                    if need > 0.9 * free:
                        pt["skipped"] = f"needs {need / 2**30:.0f} GiB, {free / 2**30:.0f} GiB free"
                        points.append(pt)
                        continue
                    params = synth.init_params(P, seed=0, device=dev)
                    opt = pkg.Scape(params, W, sp, grad_dtype=torch.float32)
                    fusion = apply_fusion(opt, args.fusion)
                    gen = synth.GradientStream(wl, seed=0, device=dev)
                    grads = gen.alloc()
                    for _ in range(args.warmup):
                        gen.next_into(grads)
                        opt.step(grads)
                        opt.refresh_mask()
                    torch.cuda.synchronize()
                    step_ms, _ = time_steps(opt, gen, grads, args.steps)
                    # per-kernel split of two more steps
                    opt.profile(True)
                    opt.profile_reset()
                    for _ in range(2):
                        gen.next_into(grads)
                        opt.step(grads)
                        opt.refresh_mask()
                    torch.cuda.synchronize()
                    opt.profile_collect()
                    prof = opt.profile_read()
                    opt.close()
                    del grads, params, opt, gen
                    ms = sorted(step_ms)[len(step_ms) // 2]
                    ab = algorithmic_bytes(wl, k, fusion=fusion)
                    pt["fusion"] = fusion
                    alg = ab["total"]
                    ef_ms = prof["ef_compact"][0] / max(prof["ef_compact"][1], 1)
                    pt.update({"ms_per_step": ms, "ms_each": step_ms,
                               "params_per_s": P / (ms / 1000.0),
                               "hbm_gbs": alg / (ms / 1000.0) / 1e9,
                               "hbm_frac": alg / (ms / 1000.0) / 1e9 / peak,
                               "ef_compact_ms": ef_ms,
                               "ef_compact_frac": ab["ef_compact"] / (ef_ms / 1000.0) / 1e9 / peak,
                               "kernels_ms_per_step": {n: m / 2 for n, (m, c) in prof.items()
                                                       if c}})
                    points.append(pt)
    torch.cuda.empty_cache()
    done = [p for p in points if "ms_per_step" in p]
    big = [p for p in done if p["log2P"] == max(q["log2P"] for q in done)] if done else []
    line = {"metric": METRIC, "value": (max(p["params_per_s"] for p in big) if big else None),
            "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "flat sweep", "exponents": list(args.sweep_exps),
                       "W": list(SWEEP_W), "sparsity": list(SWEEP_S), "grad_dtype": "f32",
                       "quantum": 2.0 ** -15, "fusion": args.fusion,
                       "value_is": "best params/s at the largest P that fits"},
            "peak": peak, "peak_kind": peak_kind, "clocks": clk.summary(), "sweep": points}
    print(json.dumps(line), flush=True)
    return 0


def bench_baselines(opt, wl, grads, dev, warmup=2, steps=5):
    """Per-step time of the dense AdamS and AdamW baselines (plain mean of the
    W gradients, every coordinate updated) on the same device buffers."""
    import torch

    P, W, G = wl.P, wl.W, _grad_bytes(wl)
    out = {}
    v = torch.zeros(P, dtype=torch.float32, device=dev)
    st = torch.cuda.current_stream()
    for name, fn, state_bytes in (("dense_adams", lambda: opt.dense_adams_step(grads), 16),
                                  ("adamw", lambda: opt.adamw_step(grads, v), 24)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(st)
        for _ in range(steps):
            fn()
        ev1.record(st)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / steps
        alg = W * P * G + state_bytes * P
        out[name] = {"ms_per_step": ms, "params_per_s": P / (ms / 1000.0),
                     "hbm_gbs": alg / (ms / 1000.0) / 1e9}
    del v
    # union-mask gradient top-k (each worker's own top-k, OR-ed into one mask):
    # step time and how much the union fills in relative to one worker's k
    kw = (P * (1000000 - round(wl.sparsity * 1e6)) + 999999) // 1000000
    sizes, ms_list = [], []
    for it in range(warmup + 3):
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(st)
        ku = opt.union_step(grads)
        ev1.record(st)
        torch.cuda.synchronize()
        if it >= warmup:
            sizes.append(ku)
            ms_list.append(ev0.elapsed_time(ev1))
    out["union_topk"] = {"ms_per_step": sum(ms_list) / len(ms_list), "k_worker": kw,
                         "k_union": sizes, "fill_in": sum(sizes) / len(sizes) / kw,
                         "union_density": sum(sizes) / len(sizes) / P,
                         "scape_k": opt.k}
    opt._union_ws = None
    opt._union_cap = None
    torch.cuda.empty_cache()
    return out


def bench_e2e(opt, wl, dev_grads, steps, dev, shared_source=False):
    """Same step through scape_step_host: per step the W gradients are copied
    from pinned host memory, the step and refresh run, and w[P] is copied back."""
    import torch

    P, W = opt.P, wl.W  # the parameters this rank's handle covers
    gdt = dev_grads[0].dtype
    esz = dev_grads[0].element_size()
    need = W * P * esz + 4 * P
    near = _bind_near_gpu(dev)
    if not shared_source and _mem_available() > 3 * need:
        host = [torch.empty(P, dtype=gdt).pin_memory() for _ in range(W)]
        shared = False
    else:
        # too little host memory for W distinct pinned buffers: one pinned
        # buffer is the source of every worker (the same bytes are copied)
        host = [torch.empty(P, dtype=gdt).pin_memory()] * W
        shared = True
    for h_, d in zip(host, dev_grads):
        h_.copy_(d)
    out = torch.empty(P, dtype=torch.float32).pin_memory()
    st = torch.cuda.current_stream()
    # untimed: the first transfers from freshly pinned pages, and the library's
    # copy stream and events, are one-time costs
    for _ in range(2):
        opt.step_host(host, dev_grads, out)
    st.synchronize()
    times = []
    for _ in range(steps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        opt.step_host(host, dev_grads, out)
        st.synchronize()
        times.append(time.perf_counter() - t0)
    # mean over the steps: on some boxes the host link alternates between a
    # fast and a slow transfer batch (plain copies show the same), so an even
    # number of steps and their mean give the long-run rate; every step is
    # listed in ms_each
    secs = sum(times) / len(times)
    # the host link alone on this machine: the same uploads and download as plain
    # copies with no kernels, for reading the end-to-end number against it
    link = []
    for _ in range(max(steps, 2)):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for h_, d in zip(host, dev_grads):
            d.copy_(h_, non_blocking=True)
        out.copy_(opt.params, non_blocking=True)
        torch.cuda.synchronize()
        link.append(time.perf_counter() - t0)
    del host
    return {"value": P / secs, "unit": UNIT, "h2d_bytes_per_step": W * P * esz,
            "d2h_bytes_per_step": 4 * P, "ms_per_step": 1000 * secs,
            "ms_each": [1000 * x for x in times],
            "host_cores": f"{len(near)} cores local to the GPU" if near else "unbound",
            "min_ms": 1000 * min(times),
            "link_only_ms": {"mean": 1000 * sum(link) / len(link), "min": 1000 * min(link),
                             "each": [1000 * x for x in link]},
            "shared_host_source": shared}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="llama500m")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--cpu-steps", type=int, default=5,
                    help="lagged sparse steps of the CPU oracle leg (0 to skip)")
    ap.add_argument("--other-steps", type=int, default=10,
                    help="timed steps of each of the two other workload shapes (0 to skip)")
    ap.add_argument("--residuals", default="device", choices=["device", "host"],
                    help="error-feedback buffers in HBM or in pinned host memory")
    ap.add_argument("--staging-rows", type=int, default=None,
                    help="with --residuals host: device rows staging the residuals "
                         "(default min(W, 12); 0 = kernels access host memory in place)")
    ap.add_argument("--fusion", default="auto", choices=sorted(FUSION) + ["auto"],
                    help="what the compaction pass also does: none (separate reduce and "
                         "adams_sparse), sum (writes g_bar), update (also AdamS); auto: the "
                         "library's default for the density (update from 5%% selected)")
    ap.add_argument("--baselines", type=int, default=1,
                    help="also time the dense AdamS and AdamW baselines (0 to skip)")
    ap.add_argument("--exchange", action="store_true",
                    help="time the exchange-based multi-rank step instead (each rank owns W/N "
                         "workers and optimizer shards; NCCL all-to-all + all-gathers)")
    ap.add_argument("--sweep", action="store_true",
                    help="run the flat sweep (2^e fp32 parameters, W in {1, 8, 32}, sparsity "
                         "in {0, 90, 99, 99.9}%%, 256-level gradients) instead")
    ap.add_argument("--sweep-exps", type=int, nargs="+", default=[20, 22, 24, 26, 28, 30],
                    help="exponents e of the flat sweep's P = 2^e")
    ap.add_argument("--P", type=int, default=None,
                    help="with --workload custom: flat parameter count")
    ap.add_argument("--workers", type=int, default=8, help="with --workload custom: W")
    ap.add_argument("--sparsity", type=float, default=0.99, help="with --workload custom")
    ap.add_argument("--grad-dtype", default="bf16", choices=["bf16", "f32"],
                    help="with --workload custom")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from sparse_communication_sharded_gb300 import synth
    if args.sweep:
        if args.impl == "reference":
            ap.error("--sweep times the GPU path only")
        return bench_sweep(args)
    if args.workload == "custom":
        if not args.P:
            ap.error("--workload custom needs --P")
        wl = synth.Workload(f"custom_p{args.P}_w{args.workers}_s{args.sparsity}",
                            (("flat", args.P),), W=args.workers, sparsity=args.sparsity,
                            steps=args.steps, grad_dtype=args.grad_dtype)
    else:
        wl = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        return bench_reference(args, wl)
    if args.exchange:
        return bench_exchange(args, wl)
    return bench_gpu(args, wl)


if __name__ == "__main__":
    sys.exit(main())
