"""Benchmark of the SCAPE sharded optimizer step on GB300.

One step = the whole hot path over one batch of synthetic per-worker gradients:
scape_step (error-feedback compaction, ordered sparse reduce, sparse AdamS)
plus scape_refresh_mask (the partitioned top-k that the next step uses).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama500m]
    python bench.py --impl reference ...     # the CPU oracle, same metric

Rank 0 prints one JSON line.  With N > 1 (torchrun) every rank runs its own
independent problem of the same shape (optimizer shards are independent), no
data-path collective runs, and the value is the sum over ranks of the
parameters stepped divided by the slowest rank's time (weak scaling).
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


def algorithmic_bytes(wl, k, fusion="sum"):
    """Bytes the method must move per step, by kernel (see the design notes).
    fusion "sum": the compaction also writes g_bar, so the packed buffers are
    written but never re-read; "update": it also updates w and m at the k
    selected coordinates (no index list or g_bar to read back)."""
    P, W, G = wl.P, wl.W, _grad_bytes(wl)
    ntiles = (P + 2047) // 2048
    ef = W * P * (G + 8) + P / 8 + 4 * ntiles + 4 * k * W
    refresh = 4 * P + P / 8 + P / 8 + 4 * k
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


# --------------------------------------------------------------------- oracle sample
def run_oracle_sample(wl, steps, seed=0, device=None):
    """Time the CPU oracle (single thread) on one optimizer shard of the
    workload: a dense first step (untimed), then `steps` lagged sparse steps
    with their mask refreshes (timed).  Gradients are drawn on `device` (GPU if
    given) and copied to host memory.  Returns (params/s, seconds, n_shard)."""
    import numpy as np
    import torch

    from oracle import oracle as O
    from sparse_communication_sharded_gb300 import synth

    start, ks = O.layout(wl.P, wl.W, wl.sparsity)
    sh = wl.W // 2
    lo, hi = int(start[sh]), int(start[sh + 1])
    n = hi - lo
    gdev = device if device is not None else "cpu"
    gen = synth.GradientStream(wl, seed=seed, device=gdev, P=n, offset=lo)
    w0 = synth.init_params(n, seed=seed, device=gdev).cpu().numpy()
    st = O.new_state(w0, wl.W, wl.sparsity, O.Hyper(),
                     shard_start=np.array([0, n], np.int64), shard_k=np.array([ks[sh]], np.int64))
    bufs = gen.alloc()

    def host_grads():
        gen.next_into(bufs)
        return [synth.to_numpy_grad(b) for b in bufs]

    O.advance(st, host_grads(), keep=())          # dense first step, untimed
    total = 0.0
    for _ in range(steps):
        g = host_grads()
        t0 = time.perf_counter()
        O.advance(st, g, keep=())
        total += time.perf_counter() - t0
    del bufs
    if device is not None:
        torch.cuda.empty_cache()
    return n * steps / total, total, n


# --------------------------------------------------------------------- reference arm
def bench_reference(args, wl):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import torch
    dev = torch.device("cuda:0") if torch.cuda.is_available() else None
    steps = max(1, args.steps)
    rate, secs, n = run_oracle_sample(wl, steps, device=dev)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": ws,
        "steps": steps, "warmup": args.warmup, "ms_per_step": 1000.0 * secs / steps * wl.P / n,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl.name, "P": wl.P, "W": wl.W, "sparsity": wl.sparsity,
                   "grad_dtype": wl.grad_dtype},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"one optimizer shard ({n} params x {wl.W} workers), "
                                   f"{steps} lagged sparse steps + refreshes after an untimed "
                                   f"dense step; ms_per_step scaled to the full P"},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------- GPU arm
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
    seed = 1000 * rank
    params = synth.init_params(P, seed=seed, device=dev)
    opt = pkg.Scape(params, W, wl.sparsity, layer_numel=[n for _, n in wl.layers],
                    grad_dtype=gdt, residuals=args.residuals, staging_rows=args.staging_rows)
    opt.set_fusion(FUSION[args.fusion])
    gen = synth.GradientStream(wl, seed=seed, device=dev)
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
    step_ms, wall = [], []
    st = torch.cuda.current_stream()
    with ClockSampler(local) as clk:
        for _ in range(args.steps):
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
    opt.profile(False)

    my_ms = sum(step_ms) / len(step_ms)
    t_max = my_ms
    if ws > 1:
        tt = torch.tensor([my_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t_max = float(tt.item())
    value = ws * P / (t_max / 1000.0)
    alg = algorithmic_bytes(wl, opt.k, fusion=args.fusion)
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

    # dense baselines on the same workload and buffers (after the SCAPE timing)
    baselines = None
    if args.baselines and ws == 1:
        baselines = bench_baselines(opt, wl, grads, dev)

    # end to end through the C ABI from pinned host memory
    e2e = None
    if args.e2e_steps > 0:
        e2e = bench_e2e(opt, wl, grads, args.e2e_steps, dev, shared_source=ws > 1)
        if ws > 1:
            # whole job: every rank stepped P parameters; the slowest rank sets the time
            t_e2e = multirank.max_over_ranks(e2e["ms_per_step"], device=dev)
            e2e["ms_per_step"] = t_e2e
            e2e["value"] = ws * P / (t_e2e / 1000.0)
            e2e["h2d_bytes_per_step"] *= ws
            e2e["d2h_bytes_per_step"] *= ws

    cpu = None
    if rank == 0 and ws == 1 and args.cpu_steps > 0:
        rate, secs, n = run_oracle_sample(wl, args.cpu_steps, device=dev)
        cpu = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"one optimizer shard ({n} of {P} params, {W} workers), "
                         f"{args.cpu_steps} lagged sparse steps + refreshes after an untimed "
                         f"dense step, single-threaded C, {secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.name, "P": P, "W": W, "sparsity": wl.sparsity,
                       "k": opt.k, "grad_dtype": wl.grad_dtype, "state_dtype": "f32",
                       "residuals": args.residuals, "fusion": args.fusion,
                       "staging_rows": (opt.staging.numel() // (4 * ((P + 63) // 64 * 64))
                                        if opt.staging is not None else 0),
                       "l2": "inputs larger than L2 (gradients + residuals far beyond 129 MB)",
                       "parallelism": f"{ws} independent problems (weak)"},
            "hbm_gbs": alg["total"] / (t_max / 1000.0) / 1e9,
            "hbm_frac": alg["total"] / (t_max / 1000.0) / 1e9 / peak,
            "alg_bytes_per_step": alg["total"],
            "roofline": {"kernel": "ef_compact", "bound": "hbm", "achieved": ef_gbs,
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": ef_gbs / peak, "traffic": traffic,
                         "alg_bytes_per_launch": alg["ef_compact"], "ms_per_launch": ef_avg},
            "kernels": kernels,
            "kernels_measured_over": f"{n_break} profiled steps after the timed ones",
            "refresh_ms_per_step": refresh_ms,
            "mask_churn_per_refresh": churn,
            "wall_ms_per_step": 1000.0 * sum(wall) / len(wall),
            "gpu_launches": launches,
            "clocks": clocks,
            "e2e": e2e,
            "baselines": baselines,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    opt.close()
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

    P, W = wl.P, wl.W
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
    ap.add_argument("--cpu-steps", type=int, default=2)
    ap.add_argument("--residuals", default="device", choices=["device", "host"],
                    help="error-feedback buffers in HBM or in pinned host memory")
    ap.add_argument("--staging-rows", type=int, default=None,
                    help="with --residuals host: device rows staging the residuals "
                         "(default min(W, 12); 0 = kernels access host memory in place)")
    ap.add_argument("--fusion", default="sum", choices=sorted(FUSION),
                    help="what the compaction pass also does: none (separate reduce and "
                         "adams_sparse), sum (writes g_bar), update (also AdamS)")
    ap.add_argument("--baselines", type=int, default=1,
                    help="also time the dense AdamS and AdamW baselines (0 to skip)")
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
    return bench_gpu(args, wl)


if __name__ == "__main__":
    sys.exit(main())
