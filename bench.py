#!/usr/bin/env python3
"""Benchmark of the fused SH + CG tensor product + receiver sum layer.

One step = one eqmp_fused call (the whole hot path: CSR walk, SH in
registers, sender-row gather, CG tensor product, receiver sum, store) over
one seeded synthetic graph.  Headline workload: 1000 atoms, 32 channels,
~16.5 neighbours per atom, shared per-path weights, fp32 - the workload the
Batmobile blog quotes (1000 atoms, 32 channels, about 20 neighbours).

Prints ONE JSON line (rank 0):
  value        edges/s over all ranks, inputs resident in HBM, L2 flushed
               (256 MB write) before every timed step, device time of the
               layer kernel from CUDA events on the launching stream (the
               host queues each group of steps behind a short GPU spin, so
               host-side enqueue jitter never shows up as device time);
  e2e          the same metric through the public API with pinned host
               buffers: H2D of the step's inputs, the layer, D2H of out
               (for eqmp_fused: one eqmp_fused_staged call per step);
  roofline     t_roof = max(FMA count / FP32 peak, compulsory bytes / HBM
               peak); frac = t_roof / measured time, bound = the larger
               term.  FMA count of the lowest-FMA exact schedule (shared
               weights: accumulate x (x) Y, contract once per receiver;
               radial weights: the aligned-frame schedule), FP32 peak = the
               higher of the derived one (SM count x 128 lanes x 2 flops x
               max SM clock) and the measured one (eqmp_fp32_peak_probe);
  workloads    the same measurement (time, roofline, clocks) for the
               100k-atom, the dense bf16 and the radial-weight workloads,
               the 100k-atom workload renumbered in Morton order, and the
               rows past the layer: the backward pass, the open and the
               periodic radius graph, the degree-6 layer;
  cpu_baseline the CPU oracle (numpy, fp64) on a bounded sample of the same
               workload on this host's cores, plus one-thread runs of the
               tiny, pages and radial workloads.
--impl reference times the CPU oracle alone (the reference arm).
Multi-GPU: independent replicas (weak scaling), no collective on the data
path; barrier + max over ranks for timing.
"""
import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "edges/s fused SH+CG-TP+scatter (1k atoms, C=32, ~20 nbrs); % of roofline"
METRIC_GRAPH = "edges/s radius graph (CSR by receiver, edge vectors)"
FLUSH_BYTES = 256 << 20
HEADLINE = "pages_1k_c32"
# Measured beside the headline in the default run (the other full-size configurations).
EXTRA_WORKLOADS = ("scale_100k_c64", "dense_10k_c128_bf16", "radial_1k_c32", "scale_100k_c64_morton")
# The rows past the layer, measured in the same run: (label, workload, pass).
EXTRA_PASSES = (("backward pages_1k_c32", "pages_1k_c32", "backward"),
                ("backward radial_1k_c32", "radial_1k_c32", "backward"),
                ("backward scale_100k_c64", "scale_100k_c64", "backward"),
                ("radius graph scale_100k_c64", "scale_100k_c64", "graph"),
                ("periodic radius graph scale_100k_c64", "scale_100k_c64", "graph_pbc"),
                ("degree-6 layer pages_1k_c32", "pages_1k_c32", "lmax6"))
# One-thread oracle runs (the small configurations).
SINGLE_THREAD_WORKLOADS = ("tiny_64", "pages_1k_c32", "radial_1k_c32")
GROUP = 32  # timed steps queued behind one GPU spin
PIPE = 6  # streams (and buffer sets) of the pipelined end-to-end measurement
# DRAM bytes per launch of the layer kernel from the ncu capture recorded in
# profiles/ (None until captured for the current kernel version).
# Keyed by (workload, kernel version); a changed kernel gets a new version
# tag, which makes its entry missing (traffic null) until re-captured.
KERNEL_VERSION = {"shared": "k_shared-pairs-v5", "radial": "k_so2-pairs-v7"}
NCU_TRAFFIC = {
    ("pages_1k_c32", "k_shared-pairs-v5"): 2357504 + 0,
    ("scale_100k_c64", "k_shared-pairs-v5"): 6207318016 + 407371008,
    ("dense_10k_c128_bf16", "k_shared-pairs-v5"): 48796160 + 11876864,
    ("radial_1k_c32", "k_so2-v4"): 2888704 + 0,
    ("radial_1k_c32", "k_so2-v5"): 2899456 + 0,
    ("radial_1k_c32", "k_so2-pairs-v6"): 2906368 + 0,
    ("radial_1k_c32", "k_so2-pairs-v7"): 2906624 + 0,
    ("scale_100k_c64_morton", "k_shared-pairs-v5"): 1679304960 + 394390272,
}

# aligned-frame terms per degree (one per output order and path with m2 = 0)
ALIGNED_TERMS = {3: 111, 4: 272, 5: 565, 6: 1036}


def fma_count(wl):
    """FMAs of the dense schedules of the l <= 3 layer (per launch).

    shared weights: 256*C per edge (A += x (x) Y) + (611 + 156)*C per receiver
    (the lowest-FMA exact schedule for shared weights);
    radial weights: (611 + 156 + 272)*C + 611 per edge (W = R.M per path and
    channel, CG terms, weighted sum; the Y-side products shared by channels).
    """
    C, E, N = wl.channels, wl.n_edges, wl.n_atoms
    if wl.w is not None:
        return 256 * C * E + 767 * C * N
    return ((611 + 156 + 272) * C + 611) * E


def sum_rot(l_max):
    """FMAs of one rotation of all blocks l = 1..l_max: sum (2l+1)^2."""
    return sum((2 * l + 1) ** 2 for l in range(1, l_max + 1))


def aligned_fma_count(wl, l_max):
    """FMAs of the aligned-frame schedule at degree l_max (per launch):
    rotate in and out (2 sum (2l+1)^2), one FMA per aligned term, and for
    radial weights 8 per path; per edge and channel.  At l_max = 3 with
    radial weights this is 549 per edge and channel, the lowest-FMA exact
    schedule for per-edge weights (the dense one needs 1039)."""
    from equivariant_gnn_message_gb300.inputs import n_paths

    per = 2 * sum_rot(l_max) + ALIGNED_TERMS[l_max] + (8 * n_paths(l_max) if wl.w is None else 0)
    return per * wl.channels * wl.n_edges


def compulsory_bytes(wl):
    """x read once, vec, src, offsets, weights (or R and M), out written once."""
    s = 2 if wl.storage == "bf16" else 4
    C, E, N = wl.channels, wl.n_edges, wl.n_atoms
    nc = wl.x.shape[2]
    b = N * C * nc * s + 12 * E + 4 * E + 4 * (N + 1) + N * C * nc * s
    b += 4 * 34 * C if wl.w is not None else 32 * E + 4 * 8 * 34 * C
    return b


def layer_flops(wl, which, l_max):
    """(algorithmic flops per launch, basis name, extra) for the roofline."""
    if which == "backward":
        # three forward-sized contractions (dx, the weight gradient, dY) of
        # the dense schedule plus the SH Jacobian (48 FMA per edge)
        return 2.0 * (3 * fma_count(wl) + 48 * wl.n_edges), "backward: 3 x forward schedule + SH Jacobian", {}
    if l_max != 3 or wl.w is None:
        f = 2.0 * aligned_fma_count(wl, l_max)
        extra = {}
        if l_max == 3:
            extra["flops_dense_basis"] = 2.0 * fma_count(wl)
        return f, f"aligned frame (2*rot + {ALIGNED_TERMS[l_max]} terms" + \
            (" + 8 per path" if wl.w is None else "") + " per edge and channel)", extra
    return 2.0 * fma_count(wl), "accumulate-then-contract (256*C per edge + 767*C per receiver)", {}


def roofline(flops, nbytes, ms, fp32_peak, hbm_peak, kernel, traffic, basis, extra=None):
    """t_roof = max(flops / FP32 peak, bytes / HBM peak); frac = t_roof / t."""
    t = ms * 1e-3
    t_alu = flops / (fp32_peak * 1e12)
    t_hbm = nbytes / (hbm_peak * 1e9)
    if t_alu >= t_hbm:
        r = {"bound": "alu", "achieved": flops / t / 1e12, "peak": fp32_peak, "unit": "TFLOP/s"}
    else:
        r = {"bound": "hbm", "achieved": nbytes / t / 1e9, "peak": hbm_peak, "unit": "GB/s"}
    r.update({"frac": max(t_alu, t_hbm) / t, "traffic": traffic, "traffic_unit": "bytes/launch",
              "kernel": kernel, "flops": flops, "compulsory_bytes": nbytes, "fma_basis": basis,
              "t_alu_us": t_alu * 1e6, "t_hbm_us": t_hbm * 1e6,
              "hbm_gbs_compulsory": nbytes / t / 1e9})
    for k, v in (extra or {}).items():
        if k == "flops_dense_basis":
            r["frac_dense_basis"] = v / (fp32_peak * 1e12) / t
        else:
            r[k] = v
    return r


class ClockSampler:
    """nvidia-smi clock / throttle samples, 100 ms apart, in a thread."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [p.strip() for p in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self._t is not None:
            self._t.join(timeout=2)

    def summary(self, t0, t1, pad=0.3):
        win = [s for (t, s) in self.samples if t0 - pad <= t <= t1 + pad] or [s for _, s in self.samples]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(s[1]) for s in win if num(s[1]) is not None]
        mx = [num(s[2]) for s in win if num(s[2]) is not None]
        pw = [num(s[3]) for s in win if len(s) > 3 and num(s[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4) if len(s) > 5 + i and s[5 + i] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(win),
                "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------- CPU oracle
def _oracle_chunk(args):
    """Child-process worker: oracle on a receiver subset, `reps` times
    (single-threaded BLAS); returns the wall time of the oracle calls."""
    name, receivers, l_max, reps = args
    from equivariant_gnn_message_gb300.inputs import make_workload
    from oracle import layer

    wl = make_workload(name, l_max=l_max)
    kw = dict(w=wl.w) if wl.w is not None else dict(R=wl.R, M=wl.M)
    receivers = np.arange(wl.n_atoms) if receivers is None else np.asarray(receivers)
    t = time.perf_counter()
    for _ in range(reps):
        layer.message_pass(wl.vec, wl.x, wl.off, wl.src, receivers=receivers, **kw)
    return time.perf_counter() - t


def make_pool(cores):
    """Spawned worker pool for the oracle, one single-threaded worker per core."""
    import multiprocessing as mp

    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    old = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "1"
    try:
        return mp.get_context("spawn").Pool(cores)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def cpu_oracle_rate(name, wl, seconds_target=12.0, pool=None, cores=1):
    """edges/s of the CPU oracle on a bounded sample of the workload's receivers.

    The sample is a contiguous run of receivers from the start of the CSR
    (all with their full edge lists), sized from a short probe so that the
    whole measurement takes about `seconds_target` seconds of wall time.
    """
    from oracle import layer

    kw = dict(w=wl.w) if wl.w is not None else dict(R=wl.R, M=wl.M)
    probe_r = max(1, min(wl.n_atoms, 8))
    t = time.perf_counter()
    layer.message_pass(wl.vec, wl.x, wl.off, wl.src, receivers=np.arange(probe_r), **kw)
    rate1 = max(1.0, (wl.off[probe_r] - wl.off[0]) / max(1e-6, time.perf_counter() - t))
    want_edges = int(rate1 * seconds_target * cores)
    n_recv = int(np.searchsorted(wl.off - wl.off[0], want_edges))
    n_recv = max(1, min(wl.n_atoms, n_recv))
    receivers = np.arange(n_recv)
    edges = int(wl.off[n_recv] - wl.off[0])
    # a workload smaller than the target is run several times over
    reps = int(min(50, max(1, round(want_edges / max(1, edges)))))
    t = time.perf_counter()
    if pool is not None and cores > 1:
        parts = np.array_split(receivers, cores)
        # each worker times its own oracle calls (graph generation excluded);
        # the parallel wall time is the slowest worker's
        l_max = int(round(np.sqrt(wl.x.shape[2]))) - 1
        wall = max(pool.map(_oracle_chunk, [(name, p.tolist(), l_max, reps) for p in parts if len(p)]))
    else:
        for _ in range(reps):
            layer.message_pass(wl.vec, wl.x, wl.off, wl.src, receivers=receivers, **kw)
        wall = time.perf_counter() - t
    return (edges * reps / wall,
            f"receivers 0..{n_recv - 1} ({edges} edges of {wl.n_edges}) x {reps}, {wall:.1f} s wall")


def single_thread_rates(pool, names, seconds=2.5):
    """One worker of the pool (one thread) runs the oracle over every
    receiver of each small workload, repeated to about `seconds`."""
    from equivariant_gnn_message_gb300.inputs import make_workload

    res = []
    for name in names:
        E = make_workload(name).n_edges
        t1 = pool.apply(_oracle_chunk, ((name, None, 3, 1),))
        reps = max(1, int(round(seconds / max(t1, 1e-3))))
        wall = pool.apply(_oracle_chunk, ((name, None, 3, reps),))
        res.append({"workload": name, "value": E * reps / wall, "unit": "edges/s", "cores": 1,
                    "ms_per_layer": 1e3 * wall / reps,
                    "sample": f"all {E} edges x {reps}, {wall:.2f} s wall"})
    return res


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    pool = make_pool(cores)
    try:
        per_step = max(1.0, 150.0 / max(1, args.steps + args.warmup))
        for _ in range(args.warmup):
            cpu_oracle_rate(args.workload, wl, seconds_target=min(per_step, 2.0), pool=pool, cores=cores)
        rates = []
        t0 = time.perf_counter()
        for _ in range(args.steps):
            r, sample = cpu_oracle_rate(args.workload, wl, seconds_target=per_step, pool=pool, cores=cores)
            rates.append(r)
        total = time.perf_counter() - t0
    finally:
        pool.terminate()
    value = float(np.median(rates))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "edges/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * wl.n_edges / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, wl, args.entry, 1),
        "cpu_baseline": {"value": value, "unit": "edges/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "edges/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "timed_wall_s": round(total, 2),
    }
    print(json.dumps(line), flush=True)


def workload_config(name, wl, entry, world):
    return {"workload": name, "n_atoms": wl.n_atoms, "n_edges": wl.n_edges,
            "channels": wl.channels, "storage": wl.storage,
            "weights": "shared" if wl.w is not None else "radial", "entry": entry,
            "l2": "flushed (256 MB write) before every timed step",
            "parallelism": f"replicas x{world}"}


# ---------------------------------------------------------------- GPU timing
class Timer:
    """CUDA-event timing of `step` on `stream`, L2 flushed before each step.

    The host queues GROUP steps (flush, start event, step, end event) behind
    one GPU spin long enough to cover their enqueue time, so every step runs
    back to back on the device and the events hold device time only.
    """

    def __init__(self, torch, stream, flush):
        self.torch = torch
        self.stream = stream
        self.flush = flush
        self.host_s = 60e-6  # host enqueue time per step; refined by warm()

    def warm(self, step, n):
        torch = self.torch
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(n):
            self.flush.zero_()
            step()
        self.host_s = max(self.host_s, (time.perf_counter() - t) / max(1, n))
        torch.cuda.synchronize()

    def _spin(self, n_steps):
        sleep = getattr(self.torch.cuda, "_sleep", None)
        if sleep is not None:
            seconds = min(0.05, 3.0 * n_steps * self.host_s + 2e-4)
            sleep(int(seconds * 2.2e9))  # cycles at up to 2.2 GHz

    def run(self, step, steps):
        torch = self.torch
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        i = 0
        while i < steps:
            n = min(GROUP, steps - i)
            self._spin(n)
            for _ in range(n):
                self.flush.zero_()  # evict L2 between timed steps
                starts[i].record(self.stream)
                step()
                ends[i].record(self.stream)
                i += 1
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def copy_floor_ms(torch, h_in, d_in, h_out, d_out, pairs=20, reps=10):
    """Device time of one step's copies alone (h_in -> d_in on one stream,
    d_out -> h_out on another, recorded as a CUDA graph of `pairs` steps):
    the host link's floor for the pipelined end-to-end step."""
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s1):
        ev = torch.cuda.Event()
        ev.record(s1)
        s2.wait_event(ev)
        for _ in range(pairs):
            d_in.copy_(h_in, non_blocking=True)
            with torch.cuda.stream(s2):
                h_out.copy_(d_out, non_blocking=True)
        ev2 = torch.cuda.Event()
        ev2.record(s2)
        s1.wait_event(ev2)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * pairs)


def device_inputs(torch, wl, dev):
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    d = dict(vec=t(wl.vec), off=t(wl.off), src=t(wl.src), w=t(wl.w), R=t(wl.R), M=t(wl.M))
    if wl.storage == "bf16":
        d["x"] = torch.from_numpy(wl.x_bf16_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        d["x"] = t(wl.x)
    return d


def layer_step(eq, entry, l_max, d, out, Yb=None):
    wkw = dict(w=d["w"]) if d["w"] is not None else dict(R=d["R"], M=d["M"])
    if l_max != 3:
        return lambda: eq.eqmp_fused_lmax(l_max, d["vec"], d["x"], d["off"], d["src"], out=out, **wkw)
    if entry == "fused":
        return lambda: eq.eqmp_fused(d["vec"], d["x"], d["off"], d["src"], out=out, **wkw)
    if entry == "so2":
        return lambda: eq.eqmp_fused_so2(d["vec"], d["x"], d["off"], d["src"], out=out, **wkw)

    def two():
        eq.eqmp_sh(d["vec"], Yb)
        eq.eqmp_tp_scatter(Yb, d["x"], d["off"], d["src"], out=out, **wkw)
    return two


def kernel_version(wl, which, l_max, entry):
    if which == "backward":
        return "k_bwd-v1"
    if l_max != 3:
        return f"k_hl<{l_max}>-producer-v5"
    if entry == "tp_scatter":
        return "k_sh+" + ("k_shared-tp" if wl.w is not None else "k_radial")
    if entry == "so2":
        return KERNEL_VERSION["radial"]
    return KERNEL_VERSION["shared" if wl.w is not None else "radial"]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time the chosen workload only (no scale / dense / radial entries)")
    ap.add_argument("--entry", default="fused", choices=["fused", "tp_scatter", "so2"])
    ap.add_argument("--lmax", type=int, default=3,
                    help="4..6: the higher-degree layer (eqmp_fused_lmax) on the workload's graph")
    ap.add_argument("--pass", dest="which", default="forward", choices=["forward", "backward", "graph"],
                    help="backward: time eqmp_fused_backward (dx, dw or dR/dM, dvec) instead; "
                         "graph: time eqmp_radius_graph on the workload's atom positions")
    ap.add_argument("--pbc", action="store_true",
                    help="with --pass graph: periodic boundaries (eqmp_radius_graph_pbc) in the generator's cube")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    from equivariant_gnn_message_gb300.inputs import DENSITY, make_workload
    from equivariant_gnn_message_gb300.sharding import max_over_ranks

    wl = make_workload(args.workload, l_max=args.lmax)
    if args.pbc and args.which != "graph":
        raise SystemExit("--pbc goes with --pass graph")
    if args.lmax != 3 and (args.which != "forward" or wl.storage != "f32"):
        raise SystemExit("--lmax: forward pass on fp32 workloads only")
    if args.impl == "reference":
        run_reference(args, wl)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    # The oracle's process pool is started before the first CUDA call.
    pool, cores = None, os.cpu_count() or 1
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pool = make_pool(cores)

    import torch

    import __graft_entry__

    __graft_entry__.build()
    import equivariant_gnn_message_gb300 as eq

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    timer = Timer(torch, stream, flush)
    sampler = ClockSampler(local)
    sampler.start()

    d = device_inputs(torch, wl, dev)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    out = torch.empty((wl.n_atoms, wl.channels, (args.lmax + 1) ** 2), dtype=d["x"].dtype, device=dev)
    Yb = torch.empty((wl.n_edges, 16), dtype=torch.float32, device=dev) if args.entry == "tp_scatter" else None
    wkw = dict(w=d["w"]) if d["w"] is not None else dict(R=d["R"], M=d["M"])
    n_edges = wl.n_edges

    if args.which == "backward":
        if wl.storage != "f32":
            raise SystemExit("the backward pass takes fp32 features")
        so, se = eq.sender_view(wl.src, wl.n_atoms)
        gout = torch.randn((wl.n_atoms, wl.channels, 16), device=dev,
                           generator=torch.Generator(device=dev).manual_seed(0))
        need = ("x", "vec", "w") if d["w"] is not None else ("x", "vec", "R", "M")
        bargs = (d["vec"], d["x"], d["off"], d["src"], t(wl.dst), t(so), t(se), gout)
        step = lambda: eq.eqmp_fused_backward(*bargs, need=need, **wkw)
        launches_per_step = 3
    elif args.which == "graph":
        import ctypes

        lib = eq.load_library()
        N = wl.n_atoms
        box = None
        pos_np = wl.pos
        if args.pbc:  # the generator's cube as a periodic box; positions strictly inside it
            side = float((N / DENSITY) ** (1.0 / 3.0))
            box = (side, side, side)
            pos_np = np.minimum(np.maximum(wl.pos, np.float32(0)), np.nextafter(np.float32(side), np.float32(0)))
        g_pos = t(pos_np)
        g_ws = torch.empty(lib.eqmp_radius_graph_workspace_size(N), dtype=torch.uint8, device=dev)
        g_E = torch.empty(1, dtype=torch.int64, device=dev)
        g_out, E_graph = eq.eqmp_radius_graph(g_pos, wl.cutoff, box=box)
        g_off, g_src, g_vec = g_out["off"], g_out["src"], g_out["vec"]
        if box is None:
            graph_args = (g_pos.data_ptr(), N, ctypes.c_float(wl.cutoff), g_off.data_ptr(), g_src.data_ptr(),
                          g_vec.data_ptr(), None, None, E_graph, g_E.data_ptr(), g_ws.data_ptr(), g_ws.numel(),
                          stream.cuda_stream)
            step = lambda: lib.eqmp_radius_graph(*graph_args)
        else:
            g_img = g_out["img"]
            lengths = (ctypes.c_float * 3)(*box)
            graph_args = (g_pos.data_ptr(), N, ctypes.c_float(wl.cutoff), lengths, g_off.data_ptr(),
                          g_src.data_ptr(), g_vec.data_ptr(), g_img.data_ptr(), None, None, E_graph, g_E.data_ptr(),
                          g_ws.data_ptr(), g_ws.numel(), stream.cuda_stream)
            step = lambda: lib.eqmp_radius_graph_pbc(*graph_args)
        coop = N <= 16384  # the library's single cooperative launch covers up to 16,384 atoms
        launches_per_step = 1 if coop else 12
        n_edges = E_graph
    else:
        step = layer_step(eq, args.entry, args.lmax, d, out, Yb)
        launches_per_step = 2 if args.entry == "tp_scatter" else 1

    timer.warm(step, args.warmup)
    barrier()
    if eq.eqmp_device_error() != 0:
        raise RuntimeError("device watchdog tripped during warm-up")
    barrier()
    t0 = time.time()
    kernel_ms = timer.run(step, args.steps)
    barrier()
    t1 = time.time()
    ms = max_over_ranks(float(np.mean(kernel_ms)))

    # ---- e2e through the public API with pinned host buffers.  The step's
    # inputs sit in one pinned host block (each array 256-byte aligned) and
    # go over in one host->device copy; the result comes back in one copy.
    e2e_ms, h2d, d2h = None, 0, 0
    pipe_sets, e2e_serial_ms, e2e_mode, e2e_copy_floor = None, None, None, None
    if args.which == "forward":
        parts = {"vec": wl.vec, "off": wl.off, "src": wl.src,
                 "x": wl.x_bf16_bits.view(np.int16) if wl.storage == "bf16" else wl.x}
        for k in ("w", "R", "M"):
            if getattr(wl, k) is not None:
                parts[k] = getattr(wl, k)
        layout, nbytes = {}, 0
        for k, a in parts.items():
            a = np.ascontiguousarray(a)
            layout[k] = (nbytes, a.dtype, a.shape)
            nbytes = (nbytes + a.nbytes + 255) // 256 * 256
        h_pack = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        hp = h_pack.numpy()
        for k, a in parts.items():
            o, dt, shp = layout[k]
            a = np.ascontiguousarray(a)
            hp[o:o + a.nbytes] = a.view(np.uint8).reshape(-1)
        d_pack = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        tdt = {np.dtype(np.float32): torch.float32, np.dtype(np.int32): torch.int32,
               np.dtype(np.int16): torch.int16}

        def dview(k):
            o, dt, shp = layout[k]
            n = int(np.prod(shp)) * dt.itemsize
            return d_pack[o:o + n].view(tdt[dt]).view(shp)

        d_in = {k: dview(k) for k in parts}
        d_in["x"] = d_in["x"].view(torch.bfloat16) if wl.storage == "bf16" else d_in["x"]
        for k in ("w", "R", "M"):
            d_in.setdefault(k, None)
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = sum(np.ascontiguousarray(a).nbytes for a in parts.values())
        d2h = h_out.numel() * h_out.element_size()
        layer_e2e = layer_step(eq, args.entry, args.lmax, d_in, out, Yb)
        if args.entry == "fused" and args.lmax == 3:
            # one C-ABI call per step: the packed inputs' host-to-device
            # copy, the layer, the result's device-to-host copy
            e2e_api = "eqmp_fused_staged"

            def staged(dp, di, o, ho, st=None):
                # checked and marshalled once; each step is the C call alone
                return eq.eqmp_fused_staged(h_pack, dp, di["vec"], di["x"], di["off"], di["src"], o, ho,
                                            w=di["w"], R=di["R"], M=di["M"], stream=st, prepare=True)

            e2e_step = staged(d_pack, d_in, out, h_out, stream)

            # the same step on PIPE streams, one buffer set each: step k's
            # copies run while earlier steps' layers do
            pipe_sets = [(d_pack, d_in, out, h_out)]
            for _ in range(PIPE - 1):
                dp2 = torch.empty(nbytes, dtype=torch.uint8, device=dev)
                di2 = {k: None if v is None else dp2[v.data_ptr() - d_pack.data_ptr():][:v.numel() * v.element_size()]
                       .view(v.dtype).view(v.shape) for k, v in d_in.items()}
                pipe_sets.append((dp2, di2, torch.empty_like(out), torch.empty_like(h_out).pin_memory()))
        else:
            e2e_api = "torch copies + " + {"so2": "eqmp_fused_so2", "tp_scatter": "eqmp_sh + eqmp_tp_scatter"}.get(
                args.entry, "eqmp_fused_lmax")

            def e2e_step():
                d_pack.copy_(h_pack, non_blocking=True)
                layer_e2e()
                h_out.copy_(out, non_blocking=True)
    elif args.which == "graph":
        e2e_api = "torch copies + eqmp_radius_graph" + ("_pbc" if box is not None else "")
        h_pos = torch.from_numpy(np.ascontiguousarray(pos_np)).pin_memory()
        g_res = (g_off, g_src, g_vec) + ((g_img,) if box is not None else ())
        h_outs = [torch.empty(a.shape, dtype=a.dtype).pin_memory() for a in g_res]
        h2d = h_pos.numel() * 4
        d2h = sum(a.numel() * a.element_size() for a in h_outs)

        def e2e_step():
            g_pos.copy_(h_pos, non_blocking=True)
            step()
            for h, dd in zip(h_outs, g_res):
                h.copy_(dd, non_blocking=True)
    if args.which != "backward":
        for _ in range(3):
            e2e_step()
        barrier()
        e_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        e_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            e_s[i].record(stream)
            e2e_step()
            e_e[i].record(stream)
        barrier()
        e2e_ms = max_over_ranks(float(np.mean([s.elapsed_time(e) for s, e in zip(e_s, e_e)])))
        e2e_mode = "serial: one stream, L2 flushed between steps, per-step events"
        if pipe_sets is not None:
            # K steps on PIPE streams, each step's inputs copied in and its
            # result copied out and read on the host (after its step's event)
            # before its buffers take step k+PIPE; one span from the first
            # copy to the last result
            e2e_serial_ms = e2e_ms
            streams = [torch.cuda.Stream(device=dev) for _ in range(PIPE)]
            # each buffer set's step recorded once as a CUDA graph (eqmp_plan_staged)
            plans = [eq.eqmp_plan_staged(h_pack, dp, di["vec"], di["x"], di["off"], di["src"], o, ho,
                                         w=di["w"], R=di["R"], M=di["M"]) for dp, di, o, ho in pipe_sets]
            runs = [lambda b=b: plans[b].launch(streams[b]) for b in range(PIPE)]
            host_bytes = [ps[3].view(torch.uint8).numpy().reshape(-1) for ps in pipe_sets]
            for i in range(2 * PIPE):
                runs[i % PIPE]()
            torch.cuda.synchronize()
            barrier()
            t_beg, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t_beg.record(streams[0])
            for st_ in streams[1:]:
                st_.wait_event(t_beg)
            done = [torch.cuda.Event() for _ in range(args.steps)]
            check = 0.0
            for i in range(args.steps):
                if i >= PIPE:
                    done[i - PIPE].synchronize()
                    check += float(host_bytes[i % PIPE][0])  # step i-PIPE's result, read on the host
                runs[i % PIPE]()
                done[i].record(streams[i % PIPE])
            for i in range(max(0, args.steps - PIPE), args.steps):
                streams[0].wait_event(done[i])
            t_end.record(streams[0])
            torch.cuda.synchronize()
            barrier()
            e2e_ms = max_over_ranks(t_beg.elapsed_time(t_end) / args.steps)
            e2e_mode = (f"pipelined: {PIPE} streams, one device block each, each step one CUDA graph launch "
                        "(eqmp_plan_staged), no L2 flush (inputs arrive by copy)")
            e2e_api = "eqmp_plan_staged + eqmp_plan_launch"
            for p_ in plans:
                p_.destroy()
            e2e_copy_floor = copy_floor_ms(torch, h_pack, pipe_sets[0][0], pipe_sets[0][3], pipe_sets[0][2])

    # ---- the other full-size workloads, same timing, one entry each
    extra = []
    run_extra = (args.workload == HEADLINE and args.which == "forward" and args.lmax == 3
                 and args.entry == "fused" and not args.no_workloads)
    if run_extra:
        del d

        def timed(step_fn):
            timer.warm(step_fn, args.warmup)
            barrier()
            ta = time.time()
            k = timer.run(step_fn, args.steps)
            barrier()
            tb = time.time()
            return max_over_ranks(float(np.mean(k))), k, (ta, tb)

        wl_cache = {}

        def get_wl(name, l_max=3):
            if (name, l_max) not in wl_cache:
                wl_cache[(name, l_max)] = make_workload(name, l_max=l_max)
            return wl_cache[(name, l_max)]

        for name in EXTRA_WORKLOADS:
            xw = get_wl(name)
            xd = device_inputs(torch, xw, dev)
            xo = torch.empty((xw.n_atoms, xw.channels, 16), dtype=xd["x"].dtype, device=dev)
            xms, xk, tt = timed(layer_step(eq, "fused", 3, xd, xo))
            extra.append(dict(name=name, label=name, kind="forward", wl=xw, ms=xms, kernel_ms=xk, t=tt,
                              launches=1, n_edges=xw.n_edges))
            del xd, xo
            torch.cuda.empty_cache()

        for label, name, kind in EXTRA_PASSES:
            xw = get_wl(name, 6 if kind == "lmax6" else 3)
            entry = dict(name=name, label=label, kind=kind, wl=xw, n_edges=xw.n_edges)
            if kind == "backward":
                xd = device_inputs(torch, xw, dev)
                so, se = eq.sender_view(xw.src, xw.n_atoms)
                g = torch.randn((xw.n_atoms, xw.channels, 16), device=dev,
                                generator=torch.Generator(device=dev).manual_seed(0))
                need = ("x", "vec", "w") if xw.w is not None else ("x", "vec", "R", "M")
                bkw = dict(w=xd["w"]) if xw.w is not None else dict(R=xd["R"], M=xd["M"])
                bargs = (xd["vec"], xd["x"], xd["off"], xd["src"], t(xw.dst), t(so), t(se), g)
                fn = lambda: eq.eqmp_fused_backward(*bargs, need=need, **bkw)
                entry["launches"] = 3
            elif kind in ("graph", "graph_pbc"):
                import ctypes

                lib = eq.load_library()
                Ng = xw.n_atoms
                gbox = None
                gpos = xw.pos
                if kind == "graph_pbc":
                    side = float((Ng / DENSITY) ** (1.0 / 3.0))
                    gbox = (side, side, side)
                    gpos = np.minimum(np.maximum(xw.pos, np.float32(0)), np.nextafter(np.float32(side), np.float32(0)))
                xpos = t(gpos)
                gws = torch.empty(lib.eqmp_radius_graph_workspace_size(Ng), dtype=torch.uint8, device=dev)
                gE = torch.empty(1, dtype=torch.int64, device=dev)
                gout, Eg = eq.eqmp_radius_graph(xpos, xw.cutoff, box=gbox)
                gst = stream.cuda_stream
                if gbox is None:
                    gargs = (xpos.data_ptr(), Ng, ctypes.c_float(xw.cutoff), gout["off"].data_ptr(),
                             gout["src"].data_ptr(), gout["vec"].data_ptr(), None, None, Eg, gE.data_ptr(),
                             gws.data_ptr(), gws.numel(), gst)
                    fn = lambda: lib.eqmp_radius_graph(*gargs)
                else:
                    glen = (ctypes.c_float * 3)(*gbox)
                    gargs = (xpos.data_ptr(), Ng, ctypes.c_float(xw.cutoff), glen, gout["off"].data_ptr(),
                             gout["src"].data_ptr(), gout["vec"].data_ptr(), gout["img"].data_ptr(), None, None,
                             Eg, gE.data_ptr(), gws.data_ptr(), gws.numel(), gst)
                    fn = lambda: lib.eqmp_radius_graph_pbc(*gargs)
                entry["launches"] = 1 if Ng <= 16384 else 12
                entry["n_edges"] = Eg
                entry["gbytes"] = 12 * Ng + 4 * (Ng + 1) + (20 if gbox is not None else 16) * Eg
            else:  # lmax6
                xd = device_inputs(torch, xw, dev)
                xo = torch.empty((xw.n_atoms, xw.channels, 49), dtype=torch.float32, device=dev)
                lkw = dict(w=xd["w"]) if xw.w is not None else dict(R=xd["R"], M=xd["M"])
                fn = lambda: eq.eqmp_fused_lmax(6, xd["vec"], xd["x"], xd["off"], xd["src"], out=xo, **lkw)
                entry["launches"] = 1
            entry["ms"], entry["kernel_ms"], entry["t"] = timed(fn)
            extra.append(entry)
            fn = None
            torch.cuda.empty_cache()

    # ---- FP32 throughput probe (paired FMAs only), outside every timed
    # region but inside the clock sampler's window: the measured
    # counterpart of the derived FP32 peak, with the SM clock it ran at.
    probe_buf = torch.zeros(1, device=dev)
    probe_ms = []
    pt0 = time.time()
    while time.time() - pt0 < 0.8 or len(probe_ms) < 8:
        ps, pe = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ps.record(stream)
        probe_flops = eq.eqmp_fp32_peak_probe(65536, probe_buf, stream=stream)
        pe.record(stream)
        torch.cuda.synchronize()
        probe_ms.append(ps.elapsed_time(pe))
    pt1 = time.time()
    probe_ms = probe_ms[2:]
    fp32_measured = probe_flops / (float(np.median(probe_ms)) * 1e-3) / 1e12
    wd = eq.eqmp_device_error()
    time.sleep(0.25)
    sampler.stop()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    props = torch.cuda.get_device_properties(dev)
    clocks = sampler.summary(t0, t1)
    probe_clocks = sampler.summary(pt0, pt1, pad=0.05)
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks = json.load(open(peaks_path)) if os.path.exists(peaks_path) else {}
    max_mhz = clocks.get("sm_max_mhz") or peaks.get("sm_max_mhz") or 2070.0
    derived_tflops = props.multi_processor_count * 128 * 2 * max_mhz * 1e6 / 1e12
    # graded against the higher of the derived and the measured FP32 peak
    fp32_peak = max(derived_tflops, fp32_measured)
    hbm_peak = float(peaks.get("hbm_gbs", 6793.1))
    peak_basis = (f"{props.multi_processor_count} SMs x 128 FP32 lanes x 2 x {max_mhz:.0f} MHz (derived)"
                  if derived_tflops >= fp32_measured else "eqmp_fp32_peak_probe (measured, paired FMAs)")
    fp32_info = {"peak_basis": peak_basis, "fp32_derived": derived_tflops, "fp32_measured": fp32_measured,
                 "fp32_probe_sm_mhz": probe_clocks.get("sm_mhz"),
                 "hbm_peak_basis": "MEASURED_PEAKS.json hbm_gbs (measured copy)"}
    if probe_clocks.get("sm_mhz"):
        # the probe's throughput scaled to the maximum SM clock
        fp32_info["fp32_measured_at_max_clock"] = fp32_measured * max_mhz / probe_clocks["sm_mhz"]

    def layer_roof(w_, ms_, version, which, l_max, entry):
        flops, basis, xtra = layer_flops(w_, which, l_max)
        traffic = NCU_TRAFFIC.get((w_.name, version)) if entry == "fused" else None
        r = roofline(flops, compulsory_bytes(w_), ms_, fp32_peak, hbm_peak, version, traffic, basis, xtra)
        r.update(fp32_info)
        return r

    version = kernel_version(wl, args.which, args.lmax, args.entry)
    if args.which == "graph":
        # positions in; offsets, senders and edge vectors (and image indices) out
        gbytes = 12 * wl.n_atoms + 4 * (wl.n_atoms + 1) + (20 if box is not None else 16) * E_graph
        label = ("radius-graph cooperative single launch" if coop else
                 "radius-graph multi-kernel (12 launches)") + (", periodic" if box is not None else "")
        roof = roofline(0.0, gbytes, ms, fp32_peak, hbm_peak, label, None,
                        "compulsory bytes: positions, offsets, senders, edge vectors")
        roof["algorithmic_bytes"] = gbytes
    else:
        roof = layer_roof(wl, ms, version, args.which, args.lmax, args.entry)

    workloads = []
    for x in extra:
        xw, kind = x["wl"], x["kind"]
        if kind in ("graph", "graph_pbc"):
            xroof = roofline(0.0, x["gbytes"], x["ms"], fp32_peak, hbm_peak,
                            ("radius-graph cooperative single launch" if x["launches"] == 1 else
                             "radius-graph multi-kernel (12 launches)") + (", periodic" if kind == "graph_pbc" else ""),
                            None, "compulsory bytes: positions, offsets, senders, edge vectors"
                            + (", image indices" if kind == "graph_pbc" else ""))
        elif kind == "backward":
            xroof = layer_roof(xw, x["ms"], kernel_version(xw, "backward", 3, "fused"), "backward", 3, "fused")
        elif kind == "lmax6":
            xroof = layer_roof(xw, x["ms"], kernel_version(xw, "forward", 6, "fused"), "forward", 6, "fused")
        else:
            xroof = layer_roof(xw, x["ms"], kernel_version(xw, "forward", 3, "fused"), "forward", 3, "fused")
        workloads.append({
            "label": x["label"], "workload": x["name"], "pass": kind, "n_atoms": xw.n_atoms,
            "n_edges": x["n_edges"], "channels": xw.channels,
            "storage": xw.storage, "weights": "shared" if xw.w is not None else "radial",
            "ms_per_step": x["ms"], "value": x["n_edges"] * world / (x["ms"] * 1e-3), "unit": "edges/s",
            "steps": args.steps, "gpu_launches": args.steps * x["launches"],
            "kernel_ms": {"min": float(np.min(x["kernel_ms"])), "median": float(np.median(x["kernel_ms"])),
                          "max": float(np.max(x["kernel_ms"]))},
            "roofline": xroof,
            "clocks": sampler.summary(*x["t"]),
        })

    cpu = None
    if pool is not None and args.which == "graph":
        from oracle import graph as oracle_graph

        pool.terminate()
        tg = time.perf_counter()
        if box is None:
            E_cpu = len(oracle_graph.radius_graph(wl.pos, wl.cutoff)["src"])
        else:
            E_cpu = len(oracle_graph.radius_graph_pbc(pos_np, wl.cutoff, box)["src"])
        wall = time.perf_counter() - tg
        cpu = {"value": E_cpu / wall, "unit": "edges/s", "cores": 1, "kind": "oracle",
               "sample": f"whole workload ({wl.n_atoms} atoms, {E_cpu} edges), k-d tree candidates + float32 test, {wall:.2f} s"}
    elif pool is not None:
        rate, sample = cpu_oracle_rate(args.workload, wl, pool=pool, cores=cores)
        cpu = {"value": rate, "unit": "edges/s", "cores": cores, "kind": "oracle", "sample": sample}
        if args.which == "forward" and args.lmax == 3:
            cpu["single_thread"] = single_thread_rates(pool, SINGLE_THREAD_WORKLOADS)
        pool.terminate()

    value = n_edges * world / (ms * 1e-3)
    line = {
        "metric": METRIC if args.which != "graph" else METRIC_GRAPH, "value": value, "unit": "edges/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if wl.storage == "f32" else "bf16-storage/f32-compute", "data": "synthetic",
        "config": dict(workload_config(args.workload, wl, args.entry, world),
                       **({"boundaries": "periodic"} if args.which == "graph" and args.pbc else {})),
        "roofline": roof,
        "e2e": None if e2e_ms is None else {
            "value": n_edges * world / (e2e_ms * 1e-3), "unit": "edges/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "api": e2e_api,
            "mode": e2e_mode, "serial_ms_per_step": e2e_serial_ms,
            "copy_floor_ms_per_step": e2e_copy_floor},
        "pass": args.which,
        "l_max": args.lmax,
        "graph_edges": None if args.which != "graph" else E_graph,
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks,
        "kernel_ms": {"min": float(np.min(kernel_ms)), "median": float(np.median(kernel_ms)),
                      "max": float(np.max(kernel_ms))},
        "workloads": workloads,
        "fp32_probe": {"tflops": fp32_measured, "clocks": probe_clocks, "launches": len(probe_ms) + 2},
        "watchdog": wd,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
