#!/usr/bin/env python3
"""Benchmark of the fused SH + CG tensor product + receiver sum layer.

One step = one eqmp_fused call (the whole hot path: CSR walk, SH in
registers, sender-row gather, CG tensor product, receiver sum, store) over
one seeded synthetic graph.  Default workload: 1000 atoms, 32 channels,
~16.5 neighbours per atom, shared per-path weights, fp32 - the workload
the Batmobile blog quotes (1000 atoms, 32 channels, about 20 neighbours).

Prints ONE JSON line (rank 0):
  value        edges/s over all ranks, inputs resident in HBM, L2 flushed
               (256 MB write) before every timed step, device time of the
               layer kernel from CUDA events on the launching stream;
  e2e          the same metric through the public API with pinned host
               buffers: H2D of the step's inputs, the layer, D2H of out;
  roofline     FP32-ALU bound of the layer kernel (FMA count of the
               lowest-FMA exact schedule against the higher of the derived
               peak, SM count x 128 lanes x 2 flops x max SM clock, and the
               measured one from eqmp_fp32_peak_probe; both are reported);
  cpu_baseline the CPU oracle (numpy, fp64) on a bounded sample of the same
               workload on this host's cores.
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
# DRAM bytes per launch of the layer kernel from the ncu capture recorded in
# profiles/ (None until captured for the current kernel version).
# Keyed by (workload, kernel version); a changed kernel gets a new version
# tag, which makes its entry missing (traffic null) until re-captured.
KERNEL_VERSION = {"shared": "k_shared-pairs-v5", "radial": "k_so2-v4"}
NCU_TRAFFIC = {
    ("pages_1k_c32", "k_shared-pairs-v5"): 2357504 + 0,
    ("scale_100k_c64", "k_shared-pairs-v5"): 6207318016 + 407371008,
    ("dense_10k_c128_bf16", "k_shared-pairs-v5"): 48796160 + 11876864,
    ("radial_1k_c32", "k_so2-v4"): 2888704 + 0,
}


def fma_count(wl):
    """FMAs of the lowest-FMA exact schedule of the layer (per launch).

    shared weights: 256*C per edge (A += x (x) Y) + (611 + 156)*C per receiver
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


def aligned_fma_count(wl, l_max, n_terms):
    """FMAs of the aligned-frame schedule at degree l_max (per launch):
    rotate in and out (2 sum (2l+1)^2), one FMA per aligned term, and for
    radial weights 8 per path; per edge and channel."""
    from equivariant_gnn_message_gb300.inputs import n_paths

    per = 2 * sum_rot(l_max) + n_terms + (8 * n_paths(l_max) if wl.w is None else 0)
    return per * wl.channels * wl.n_edges


# aligned-frame terms per degree (one per output order and path with m2 = 0)
ALIGNED_TERMS = {4: 272, 5: 565, 6: 1036}


def compulsory_bytes(wl):
    s = 2 if wl.storage == "bf16" else 4
    C, E, N = wl.channels, wl.n_edges, wl.n_atoms
    nc = wl.x.shape[2]
    b = N * C * nc * s + 12 * E + 4 * E + 4 * (N + 1) + N * C * nc * s
    b += 4 * 34 * C if wl.w is not None else 32 * E + 4 * 8 * 34 * C
    return b


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

    def summary(self, t0, t1):
        win = [s for (t, s) in self.samples if t0 - 0.3 <= t <= t1 + 0.3] or [s for _, s in self.samples]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(s[1]) for s in win if num(s[1]) is not None]
        mx = [num(s[2]) for s in win if num(s[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4) if len(s) > 5 + i and s[5 + i] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(win)}


def _oracle_chunk(args):
    """Child-process worker: oracle on a receiver subset, `reps` times
    (single-threaded BLAS)."""
    name, receivers, l_max, reps = args
    from equivariant_gnn_message_gb300.inputs import make_workload
    from oracle import layer

    wl = make_workload(name, l_max=l_max)
    kw = dict(w=wl.w) if wl.w is not None else dict(R=wl.R, M=wl.M)
    t = time.perf_counter()
    for _ in range(reps):
        layer.message_pass(wl.vec, wl.x, wl.off, wl.src, receivers=np.asarray(receivers), **kw)
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
        "config": {"workload": args.workload, "n_atoms": wl.n_atoms, "n_edges": wl.n_edges,
                   "channels": wl.channels, "storage": wl.storage,
                   "weights": "shared" if wl.w is not None else "radial"},
        "cpu_baseline": {"value": value, "unit": "edges/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "edges/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "timed_wall_s": round(total, 2),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="pages_1k_c32")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--entry", default="fused", choices=["fused", "tp_scatter", "so2"])
    ap.add_argument("--lmax", type=int, default=3,
                    help="4..6: the higher-degree layer (eqmp_fused_lmax) on the workload's graph")
    ap.add_argument("--pass", dest="which", default="forward", choices=["forward", "backward", "graph"],
                    help="backward: time eqmp_fused_backward (dx, dw or dR/dM, dvec) instead; "
                         "graph: time eqmp_radius_graph on the workload's atom positions")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    from equivariant_gnn_message_gb300.inputs import make_workload
    from equivariant_gnn_message_gb300.sharding import max_over_ranks

    wl = make_workload(args.workload, l_max=args.lmax)
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

    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    vec, off, src, w, R, M = t(wl.vec), t(wl.off), t(wl.src), t(wl.w), t(wl.R), t(wl.M)
    if wl.storage == "bf16":
        x = torch.from_numpy(wl.x_bf16_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        x = t(wl.x)
    out = torch.empty((wl.n_atoms, wl.channels, 16), dtype=x.dtype, device=dev)
    Yb = torch.empty((wl.n_edges, 16), dtype=torch.float32, device=dev)
    wkw = dict(w=w) if w is not None else dict(R=R, M=M)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    bwd_args = None
    if args.which == "backward":
        if wl.storage != "f32":
            raise SystemExit("the backward pass takes fp32 features")
        so, se = eq.sender_view(wl.src, wl.n_atoms)
        gout = torch.randn((wl.n_atoms, wl.channels, 16), device=dev, generator=torch.Generator(device=dev).manual_seed(0))
        need = ("x", "vec", "w") if w is not None else ("x", "vec", "R", "M")
        bwd_args = ((vec, x, off, src, t(wl.dst), t(so), t(se), gout), dict(need=need, **wkw))

    graph_args = None
    if args.which == "graph":
        import ctypes

        lib = eq.load_library()
        N = wl.n_atoms
        g_pos = t(wl.pos)
        g_ws = torch.empty(lib.eqmp_radius_graph_workspace_size(N), dtype=torch.uint8, device=dev)
        g_E = torch.empty(1, dtype=torch.int64, device=dev)
        g_out, E_graph = eq.eqmp_radius_graph(g_pos, wl.cutoff)
        g_cap = E_graph
        g_off, g_src, g_vec = g_out["off"], g_out["src"], g_out["vec"]
        graph_args = (g_pos.data_ptr(), N, ctypes.c_float(wl.cutoff), g_off.data_ptr(), g_src.data_ptr(),
                      g_vec.data_ptr(), None, None, g_cap, g_E.data_ptr(), g_ws.data_ptr(), g_ws.numel(),
                      stream.cuda_stream)

    if args.lmax != 3:
        out = torch.empty((wl.n_atoms, wl.channels, (args.lmax + 1) ** 2), dtype=torch.float32, device=dev)

    def step():
        if args.lmax != 3:
            eq.eqmp_fused_lmax(args.lmax, vec, x, off, src, out=out, **wkw)
        elif graph_args is not None:
            lib.eqmp_radius_graph(*graph_args)
        elif bwd_args is not None:
            eq.eqmp_fused_backward(*bwd_args[0], **bwd_args[1])
        elif args.entry == "fused":
            eq.eqmp_fused(vec, x, off, src, out=out, **wkw)
        elif args.entry == "so2":
            eq.eqmp_fused_so2(vec, x, off, src, out=out, **wkw)
        else:
            eq.eqmp_sh(vec, Yb)
            eq.eqmp_tp_scatter(Yb, x, off, src, out=out, **wkw)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    barrier()
    if eq.eqmp_device_error() != 0:
        raise RuntimeError("device watchdog tripped during warm-up")

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()                 # evict L2 between timed steps
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    barrier()
    t1 = time.time()
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(float(np.mean(kernel_ms)))

    # ---- e2e through the public API with pinned host buffers.  The step's
    # inputs sit in one pinned host block (each array 256-byte aligned) and
    # go over in one host->device copy; the result comes back in one copy.
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
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
    tdt = {np.dtype(np.float32): torch.float32, np.dtype(np.int32): torch.int32, np.dtype(np.int16): torch.int16}

    def dview(k):
        o, dt, shp = layout[k]
        n = int(np.prod(shp)) * dt.itemsize
        return d_pack[o:o + n].view(tdt[dt]).view(shp)

    d_in = {k: dview(k) for k in parts}
    h_in = {"packed": h_pack}
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(np.ascontiguousarray(a).nbytes for a in parts.values())
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        d_pack.copy_(h_pack, non_blocking=True)
        xd = d_in["x"].view(torch.bfloat16) if wl.storage == "bf16" else d_in["x"]
        kw = dict(w=d_in["w"]) if "w" in d_in else dict(R=d_in["R"], M=d_in["M"])
        if args.lmax != 3:
            eq.eqmp_fused_lmax(args.lmax, d_in["vec"], xd, d_in["off"], d_in["src"], out=out, **kw)
        elif args.entry == "so2":
            eq.eqmp_fused_so2(d_in["vec"], xd, d_in["off"], d_in["src"], out=out, **kw)
        elif args.entry == "tp_scatter":
            eq.eqmp_sh(d_in["vec"], Yb)
            eq.eqmp_tp_scatter(Yb, xd, d_in["off"], d_in["src"], out=out, **kw)
        else:
            eq.eqmp_fused(d_in["vec"], xd, d_in["off"], d_in["src"], out=out, **kw)
        h_out.copy_(out, non_blocking=True)

    if graph_args is not None:
        h_in = {"pos": pin(wl.pos)}
        d_in = {"pos": g_pos}
        h_out = [torch.empty(a.shape, dtype=a.dtype).pin_memory() for a in (g_off, g_src, g_vec)]
        h2d = h_in["pos"].numel() * 4
        d2h = sum(a.numel() * a.element_size() for a in h_out)

        def e2e_step():
            d_in["pos"].copy_(h_in["pos"], non_blocking=True)
            lib.eqmp_radius_graph(*graph_args)
            for h, d in zip(h_out, (g_off, g_src, g_vec)):
                h.copy_(d, non_blocking=True)

    e2e_ms = None
    if bwd_args is None:  # the end-to-end figure is the forward layer's
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
    sampler.stop()
    # FP32 throughput probe (paired FMAs only), outside the timed region:
    # the measured counterpart of the derived FP32 peak.
    probe_buf = torch.zeros(1, device=dev)
    probe_ms = []
    for i in range(7):
        ps, pe = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ps.record(stream)
        probe_flops = eq.eqmp_fp32_peak_probe(65536, probe_buf, stream=stream)
        pe.record(stream)
        torch.cuda.synchronize()
        if i >= 2:
            probe_ms.append(ps.elapsed_time(pe))
    fp32_measured = probe_flops / (float(np.median(probe_ms)) * 1e-3) / 1e12
    wd = eq.eqmp_device_error()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    props = torch.cuda.get_device_properties(dev)
    clocks = sampler.summary(t0, t1)
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks = json.load(open(peaks_path)) if os.path.exists(peaks_path) else {}
    max_mhz = clocks.get("sm_max_mhz") or peaks.get("sm_max_mhz") or 2070.0
    derived_tflops = props.multi_processor_count * 128 * 2 * max_mhz * 1e6 / 1e12
    # graded against the higher of the derived and the measured FP32 peak
    peak_tflops = max(derived_tflops, fp32_measured)
    peak_basis = (f"{props.multi_processor_count} SMs x 128 FP32 lanes x 2 x {max_mhz:.0f} MHz (derived)"
                  if derived_tflops >= fp32_measured else "eqmp_fp32_peak_probe (measured, paired FMAs)")
    # backward: three forward-sized contractions (dx, the weight gradient,
    # dY) of the lowest-FMA schedule plus the SH Jacobian (48 FMA per edge)
    flops = 2.0 * fma_count(wl) if bwd_args is None else 2.0 * (3 * fma_count(wl) + 48 * wl.n_edges)
    if args.lmax != 3:
        flops = 2.0 * aligned_fma_count(wl, args.lmax, ALIGNED_TERMS[args.lmax])
    achieved = flops / (ms * 1e-3) / 1e12
    version = KERNEL_VERSION["shared" if wl.w is not None else "radial"] if bwd_args is None else "k_bwd-v1"
    if args.lmax != 3:
        version = f"k_hl<{args.lmax}>-v1"
    traffic = NCU_TRAFFIC.get((args.workload, version)) if args.entry == "fused" else None
    n_edges = wl.n_edges if graph_args is None else E_graph
    value = n_edges * world / (ms * 1e-3)
    roofline = {"bound": "alu", "achieved": achieved, "peak": peak_tflops, "unit": "TFLOP/s",
                "frac": achieved / peak_tflops, "traffic": traffic, "traffic_unit": "bytes/launch",
                "kernel": version,
                "peak_basis": peak_basis, "fp32_derived": derived_tflops, "fp32_measured": fp32_measured,
                "hbm_gbs_compulsory": compulsory_bytes(wl) / (ms * 1e-3) / 1e9}
    if graph_args is not None:
        # positions in; offsets, senders and edge vectors out
        gbytes = 12 * wl.n_atoms + 4 * (wl.n_atoms + 1) + 16 * E_graph
        hbm = float(peaks.get("hbm_gbs", 6787.2))
        gach = gbytes / (ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": gach, "peak": hbm, "unit": "GB/s", "frac": gach / hbm,
                    "traffic": None, "kernel": "radius-graph-v1 (12 launches)",
                    "algorithmic_bytes": gbytes, "peak_basis": "MEASURED_PEAKS.json hbm_gbs (measured copy)"}

    cpu = None
    if pool is not None and graph_args is not None:
        from oracle import graph as oracle_graph

        pool.terminate()
        tg = time.perf_counter()
        E_cpu = len(oracle_graph.radius_graph(wl.pos, wl.cutoff)["src"])
        wall = time.perf_counter() - tg
        cpu = {"value": E_cpu / wall, "unit": "edges/s", "cores": 1, "kind": "oracle",
               "sample": f"whole workload ({wl.n_atoms} atoms, {E_cpu} edges), k-d tree candidates + float32 test, {wall:.2f} s"}
    elif pool is not None:
        rate, sample = cpu_oracle_rate(args.workload, wl, pool=pool, cores=cores)
        pool.terminate()
        cpu = {"value": rate, "unit": "edges/s", "cores": cores, "kind": "oracle", "sample": sample}

    line = {
        "metric": METRIC if graph_args is None else METRIC_GRAPH, "value": value, "unit": "edges/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if wl.storage == "f32" else "bf16-storage/f32-compute", "data": "synthetic",
        "config": {"workload": args.workload, "n_atoms": wl.n_atoms, "n_edges": wl.n_edges,
                   "channels": wl.channels, "storage": wl.storage,
                   "weights": "shared" if wl.w is not None else "radial", "entry": args.entry,
                   "l2": "flushed (256 MB write) before every timed step",
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline,
        "e2e": None if e2e_ms is None else {
            "value": n_edges * world / (e2e_ms * 1e-3), "unit": "edges/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "pass": args.which,
        "l_max": args.lmax,
        "graph_edges": None if graph_args is None else E_graph,
        "gpu_launches": args.steps * (1 if args.lmax != 3 else 12 if graph_args is not None else
                                      (2 if args.entry == "tp_scatter" else 1) if bwd_args is None else 3),
        "clocks": clocks,
        "kernel_ms": {"min": float(np.min(kernel_ms)), "median": float(np.median(kernel_ms))},
        "watchdog": wd,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
