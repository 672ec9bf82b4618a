#!/usr/bin/env python3
"""Throughput of the activation-sparse gated FFN (TwELL) on one GB300.

One step = the whole hot path on one batch of synthetic tokens: gate GEMM
with the fused TwELL pack, hybrid ELL / dense routing, fused sparse up+down
forward (routed rows on the dense tensor-core backup), and the backward
(dX, dWg, dWu, dWd with the L1 term).  `value` is tokens/s of that
forward+backward step over all ranks; the same JSON line also carries the
forward-only rate, the library's own dense tcgen05 FFN at equal shapes, the
dominant kernel's roofline, an end-to-end figure through the C ABI with host
buffers, and the CPU oracle's rate on a bounded sample.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl own|reference]
Multi-GPU runs (torchrun) are independent replicas: the hot path has no
data-path exchange, so each rank runs the full workload and only the timing
is reduced (max over ranks).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from activation_sparse_gated_tcgen05_gb300 import synthetic  # noqa: E402

METRIC = "gated-FFN tokens/s (fwd, fwd+bwd) at 0.5% density vs own dense; % of roofline"
UNIT = "tokens/s"
L1 = 2e-5
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("own", "reference"), default="own")
    ap.add_argument("--workload", default="fwd_0p5b", choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--density", type=float, default=None,
                    help="override the workload's target gate density (density sweep)")
    ap.add_argument("--route-fraction", type=float, default=None,
                    help="fraction of rows the ELL width sends to the dense backup "
                         "(default: the workload's; 0 routes only rows with an overflowing tile)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-small-m", action="store_true",
                    help="skip the M = 1, 16, 64 forward timings at the workload's shape")
    ap.add_argument("--no-torch-dense", action="store_true",
                    help="skip the PyTorch (cuBLAS) dense FFN reference timing")
    ap.add_argument("--only", choices=("sparse_step", "sparse_fwd", "dense_fwd", "dense_step",
                                       "small_fwd"),
                    help="time just this part (a short command for kernel profiling); prints "
                         "a reduced JSON line")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def workload_config(wl, W, route_fraction):
    dens = ("lognormal median %.2g%% sigma %.2g" % (100 * wl.density, wl.lognormal_sigma)
            if wl.lognormal_sigma else "%.2g%% uniform" % (100 * wl.density))
    return {
        "workload": "%s: M=%d d_model=%d d_ff=%d T_n=%d C=%d density %s, ELL width W=%d "
                    "(%s)" % (wl.name, wl.M, wl.d_model, wl.d_ff, wl.tile_n, wl.tile_cap, dens, W,
                              "p%.0f of row_nnz" % (100 * (1 - route_fraction))
                              if route_fraction > 0 else "widest row; overflow rows routed"),
        "M": wl.M, "d_model": wl.d_model, "d_ff": wl.d_ff, "tile_n": wl.tile_n,
        "tile_cap": wl.tile_cap, "ell_width": W, "l1_coeff": L1,
        "l2": "flushed between timed steps (256 MiB write)",
        "parallelism": "replicas",
    }


# ---------------------------------------------------------------- distributed
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist

            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float, device) -> float:
        if not self.pg:
            return v
        import torch

        t = torch.tensor([v], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.idx = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.idx)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle
def oracle_step(oracle, w64, bits, rows, wl, W):
    """The oracle's training step on the given rows: gate, pack, route,
    sparse forward (dense formula for routed rows), hybrid backward."""
    x = w64["x"][rows]
    a = oracle.gate_preact(x, w64["wgT"])
    val, idx, cnt, nnz = oracle.twell_pack(a, wl.tile_n, wl.tile_cap)
    ev, ec, en, dr = oracle.hybrid_route(val, idx, cnt, nnz, wl.d_ff, wl.tile_n, W)
    y = oracle.ffn_fwd_ell(x, w64["wuT"], w64["wd"], ev, ec, en)
    if dr.size:
        y[dr] = oracle.ffn_fwd_dense(x, w64["wgT"], w64["wuT"], w64["wd"], rows=dr)
    g = oracle.ffn_bwd_hybrid(x, w64["wgT"], w64["wuT"], w64["wd"], w64["dy"][rows], ev, ec, en,
                              dr, L1)
    return y, g


def cpu_sample_rate(wl, bits, W, seconds, step_budget=None):
    """Time the oracle on a bounded sample of the workload's rows.  Returns
    (tokens/s, rows per sample, threads, seconds per sample)."""
    import oracle

    threads = os.cpu_count() or 1
    oracle.set_threads(threads)
    w64 = {k: oracle.f64(bits[k]) for k in ("x", "wgT", "wuT", "wd", "dy")}
    rows = np.arange(8)
    t0 = time.perf_counter()
    oracle_step(oracle, w64, bits, rows, wl, W)
    dt = time.perf_counter() - t0
    target = step_budget if step_budget is not None else seconds
    n = int(max(8, min(wl.M, 8 * target / max(dt, 1e-3))))
    for _ in range(2):  # the 8-row pilot overstates the per-row cost: rescale once
        rows = np.arange(n)
        t0 = time.perf_counter()
        oracle_step(oracle, w64, bits, rows, wl, W)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * target or n >= wl.M:
            break
        n = int(min(wl.M, n * target / max(dt, 1e-3)))
    return n / dt, n, threads, dt, w64


# ---------------------------------------------------------------- own arm
def algorithmic_work(family, wl, nnz_ell, n_dense):
    """(amount, unit, bound) per step of a kernel family, from the formulas
    of the hot path: flops for tensor-core GEMMs, bytes for gather kernels.
    The bytes are those of one pass over the step's inputs; the partial sums
    that L2-sized neuron passes carry between launches are not counted."""
    M, d, f = wl.M, wl.d_model, wl.d_ff
    if family == "gemm_gate_pack":
        return 2.0 * M * d * f, "flop", "tensor"
    if family == "sparse_fwd":  # weight rows gathered + x read + y written + ELL entries
        return 4.0 * d * nnz_ell + 4.0 * d * M + 4.0 * nnz_ell, "byte", "hbm"
    if family == "sparse_fwd_up":  # Wu^T rows + x read + ELL entries + per-entry h written
        return 2.0 * d * nnz_ell + 2.0 * d * M + 8.0 * nnz_ell, "byte", "hbm"
    if family == "sparse_fwd_down":  # Wd rows + y written + ELL columns + per-entry h read
        return 2.0 * d * nnz_ell + 2.0 * d * M + 6.0 * nnz_ell, "byte", "hbm"
    if family == "bwd_rows":  # 3 weight rows per entry + x, dy, dx rows + per-entry scratch
        return 6.0 * d * nnz_ell + 6.0 * d * M + 24.0 * nnz_ell, "byte", "hbm"
    if family == "bwd_dh":  # Wd rows + dy read + ELL columns + per-entry dh written
        return 2.0 * d * nnz_ell + 2.0 * d * M + 6.0 * nnz_ell, "byte", "hbm"
    if family == "bwd_grad_dx":  # Wu^T and Wg^T rows + x read, dX written + per entry:
        # column, value, dh and slot in, (du, da, h) out
        return 4.0 * d * nnz_ell + 4.0 * d * M + 28.0 * nnz_ell, "byte", "hbm"
    if family == "bwd_neurons":  # x and dy rows per entry + three fp32 dW rows per neuron
        return 4.0 * d * nnz_ell + 12.0 * f * d + 20.0 * nnz_ell, "byte", "hbm"
    if family == "bwd_neurons_dy":  # dy rows per entry + the fp32 dWd row per neuron
        return 2.0 * d * nnz_ell + 4.0 * f * d + 20.0 * nnz_ell, "byte", "hbm"
    if family == "bwd_neurons_x":  # x rows per entry + the fp32 dWu^T, dWg^T rows per neuron
        return 2.0 * d * nnz_ell + 8.0 * f * d + 20.0 * nnz_ell, "byte", "hbm"
    return None


def run_own(args, dist):
    import torch

    from activation_sparse_gated_tcgen05_gb300 import probe, twell

    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    wl = synthetic.WORKLOADS[args.workload]
    if args.density is not None:
        wl = dataclasses.replace(wl, density=args.density)
    bits = synthetic.make_workload(wl)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    x, wg, wu, wd, dy = (up(bits[k]) for k in ("x", "wgT", "wuT", "wd", "dy"))
    M, d, f = wl.M, wl.d_model, wl.d_ff
    shape = twell.make_shape(M, d, f, wl.tile_n, wl.tile_cap)
    tiles = twell.alloc_tiles(shape, dev)
    twell.twell_pack(x, wg, shape, tiles)
    nnz = twell.tiles_view(tiles, shape)[3].cpu().numpy()
    rf = wl.route_fraction if args.route_fraction is None else args.route_fraction
    W = synthetic.ell_width(nnz, rf)
    # route once with room for every row, read the routed-row count from the
    # device and size the workspace's dense-backup buffers for exactly those
    # rows (every timed step routes the same inputs the same way; a step that
    # routed more would record TWELL_ERR_CAPACITY, which voids the run)
    route = twell.alloc_hybrid(shape, W, dev)
    twell.hybrid_route(tiles, shape, route)
    route.dense_cap = int(route.n_dense[0].item())
    ws = torch.empty(twell.twell_workspace_bytes(shape, W, True, dense_cap=route.dense_cap),
                     dtype=torch.uint8, device=dev)
    y = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
    dx = torch.empty_like(y)
    dws = [torch.empty(f, d, dtype=torch.float32, device=dev) for _ in range(3)]
    # the dense comparator's buffers (not allocated for a sparse-only profiling run)
    need_dense = args.only is None or args.only.startswith("dense")
    dws_d = [torch.empty(f if need_dense else 1, d, dtype=torch.float32, device=dev)
             for _ in range(3)]
    ws_d = torch.empty(twell.twell_dense_workspace_bytes(shape, True) if need_dense else 16,
                       dtype=torch.uint8, device=dev)
    y_d, dx_d = torch.empty_like(y), torch.empty_like(y)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def make_sparse_step(xb, dyb, yb, dxb):
        def step():
            twell.twell_pack(xb, wg, shape, tiles)
            twell.hybrid_route(tiles, shape, route)
            twell.twell_ffn_fwd(xb, wg, wu, wd, shape, yb, route=route, ws=ws)
            twell.twell_ffn_bwd(xb, wg, wu, wd, dyb, shape, route, L1, dxb, *dws, ws)
        return step

    sparse_step = make_sparse_step(x, dy, y, dx)

    # inference workloads (uniform density, no routing) run the TwELL forward;
    # training workloads run the forward of their training step: pack, hybrid
    # route, ELL gather plus the dense fallback for the routed rows
    fwd_path = "hybrid" if rf > 0 else "twell"

    # the TwELL forward's optional workspace (d_model > 1024: the split gathers)
    tiles_ws_bytes = twell.twell_tiles_workspace_bytes(shape)
    ws_t = (torch.empty(tiles_ws_bytes, dtype=torch.uint8, device=dev) if tiles_ws_bytes
            else None)

    def sparse_fwd():
        twell.twell_pack(x, wg, shape, tiles)
        if fwd_path == "hybrid":
            twell.hybrid_route(tiles, shape, route)
            twell.twell_ffn_fwd(x, wg, wu, wd, shape, y, route=route, ws=ws)
        else:
            twell.twell_ffn_fwd(x, wg, wu, wd, shape, y, tiles=tiles, ws=ws_t)

    def dense_fwd():
        twell.twell_dense_ffn_fwd(x, wg, wu, wd, shape, y_d, False, ws_d)

    def dense_step():
        twell.twell_dense_ffn_fwd(x, wg, wu, wd, shape, y_d, True, ws_d)
        twell.twell_dense_ffn_bwd(x, wg, wu, wd, dy, shape, L1, dx_d, *dws_d, ws_d)

    # the unmodified SiLU-gated FFN that the ReLU recipe replaces (no L1 term)
    def dense_silu_fwd():
        twell.twell_dense_ffn_fwd_act(x, wg, wu, wd, shape, twell.ACT_SILU, y_d, False, ws_d)

    def dense_silu_step():
        twell.twell_dense_ffn_fwd_act(x, wg, wu, wd, shape, twell.ACT_SILU, y_d, True, ws_d)
        twell.twell_dense_ffn_bwd_act(x, wg, wu, wd, dy, shape, twell.ACT_SILU, 0.0, dx_d, *dws_d,
                                      ws_d)

    def graphed(fn):
        """Capture fn (a whole step of library calls) into a CUDA graph; the
        library is capture-safe (device-side routed-row counts, no host sync)."""
        fn()  # eager once: function attributes and lazy module loads happen here
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g.replay

    medians = {}

    def timed(fn, steps, warmup, profile=None, clocks=None, l2_flush=True, key=None):
        for _ in range(warmup):
            if l2_flush:
                flush.zero_()
            fn()
        torch.cuda.synchronize()
        dist.barrier()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        if clocks:
            clocks.start()
        if profile:
            twell.twell_profile_begin(profile)
        launches0 = twell.twell_launch_count()
        for s0, s1 in ev:
            if l2_flush:
                flush.zero_()
            s0.record(stream)
            fn()
            s1.record(stream)
        launches = twell.twell_launch_count() - launches0
        torch.cuda.synchronize()
        prof = twell.twell_profile_end() if profile else None
        dist.barrier()
        torch.cuda.synchronize()
        ck = clocks.stop() if clocks else None
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        if key:
            medians[key] = dist.max(statistics.median(a.elapsed_time(b) for a, b in ev), dev)
        st = twell.twell_get_device_status()
        if st != 0:  # a capacity overflow or timeout voids the number
            raise RuntimeError("device status %d after timing" % st)
        return dist.max(ms, dev), launches, prof, ck

    def small_fwd():  # the first 64 tokens through the small-batch gate and TwELL forward
        twell.twell_pack(x_small, wg, shape_small, tiles_small)
        twell.twell_ffn_fwd(x_small, wg, wu, wd, shape_small, y_small, tiles=tiles_small)

    if args.only == "small_fwd":
        ms_ = min(64, M)
        x_small = x[:ms_].contiguous()
        shape_small = twell.make_shape(ms_, d, f, wl.tile_n, wl.tile_cap)
        tiles_small = twell.alloc_tiles(shape_small, dev)
        y_small = torch.empty(ms_, d, dtype=torch.bfloat16, device=dev)

    if args.only:
        fn = {"sparse_step": sparse_step, "sparse_fwd": sparse_fwd, "dense_fwd": dense_fwd,
              "dense_step": dense_step, "small_fwd": small_fwd}[args.only]
        ms, launches, _, _ = timed(fn, args.steps, args.warmup)
        st = twell.twell_get_device_status()
        if dist.rank == 0:
            print(json.dumps({"only": args.only, "workload": wl.name, "ms": ms,
                              "tokens_per_s": dist.world * M / (ms / 1e3),
                              "gpu_launches": launches, "device_status": st}), flush=True)
        dist.close()
        if st != 0:
            raise SystemExit("device status %d" % st)
        return

    # correctness of the status word before timing anything
    sparse_step()
    torch.cuda.synchronize()
    st = twell.twell_get_device_status()
    if st != 0:
        raise RuntimeError("device status %d after the first step" % st)
    n_dense = int(route.n_dense[0].item())
    nnz_ell = int(route.ell_nnz[:M].sum().item())
    density = float(nnz.sum()) / (M * f)

    # per-kernel breakdown of both steps (untimed profiling passes); the
    # family with the largest share of the sparse step is the dominant kernel
    def breakdown(fn):
        twell.twell_profile_begin("*")
        for _ in range(2):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        fam = twell.twell_profile_end()
        total = sum(v[1] for v in fam.values())
        return fam, {k: {"launches_per_step": v[0] / 2, "ms_per_step": v[1] / 2,
                         "share": v[1] / total if total else 0.0}
                     for k, v in sorted(fam.items(), key=lambda kv: -kv[1][1])}

    fam, kernels = breakdown(sparse_step)
    _, kernels_fwd = breakdown(sparse_fwd)
    _, kernels_dense = breakdown(dense_step)
    dominant = max(fam, key=lambda k: fam[k][1])

    gpu_idx = os.environ.get("CUDA_VISIBLE_DEVICES", str(dist.local)).split(",")[0]
    clocks = ClockSampler(gpu_idx if gpu_idx.isdigit() else dist.local)
    # headline: each step replayed from a CUDA graph (sparse and dense alike)
    launches0 = twell.twell_launch_count()
    step_g = graphed(sparse_step)
    launches = twell.twell_launch_count() - launches0
    launches_per_step = launches / 2  # the eager step and the captured one
    ms_step, _, _, ck = timed(step_g, args.steps, args.warmup, clocks=clocks, key="sparse_fwd_bwd")
    fwd_g = graphed(sparse_fwd)
    ms_fwd, _, _, _ = timed(fwd_g, args.steps, args.warmup, key="sparse_fwd")
    # the same steps without the L2 flush (weights warm, as in back-to-back layers of one shape)
    ms_step_warm, _, _, _ = timed(step_g, args.steps, args.warmup, l2_flush=False)
    ms_fwd_warm, _, _, _ = timed(fwd_g, args.steps, args.warmup, l2_flush=False)
    # rows wider than 1024: the same step and forward with the pages' fused
    # gathers (h never leaves registers) in place of the default split ones
    ms_step_fused = ms_fwd_fused = None
    if d > 1024:
        twell.twell_set_split_gathers(False)
        try:
            ms_step_fused = timed(graphed(sparse_step), args.steps, args.warmup)[0]
            ms_fwd_fused = timed(graphed(sparse_fwd), args.steps, args.warmup)[0]
        finally:
            twell.twell_set_split_gathers(True)
    # classic-ELL ablation (inference path): the dense gate written to HBM in
    # bf16, converted by a separate pack kernel, then the same fused forward
    ms_classic = None
    if fwd_path == "twell":
        a_dense = torch.empty(M, f, dtype=torch.bfloat16, device=dev)

        def classic_fwd():
            twell.twell_gemm_bf16(x, wg, a_dense, M, f, d, False, False)
            twell.twell_pack_dense(a_dense, shape, tiles)
            twell.twell_ffn_fwd(x, wg, wu, wd, shape, y, tiles=tiles, ws=ws_t)

        ms_classic, _, _, _ = timed(graphed(classic_fwd), args.steps, args.warmup)
        del a_dense
    ms_dfwd, _, _, _ = timed(graphed(dense_fwd), args.steps, args.warmup)
    ms_dstep, _, _, _ = timed(graphed(dense_step), args.steps, args.warmup, key="dense_fwd_bwd")
    ms_sfwd, _, _, _ = timed(graphed(dense_silu_fwd), args.steps, args.warmup)
    ms_sstep, _, _, _ = timed(graphed(dense_silu_step), args.steps, args.warmup)
    # a second dense reference outside this library: the same ReLU-gated FFN
    # composed of PyTorch ops (cuBLAS GEMMs, autograd backward; no L1 term),
    # CUDA-graphed and timed the same way
    torch_dense = {}
    if not args.no_torch_dense:
        xt_ = x.detach().clone().requires_grad_()
        wgt_, wut_ = wg.detach().clone().requires_grad_(), wu.detach().clone().requires_grad_()
        wdt_ = wd.detach().t().contiguous().requires_grad_()  # [d][f], nn.Linear layout

        def torch_fwd():
            with torch.no_grad():
                y_t = (torch.relu(xt_ @ wgt_.T) * (xt_ @ wut_.T)) @ wdt_.T
            return y_t

        def torch_step():
            y_t = (torch.relu(xt_ @ wgt_.T) * (xt_ @ wut_.T)) @ wdt_.T
            return torch.autograd.grad(y_t, (xt_, wgt_, wut_, wdt_), dy)

        torch_step()
        torch_dense["fwd_ms"] = timed(graphed(torch_fwd), args.steps, args.warmup)[0]
        torch_dense["fwd_bwd_ms"] = timed(graphed(torch_step), args.steps, args.warmup)[0]
        torch_dense["sparse_speedup"] = {"fwd": torch_dense["fwd_ms"] / ms_fwd,
                                         "fwd_bwd": torch_dense["fwd_bwd_ms"] / ms_step}
        del xt_, wgt_, wut_, wdt_

    # small batches at this shape (M = 1, 16, 64): the TwELL forward reads all
    # of Wg once plus the distinct live rows of Wu and Wd, so it is HBM-bound;
    # the dense forward reads all three weight matrices
    small_m = {}
    if not args.no_small_m:
        peaks_, _ = load_peaks()
        for Ms in synthetic.SMALL_M:
            if Ms > M:
                continue
            xs = x[:Ms].contiguous()
            shp = twell.make_shape(Ms, d, f, wl.tile_n, wl.tile_cap)
            tl = twell.alloc_tiles(shp, dev)
            # the forward's optional workspace (rows wider than 1024): with
            # it, a handful of rows run as entry-parallel gathers
            tws = twell.twell_tiles_workspace_bytes(shp)
            wst = torch.empty(tws, dtype=torch.uint8, device=dev) if tws else None
            ys = torch.empty(Ms, d, dtype=torch.bfloat16, device=dev)
            wsd = torch.empty(twell.twell_dense_workspace_bytes(shp, False), dtype=torch.uint8,
                              device=dev)

            def small_gate():
                twell.twell_pack(xs, wg, shp, tl)

            def small_sparse():
                twell.twell_pack(xs, wg, shp, tl)
                twell.twell_ffn_fwd(xs, wg, wu, wd, shp, ys, tiles=tl, ws=wst)

            def small_dense():
                twell.twell_dense_ffn_fwd(xs, wg, wu, wd, shp, ys, False, wsd)

            t_gate = timed(graphed(small_gate), args.steps, args.warmup)[0]
            t_sp = timed(graphed(small_sparse), args.steps, args.warmup)[0]
            t_de = timed(graphed(small_dense), args.steps, args.warmup)[0]
            vt, it_, ct, _ = twell.tiles_view(tl, shp)
            T_, C_ = f // wl.tile_n, wl.tile_cap
            cols = (torch.arange(T_, device=dev).view(1, T_, 1) * wl.tile_n
                    + it_.long())[torch.arange(C_, device=dev).view(1, 1, C_)
                                  < ct.long().clamp(max=C_).unsqueeze(2)]
            n_unique = int(torch.unique(cols).numel())
            byts = 2 * f * d + 2 * 2 * n_unique * d + 2 * 2 * Ms * d
            gate_bytes = 2 * f * d + 2 * Ms * d
            small_m[str(Ms)] = {"sparse_fwd_us": t_sp * 1e3, "dense_fwd_us": t_de * 1e3,
                                "distinct_live_neurons": n_unique, "hbm_bytes": byts,
                                "frac_of_hbm": byts / (t_sp / 1e3) / 1e9 / peaks_["hbm_gbs"],
                                "gate_pack_us": t_gate * 1e3,
                                "gate_pack_frac_of_hbm": gate_bytes / (t_gate / 1e3) / 1e9
                                / peaks_["hbm_gbs"]}

    # eager steps with the dominant kernel's launches bracketed by CUDA events
    ms_eager, eager_launches, prof, _ = timed(sparse_step, args.steps, args.warmup,
                                              profile=dominant)

    # achievable row-gather bandwidth (the sparse kernels' access pattern):
    # rows of 2*d_model bytes at random ids from a table that fits in L2
    # (the weights of this workload) and from one ten times larger than L2
    def gather_rate(table_bytes, n_rows=1 << 20):
        row_bytes = 2 * d
        rows = table_bytes // row_bytes
        table = torch.empty(rows * row_bytes // 4, dtype=torch.int32, device=dev)
        idx = torch.randint(0, rows, (n_rows,), dtype=torch.int32, device=dev)
        blocks = 32 * twell.twell_num_sms()
        out = torch.empty(blocks * 8, dtype=torch.int32, device=dev)
        for _ in range(2):
            probe.gather(table, row_bytes, idx, out, blocks)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(5):
            probe.gather(table, row_bytes, idx, out, blocks)
        e1.record(stream)
        torch.cuda.synchronize()
        return 5 * n_rows * row_bytes / (e0.elapsed_time(e1) / 1e3) / 1e9

    # the L2-resident table is this workload's Wu + Wd, capped at half of L2
    # (the neuron chunk one pass of the gather kernels holds when the weights
    # exceed L2)
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    l2_table = min(2 * f * d * 2, l2_bytes // 2)
    gather_probe = {"row_bytes": 2 * d, "l2_resident_table_bytes": l2_table,
                    "l2_gbs": gather_rate(l2_table), "dram_table_bytes": 2 << 30,
                    "dram_gbs": gather_rate(2 << 30)}

    # roofline of the dominant kernel, from its events inside the timed region
    peaks, peak_src = load_peaks()
    roof = None
    cnt, dom_ms = prof.get(dominant, (0, 0.0)) if prof else (0, 0.0)
    work = algorithmic_work(dominant, wl, nnz_ell, n_dense)
    if work and cnt:
        amount, unit, bound = work
        # the formulas give a whole step's work; a family launched in several
        # L2-sized passes per step shares it among its launches
        amount /= cnt / args.steps
        per_launch_s = dom_ms / cnt / 1e3
        traffic, traffic_src = traffic_for(dominant, wl.name)
        if unit == "flop":
            achieved = amount / per_launch_s / 1e12
            roof = {"kernel": dominant, "bound": "tensor", "achieved": achieved,
                    "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": achieved / peaks["bf16_tflops"],
                    "peak_source": "%s bf16 burst (MEASURED_PEAKS.json)" % peak_src}
        else:
            # a gather whose weight rows L2 serves (DRAM traffic far below the
            # algorithmic bytes): its ceiling is the row-gather rate measured
            # in this run; the HBM copy rate is reported beside it
            achieved = amount / per_launch_s / 1e9
            roof = {"kernel": dominant, "bound": "l2", "achieved": achieved,
                    "peak": gather_probe["l2_gbs"], "unit": "GB/s",
                    "frac": achieved / gather_probe["l2_gbs"],
                    "peak_source": "row-gather probe of this run (%d-byte rows at random ids "
                                   "from an L2-resident table)" % gather_probe["row_bytes"],
                    "hbm_peak": peaks["hbm_gbs"], "frac_of_hbm": achieved / peaks["hbm_gbs"],
                    "hbm_peak_source": "%s HBM copy (MEASURED_PEAKS.json)" % peak_src}
        roof.update({"work_per_launch": amount, "work_unit": unit,
                     "ms_per_launch": dom_ms / cnt, "launches_per_step": cnt / args.steps,
                     "traffic": traffic, "traffic_source": traffic_src})

    memory = measure_memory(twell, shape, W, x, wg, wu, wd, dy, dev)

    # end to end through the C ABI with host buffers (H2D inputs, D2H results)
    xh = torch.empty((M, d), dtype=torch.bfloat16).pin_memory()
    dyh = torch.empty((M, d), dtype=torch.bfloat16).pin_memory()
    xh.copy_(x.cpu())
    dyh.copy_(dy.cpu())
    yh = torch.empty((M, d), dtype=torch.bfloat16).pin_memory()
    dxh = torch.empty((M, d), dtype=torch.bfloat16).pin_memory()

    # double-buffered: while step i computes (graph replay on the compute
    # stream, after its L2 flush), step i+1's inputs are copied in and step
    # i-1's results copied out on two copy streams; events keep a buffer set
    # from being overwritten while a copy or the compute still uses it
    # (the second set starts as a copy of the first: the eager call made
    # before each graph capture then routes the same rows, within the
    # route's capacity)
    bufs = [(x, dy, y, dx), (x.clone(), dy.clone(), torch.empty_like(y), torch.empty_like(dx))]
    step_graphs = [graphed(make_sparse_step(*b)) for b in bufs]
    comp = stream
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of set b copied in
    ev_done = [torch.cuda.Event() for _ in range(2)]  # compute on set b finished
    ev_out = [torch.cuda.Event() for _ in range(2)]   # results of set b copied out

    def copy_in(b):
        with torch.cuda.stream(h2d):
            h2d.wait_event(ev_done[b])
            bufs[b][0].copy_(xh, non_blocking=True)
            bufs[b][1].copy_(dyh, non_blocking=True)
            ev_in[b].record(h2d)

    def e2e_run(n_steps):
        copy_in(0)
        for i in range(n_steps):
            b = i % 2
            if i + 1 < n_steps:
                copy_in(1 - b)
            comp.wait_event(ev_out[b])
            flush.zero_()
            comp.wait_event(ev_in[b])
            step_graphs[b]()
            ev_done[b].record(comp)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev_done[b])
                yh.copy_(bufs[b][2], non_blocking=True)
                dxh.copy_(bufs[b][3], non_blocking=True)
                ev_out[b].record(d2h)
        comp.wait_stream(h2d)
        comp.wait_stream(d2h)

    e2e_run(args.warmup)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    e2e_run(args.steps)
    e1.record(comp)
    torch.cuda.synchronize()
    dist.barrier()
    ms_e2e = dist.max(e0.elapsed_time(e1) / args.steps, dev)
    if twell.twell_get_device_status() != 0:
        raise RuntimeError("device status after the end-to-end run")
    bi = 2 * M * d * 2
    bo = 2 * M * d * 2

    n = dist.world
    line = {
        "metric": METRIC, "value": n * M / (ms_step / 1e3), "unit": UNIT, "n_gpus": n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; gate offsets set for the target density)",
        "config": workload_config(wl, W, rf),
        "fwd_tokens_per_s": n * M / (ms_fwd / 1e3),
        "dense_fwd_tokens_per_s": n * M / (ms_dfwd / 1e3),
        "dense_fwd_bwd_tokens_per_s": n * M / (ms_dstep / 1e3),
        "speedup_vs_dense": {"fwd": ms_dfwd / ms_fwd, "fwd_bwd": ms_dstep / ms_step},
        "speedup_vs_dense_silu": {"fwd": ms_sfwd / ms_fwd, "fwd_bwd": ms_sstep / ms_step},
        "fwd_path": fwd_path,
        "ms": {"sparse_fwd_bwd": ms_step, "sparse_fwd": ms_fwd, "dense_fwd": ms_dfwd,
               "dense_fwd_bwd": ms_dstep, "sparse_fwd_bwd_eager": ms_eager,
               "sparse_fwd_bwd_warm_l2": ms_step_warm, "sparse_fwd_warm_l2": ms_fwd_warm,
               "classic_ell_fwd": ms_classic, "sparse_fwd_bwd_fused_gathers": ms_step_fused,
               "sparse_fwd_fused_gathers": ms_fwd_fused, "dense_silu_fwd": ms_sfwd,
               "dense_silu_fwd_bwd": ms_sstep},
        "ms_median": medians,
        "ms_per_step_median": medians.get("sparse_fwd_bwd"),
        "saved_for_backward_bytes": saved_bytes(shape, W, M, f, d),
        "memory": memory,
        "measured_density": density, "routed_rows": n_dense, "ell_entries": nnz_ell,
        "roofline": roof, "gather_probe": gather_probe, "kernels": kernels,
        "kernels_fwd": kernels_fwd, "kernels_dense_step": kernels_dense,
        "torch_cublas_dense": torch_dense or None,
        "small_m": small_m or None,
        "e2e": {"value": n * M / (ms_e2e / 1e3), "unit": UNIT, "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo, "ms_per_step": ms_e2e,
                "pipeline": "x, dY copied in from pinned host memory and y, dX copied out "
                            "every step on two copy streams, double-buffered so the copies "
                            "of steps i+1 and i-1 overlap step i's compute; the L2 flush "
                            "before each step's compute is inside the timed region"},
        "gpu_launches": int(launches_per_step * args.steps),
        "gpu_launches_per_step": launches_per_step,
        "timing": "each step replayed from a CUDA graph of the library calls; "
                  "ms.sparse_fwd_bwd_eager = the same step launched eagerly",
        "clocks": ck,
    }
    if dist.rank == 0 and n == 1 and not args.no_cpu_baseline:
        rate, rows, threads, secs, _ = cpu_sample_rate(wl, bits, W, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "oracle training step (gate, pack, route, sparse fwd, hybrid bwd) on "
                      "the first %d rows of the workload, %.1f s" % (rows, secs)}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


def measure_memory(twell, shape, W, x, wg, wu, wd, dy, dev):
    """Device memory of one training step, measured with the caching
    allocator's peak counter: every buffer a step allocates (packed format,
    routing arrays, workspace, y, dX, dW) from a state holding only the
    inputs and weights, the step run, and the peak read after it.  Also the
    bytes alive between forward and backward beyond y (what a training
    framework keeps for the backward)."""
    import torch

    M, d, f = shape.M, shape.d_model, shape.d_ff

    def window(run):
        torch.cuda.synchronize(dev)
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        kept = run()
        torch.cuda.synchronize(dev)
        peak = torch.cuda.max_memory_allocated(dev) - base
        return peak, kept

    def sparse():
        tiles = twell.alloc_tiles(shape, dev)
        twell.twell_pack(x, wg, shape, tiles)
        route = twell.alloc_hybrid(shape, W, dev)
        twell.hybrid_route(tiles, shape, route)
        del tiles  # transient: the route holds what the backward reads
        route.dense_cap = int(route.n_dense[0].item())
        ws = torch.empty(twell.twell_workspace_bytes(shape, W, True, dense_cap=route.dense_cap),
                         dtype=torch.uint8, device=dev)
        y = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
        twell.twell_ffn_fwd(x, wg, wu, wd, shape, y, route=route, ws=ws)
        torch.cuda.synchronize(dev)
        saved = torch.cuda.memory_allocated(dev) - base0[0] - y.numel() * 2
        dx = torch.empty_like(y)
        dws = [torch.empty(f, d, dtype=torch.float32, device=dev) for _ in range(3)]
        twell.twell_ffn_bwd(x, wg, wu, wd, dy, shape, route, L1, dx, *dws, ws)
        return saved, ws.numel()

    def dense():
        ws = torch.empty(twell.twell_dense_workspace_bytes(shape, True), dtype=torch.uint8,
                         device=dev)
        y = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
        twell.twell_dense_ffn_fwd(x, wg, wu, wd, shape, y, True, ws)
        torch.cuda.synchronize(dev)
        saved = torch.cuda.memory_allocated(dev) - base0[0] - y.numel() * 2
        dx = torch.empty_like(y)
        dws = [torch.empty(f, d, dtype=torch.float32, device=dev) for _ in range(3)]
        twell.twell_dense_ffn_bwd(x, wg, wu, wd, dy, shape, L1, dx, *dws, ws)
        return saved, ws.numel()

    base0 = [torch.cuda.memory_allocated(dev)]
    sp_peak, (sp_saved, sp_ws) = window(sparse)
    torch.cuda.synchronize(dev)
    base0[0] = torch.cuda.memory_allocated(dev)
    de_peak, (de_saved, de_ws) = window(dense)
    if twell.twell_get_device_status() != 0:
        raise RuntimeError("device status after the memory measurement")
    outputs = 2 * M * d * 2 + 3 * f * d * 4
    return {"sparse_step_peak_bytes": sp_peak, "dense_step_peak_bytes": de_peak,
            "sparse_over_dense_peak": sp_peak / de_peak,
            "sparse_saved_for_bwd_bytes": sp_saved, "dense_saved_for_bwd_bytes": de_saved,
            "sparse_workspace_bytes": sp_ws, "dense_workspace_bytes": de_ws,
            "outputs_bytes": outputs,
            "how": "torch.cuda.max_memory_allocated over one fwd+bwd step that allocates its "
                   "own buffers (packed tiles, routing arrays, workspace sized for the routed "
                   "rows, y, dX, dW; inputs and weights resident before); saved_for_bwd = bytes "
                   "alive after the forward beyond y"}


def saved_bytes(shape, W, M, f, d):
    """Activation memory kept from the forward for the backward: the sparse
    path keeps the hybrid ELL arrays (the TwELL tiles are transient: routing
    reads them once), the dense path keeps g, u and h (bf16 [M][d_ff] each)."""
    T, C = f // shape.tile_n, shape.tile_cap
    ell = M * W * (2 + 2) + M * 4 + M * 4 + 4
    tiles = M * T * C * (2 + 1) + M * T + M * 4
    dense = 3 * M * f * 2
    return {"sparse_ell": ell, "sparse_twell_tiles_transient": tiles, "dense_g_u_h": dense,
            "dense_over_sparse": dense / ell}


# device sources each kernel family is built from: a committed DRAM capture
# counts only while these files are unchanged
FAMILY_SOURCES = {
    "gemm": ("gemm_tc.cuh", "gemm_tc.cu", "common.cuh"),
    "sparse_fwd": ("sparse_fwd.cu", "ell_gather.cuh", "common.cuh"),
    "bwd": ("sparse_bwd.cu", "ell_gather.cuh", "common.cuh"),
}


def source_sha(kernel):
    """Fingerprint (sha256, 16 hex digits) of the sources of a kernel family."""
    import hashlib

    key = ("gemm" if kernel.startswith("gemm") else
           "sparse_fwd" if kernel.startswith("sparse_fwd") else "bwd")
    h = hashlib.sha256()
    for name in FAMILY_SOURCES[key]:
        with open(os.path.join(ROOT, "activation_sparse_gated_tcgen05_gb300", "csrc", name),
                  "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel, workload):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum)
    from a committed ncu capture of this kernel and workload
    (profiles/dram_traffic.json), and where it came from.  None when there
    is no capture or the kernel's sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as fh:
            e = json.load(fh).get(workload, {}).get(kernel)
    except (OSError, ValueError):
        e = None
    if not isinstance(e, dict) or "bytes" not in e:
        return None, "no ncu capture of this kernel and workload"
    if e.get("source_sha16") != source_sha(kernel):
        return None, "ncu capture predates the current kernel sources"
    return float(e["bytes"]), "ncu capture %s (profiles/dram_traffic.json)" % e.get("capture", "")


# ---------------------------------------------------------------- reference arm
def run_reference(args, dist):
    """The oracle as it stands on the host cores, same metric and workload,
    each step a bounded sample of the workload's rows."""
    if dist.rank != 0:
        return
    wl = synthetic.WORKLOADS[args.workload]
    bits = synthetic.make_workload(wl)
    import oracle

    # the ELL width from every row of the workload, as the GPU arm takes it
    oracle.set_threads(os.cpu_count() or 1)
    wg64 = oracle.f64(bits["wgT"])
    nnz = []
    for r0 in range(0, wl.M, 4096):  # row blocks bound the fp64 pre-activation's memory
        a = oracle.gate_preact(oracle.f64(bits["x"][r0:r0 + 4096]), wg64)
        nnz.append(oracle.twell_pack(a, wl.tile_n, wl.tile_cap)[3])
        del a
    nnz = np.concatenate(nnz)
    rf = wl.route_fraction if args.route_fraction is None else args.route_fraction
    W = synthetic.ell_width(nnz, rf)
    budget = 150.0 / max(1, args.steps + args.warmup)  # whole run within a few minutes
    _, rows, threads, _, w64 = cpu_sample_rate(wl, bits, W, None, step_budget=budget)
    import oracle as orc

    sample = np.arange(rows)
    for _ in range(args.warmup):
        oracle_step(orc, w64, bits, sample, wl, W)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(orc, w64, bits, sample, wl, W)
        times.append(time.perf_counter() - t0)
    sec = statistics.mean(times)
    value = rows / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; gate offsets set for the target density)",
        "config": workload_config(wl, W, rf),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "first %d rows of the workload per step" % rows},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    dist = Dist()
    if args.impl == "reference":
        run_reference(args, dist)
    else:
        run_own(args, dist)


if __name__ == "__main__":
    main()
