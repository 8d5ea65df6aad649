"""Benchmark of the batched block-preconditioner step (DASH-style Shampoo) on GB300.

Workload (default): a 24-layer Llama-style stack with d = 2048 -- per layer four
2048 x 2048 attention weights and three 2048 x 5632 MLP weights -- cut into
1024 x 1024 gradient blocks (Ng = 1248, the 512-wide MLP remainders
zero-padded), so that the L and R factors of all blocks form one
(2496, 1024, 1024) fp32 stack.  One step is the whole hot path with
preconditioner refresh every step (f = 1):
    accumulate (beta = 0.95, bf16 gradients) -> multi-vector power-iteration
    scale (32 vectors, 10 products, ridge 1e-6) -> Coupled Newton inverse 4th
    root in FP16 (10 iterations) -> preconditioned update L^-1/4 G R^-1/4 (TF32).
value  = factor blocks (inverse 4th roots) per second over the whole step;
ms_per_step = optimizer-step milliseconds.  Inputs (10.5 GB of factors) exceed
L2 (129 MB) many times over, so no flush is needed between steps.

--impl reference times the float64 CPU oracle instead (the only reference this
method has here), on a bounded sample of the same workload.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

LAYERS = 24
BS = 1024
BETA = 0.95
RIDGE = 1e-6
POWER_ITERS = 10
NVEC = 32
CN_ITERS = 10
NDB_ITERS = 10
SEED = 1004

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal dense ratios to bf16 (GB300): tf32 1.1 / 2.25 PFLOP/s.
TF32_RATIO = 1.1 / 2.25

# DRAM bytes (read + write) per launch of the FP16 GEMM class, averaged over the
# class's launches in one benchmark step at full size: an ncu capture of
# `bench.py --case step` with gpu__time_duration.sum, dram__bytes_read.sum and
# dram__bytes_write.sum (one pass).  Valid only for the sources it was taken on,
# identified by GEMM_TRAFFIC_SRC (None: not measured for these sources).
GEMM_TRAFFIC_PER_LAUNCH = 14.967e9  # 36 launches: 538.8 GB in 127.3 ms (serialised)
GEMM_TRAFFIC_SRC = "d1ec292ae7b61eb2"
GEMM_SOURCES = ("matrix_inverse_roots_gb300/csrc/gemm_tc.cu",
                "matrix_inverse_roots_gb300/csrc/dash_common.cuh",
                "matrix_inverse_roots_gb300/csrc/dash_api.cu")


def gemm_source_hash():
    import hashlib

    h = hashlib.sha256()
    root = os.path.dirname(os.path.abspath(__file__))
    for f in GEMM_SOURCES:
        with open(os.path.join(root, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def gemm_traffic():
    """Measured DRAM bytes of an average FP16-GEMM launch of the step, or None if the
    sources changed since the capture."""
    if GEMM_TRAFFIC_PER_LAUNCH is None or gemm_source_hash() != GEMM_TRAFFIC_SRC:
        return None
    return GEMM_TRAFFIC_PER_LAUNCH


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["_source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["_source"] = "fallback"
    return d


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------- GPU arm


class Workload:
    """The step on this rank's stack.  With world > 1 (data parallel, weak scaling)
    the model is `world` copies of the 24-layer stack; every rank holds its own
    data's gradients of all world x 1248 blocks (G_global), owns 1248 of them, and
    each step reduce-scatters the gradients to their owners, runs the hot path on
    the owned blocks and all-gathers the updates (shard.DataParallelStep)."""

    def __init__(self, torch, dr, synth, device, root_prec, ndb=False, power="fp16", rank=0,
                 world=1):
        self.torch = torch
        self.dr = dr
        dev = device
        G, vr, vc = synth.llama_layer_blocks(LAYERS, seed=SEED, var=1e-2, bs=BS, device=dev)
        self.G, self.vr, self.vc = G, vr, vc
        self.ng = G.shape[0]
        self.dp = None
        self.G_global = None
        if world > 1:
            from matrix_inverse_roots_gb300.shard import DataParallelStep

            self.G_global = torch.empty((world * self.ng, BS, BS), dtype=G.dtype, device=dev)
            for c in range(world):
                Gc, _, _ = synth.llama_layer_blocks(LAYERS, seed=SEED + 100 * rank + c, var=1e-2,
                                                    bs=BS, device=dev)
                self.G_global[c * self.ng:(c + 1) * self.ng].copy_(Gc)
                del Gc
            self.dp = DataParallelStep(world * self.ng, self.local_step)
        self.nf = 2 * self.ng
        self.F = torch.zeros((self.nf, BS, BS), dtype=torch.float32, device=dev)
        self.Froot = torch.empty_like(self.F)
        self.U = torch.empty((self.ng, BS, BS), dtype=torch.float32, device=dev)
        self.V0 = synth.start_vectors(self.nf, BS, NVEC, seed=SEED + 1, device=dev)
        self.lam = torch.empty(self.nf, dtype=torch.float32, device=dev)
        self.root_prec = root_prec
        self.apply_prec = dr.TF32 if root_prec in (dr.FP16, dr.BF16, dr.TF32) else dr.FP32_3XTF32
        # With a TF32 apply the root solver writes its roots already rounded to TF32
        # and apply reads them as they are (no conversion pass over both roots).
        fuse = self.apply_prec == dr.TF32 and not ndb
        self.root_out = root_prec | (dr.ROOT_TF32 if fuse else 0)
        self.apply_in = self.apply_prec | (dr.ROOT_TF32 if fuse else 0)
        self.ndb = ndb
        cap = 48 << 30
        # The pages' power iteration runs in half precision; "3xtf32" keeps it fp32-accurate.
        self.power_mode = {"3xtf32": dr.SCALE_POWER, "fp16": dr.SCALE_POWER_F16,
                           "bf16": dr.SCALE_POWER_BF16}[power]
        wprec = {"3xtf32": dr.FP32_3XTF32, "fp16": dr.FP16, "bf16": dr.BF16}[power]
        self.ws_scale = dr.workspace(dr.OP_SPECTRAL_SCALE, self.nf, BS, wprec, NVEC, device=dev)
        op = dr.OP_INV_ROOT_NDB if ndb else dr.OP_INV_ROOT_CN
        self.ws_root = dr.workspace(op, self.nf, BS, root_prec, NDB_ITERS if ndb else CN_ITERS,
                                    device=dev, max_bytes=cap)
        self.ws_apply = dr.workspace(dr.OP_PRECONDITION_APPLY, self.ng, BS, self.apply_prec,
                                     device=dev, max_bytes=16 << 30)

    def local_step(self, G_own):
        """The hot path on the owned gradient blocks; returns their updates."""
        self.G = G_own
        self.step_local()
        return self.U

    def step(self):
        if self.dp is not None:
            return self.dp(self.G_global)
        self.step_local()
        return self.U

    def step_local(self):
        dr = self.dr
        dr.shampoo_accumulate(self.G, self.F, BETA, self.vr, self.vc)
        dr.spectral_scale(self.F, self.power_mode, self.V0, POWER_ITERS, ridge=RIDGE,
                          out=self.lam, ws=self.ws_scale)
        if self.ndb:
            dr.inv_root_ndb(self.F, self.lam, NDB_ITERS, self.root_prec, ridge=RIDGE, X=self.Froot,
                            ws=self.ws_root)
        else:
            dr.inv_root_cn(self.F, self.lam, CN_ITERS, self.root_out, ridge=RIDGE, X=self.Froot,
                           ws=self.ws_root)
        dr.precondition_apply(self.G, self.Froot, self.apply_in, U=self.U, ws=self.ws_apply)

    def tiered_step(self, tiers, ws_auto, lam_min):
        """The step with the root solver chosen per block (inv_root_auto)."""
        dr = self.dr
        dr.shampoo_accumulate(self.G, self.F, BETA, self.vr, self.vc)
        dr.spectral_scale(self.F, self.power_mode, self.V0, POWER_ITERS, ridge=RIDGE,
                          out=self.lam, ws=self.ws_scale)
        # lambda_min in the fp32-accurate mode: a 16-bit copy of the shifted block
        # rounds lambda_max - lambda_min, so it cannot resolve lambda_min below about
        # u lambda_max (every block would look well conditioned).
        dr.spectral_lambda_min(self.F, self.lam, dr.SCALE_POWER, self.V0, POWER_ITERS,
                               ridge=RIDGE, out=lam_min, ws=self.ws_lmin)
        _, choice = dr.inv_root_auto(self.F, self.lam, lam_min, tiers, ridge=RIDGE,
                                     X=self.Froot, ws=ws_auto)
        dr.precondition_apply(self.G, self.Froot, self.apply_prec, U=self.U, ws=self.ws_apply)
        return choice

    def free(self):
        for k in ("G", "F", "Froot", "U", "V0", "ws_scale", "ws_root", "ws_apply", "G_global",
                  "dp"):
            setattr(self, k, None)


def timed_steps(torch, fn, steps, dist=None):
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        fn()
    t1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return t0.elapsed_time(t1) / steps


def e2e_steps(torch, wl, G_host, U_host, steps, dist=None):
    """End-to-end steps through the public API with host buffers.

    Every step uploads its gradient stack from pinned host memory and reads its update
    back to pinned host memory, all inside the timed region.  G and U are double
    buffered: step k's read-back and step k+1's upload run on two copy streams while
    the neighbouring steps compute (the uploads wait until the step two back has
    finished reading that G buffer; a step waits until the read-back of the U buffer it
    is about to overwrite has finished).  Each copy is bracketed by timing events on its
    own stream, so the link's achieved bandwidth is known: when the uploads plus the
    read-backs take longer than the compute, the step is bound by the host link.
    Returns (ms per step, upload ms per step, read-back ms per step)."""
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    # Data parallel: the input is this rank's gradients of every block, the result
    # read back is the update of the blocks this rank owns.
    gname = "G_global" if wl.dp is not None else "G"
    Gb = [getattr(wl, gname), torch.empty_like(getattr(wl, gname))]
    Ub = [wl.U, torch.empty_like(wl.U)]
    used = [torch.cuda.Event() for _ in range(2)]
    uploaded = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]
    spans = {"up": [], "down": []}

    def timed_copy(kind, stream, dst, src):
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dst.copy_(src, non_blocking=True)
        z.record(stream)
        spans[kind].append((a, z))
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    up.wait_stream(comp)
    with torch.cuda.stream(up):
        timed_copy("up", up, Gb[0], G_host)
        uploaded[0].record(up)
    for k in range(steps):
        b = k % 2
        if k + 1 < steps:
            nb = 1 - b
            if k >= 1:
                up.wait_event(used[nb])
            with torch.cuda.stream(up):
                timed_copy("up", up, Gb[nb], G_host)
                uploaded[nb].record(up)
        comp.wait_event(uploaded[b])
        if k >= 2:
            comp.wait_event(read[b])
        setattr(wl, gname, Gb[b])
        wl.U = Ub[b]
        wl.step()
        used[b].record(comp)
        down.wait_event(used[b])
        with torch.cuda.stream(down):
            timed_copy("down", down, U_host, Ub[b])
            read[b].record(down)
    comp.wait_stream(up)
    comp.wait_stream(down)
    t1.record(comp)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    setattr(wl, gname, Gb[0])
    wl.U = Ub[0]
    del Gb, Ub
    up_ms = sum(a.elapsed_time(z) for a, z in spans["up"]) / steps
    down_ms = sum(a.elapsed_time(z) for a, z in spans["down"]) / steps
    return t0.elapsed_time(t1) / steps, up_ms, down_ms


def full_optimizer_step(torch, dr, synth, wl, dev, steps, dist, peaks, lr=1e-3):
    """Times pack + accumulate + scale + CN + fused weight step on the bench workload."""
    shapes = synth.llama_weight_shapes(LAYERS)
    g = torch.Generator(device=dev).manual_seed(SEED + 7)
    Gw = [(0.1 * torch.randn((r, c), generator=g, device=dev)).to(torch.bfloat16)
          for r, c in shapes]
    offs, o = [], 0
    for r, c in shapes:
        offs.append(o)
        o += -(-r // BS) * -(-c // BS)
    assert o == wl.ng
    W = torch.zeros((wl.ng, BS, BS), dtype=torch.float32, device=dev)

    def step(refresh=True):
        for Gi, off in zip(Gw, offs):
            nb = -(-Gi.shape[0] // BS) * -(-Gi.shape[1] // BS)
            dr.pack_blocks(Gi, BS, out=wl.G[off:off + nb], valid=False)
        dr.shampoo_accumulate(wl.G, wl.F, BETA, wl.vr, wl.vc)
        if refresh:
            dr.spectral_scale(wl.F, wl.power_mode, wl.V0, POWER_ITERS, ridge=RIDGE, out=wl.lam,
                              ws=wl.ws_scale)
            dr.inv_root_cn(wl.F, wl.lam, CN_ITERS, wl.root_out, ridge=RIDGE, X=wl.Froot,
                           ws=wl.ws_root)
        dr.precondition_update(wl.G, wl.Froot, W, lr, wl.apply_in, ws=wl.ws_apply)

    step()
    dr.trace_start(400 * steps + 64)
    ms = timed_steps(torch, step, steps, dist)
    recs = dr.trace_records()
    dr.trace_stop()
    # Steps between root refreshes (f > 1) reuse the stale roots.
    stale_ms = timed_steps(torch, lambda: step(False), steps, dist)
    pack = [r for r in recs if r[0] == "pack"]
    pack_bytes = sum(r[2] for r in pack)
    pack_ms = sum(r[3] for r in pack)
    gbs = pack_bytes / (pack_ms * 1e-3) / 1e9 if pack_ms else None
    del Gw, W
    return {"ms_per_step": round(ms, 3),
            "blocks_per_s": round(wl.nf / (ms * 1e-3), 2),
            "what": "pack %d bf16 weight gradients -> (%d,1024,1024) + accumulate + scale + CN "
                    "fp16 x10 + fused W -= lr L^-1/4 G R^-1/4 (block layout)" % (len(shapes), wl.ng),
            "stale_root_step_ms": round(stale_ms, 3),
            "f10_ms_per_step": round((ms + 9 * stale_ms) / 10, 3),
            "pack_ms_per_step": round(pack_ms / steps, 3),
            "pack_gbs": None if gbs is None else round(gbs, 1),
            "pack_frac_hbm": None if gbs is None else round(gbs / peaks["hbm_gbs"], 4)}


def roofline_from_trace(records, peaks):
    by = {}
    for kind, fl, b, ms in records:
        e = by.setdefault(kind, [0, 0.0, 0.0, 0.0])
        e[0] += 1
        e[1] += fl
        e[2] += b
        e[3] += ms
    total_ms = sum(v[3] for v in by.values())
    dom = max(by, key=lambda k: by[k][3])
    n, fl, b, ms = by[dom]
    shares = {k: {"launches": v[0], "ms": round(v[3], 3),
                  "share": round(v[3] / total_ms, 4) if total_ms else 0.0} for k, v in by.items()}
    if dom.startswith("gemm"):
        base = peaks["bf16_tflops_sustained"]
        if dom == "gemm_tf32":
            peak = base * TF32_RATIO
        elif dom == "gemm_3xtf32":
            peak = base * TF32_RATIO / 3.0
        else:
            peak = base
        achieved = fl / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": "gemm_tc_kernel (%s)" % dom,
                "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4),
                "peak_note": "%s bf16 sustained%s" % (
                    peaks["_source"], "" if dom in ("gemm_f16", "gemm_bf16")
                    else " x nominal tf32/bf16 ratio" + (" / 3" if dom == "gemm_3xtf32" else "")),
                "launches": n, "avg_launch_ms": round(ms / n, 4),
                "flops_per_launch": fl / n,
                # Average over the class's launches in one step (ncu capture).
                "traffic": gemm_traffic() if dom == "gemm_f16" else None}
    else:
        peak = peaks["hbm_gbs"]
        achieved = b / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4), "launches": n,
                "avg_launch_ms": round(ms / n, 4), "traffic": None}
    return roof, shares, sum(v[0] for v in by.values())


def cpu_sample(ng_sample, rng_seed=SEED):
    """One oracle step on ng_sample gradient blocks (2*ng_sample factor blocks)."""
    import oracle

    rng = np.random.default_rng(rng_seed)
    G = rng.standard_normal((ng_sample, BS, BS)) * 0.1
    G = G.astype(np.float32).astype(np.float64)
    F = np.zeros((2 * ng_sample, BS, BS))
    V0 = rng.standard_normal((2 * ng_sample, BS, NVEC))
    t0 = time.perf_counter()
    F = oracle.accumulate(F, G, BETA)
    lam = oracle.power_lambda(F, V0, POWER_ITERS, ridge=RIDGE)
    X, _, _ = oracle.cn_inv_root(F, lam, CN_ITERS, ridge=RIDGE)
    oracle.apply_preconditioner(G, X)
    return time.perf_counter() - t0


def cpu_baseline(ng_sample=32):
    secs = cpu_sample(ng_sample)
    blocks = 2 * ng_sample
    return {"value": round(blocks / secs, 4), "unit": "blocks/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": "float64 oracle step (accumulate, 32-vector power x10, CN x10, apply) on "
                      "%d gradient blocks = %d factor blocks of 1024^2, %.1f s; numpy BLAS on "
                      "all host cores" % (ng_sample, blocks, secs)}


def run_gpu(args):
    import torch

    import matrix_inverse_roots_gb300 as dr
    import synth
    from matrix_inverse_roots_gb300.shard import job_throughput, max_over_ranks

    rank, world, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as tdist

        # NCCL's communicator set-up lines (rank count, transport) in the log.
        os.environ.setdefault("NCCL_DEBUG", "INFO")
        os.environ.setdefault("NCCL_DEBUG_SUBSYS", "INIT")
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = tdist
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    dr.load_library()
    peaks = load_peaks()

    wl = Workload(torch, dr, synth, dev, dr.FP16, power=args.power, rank=rank, world=world)
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    # Timed region: library kernel trace on, clocks sampled.
    launches_per_step = 250
    dr.trace_start(launches_per_step * args.steps + 64)
    clk = ClockSampler(dev.index)
    clk.start()
    ms = timed_steps(torch, wl.step, args.steps, dist)
    clocks = clk.stop()
    records = dr.trace_records()
    dr.trace_stop()
    assert dr.device_status() == 0, "device-side wait timed out"
    roof, shares, launches = roofline_from_trace(records, peaks)
    # Weak scaling: every rank refreshes its own stack of wl.nf blocks; the job
    # time is the slowest rank's and throughput counts the blocks of all ranks.
    value, ms = job_throughput(wl.nf, ms, device=dev)

    # The data-parallel exchange, when there is one, as its share of the step.
    exchange = None
    if wl.dp is not None:
        exchange = {"reduce_scatter_gb_per_rank": round(wl.G_global.numel() * 2 / 1e9, 2),
                    "all_gather_gb_per_rank": round(wl.G_global.numel() * 4 / 1e9, 2),
                    "what": "NCCL reduce-scatter of bf16 gradient blocks to their owners before "
                            "accumulate, all-gather of fp32 U after apply"}

    # Root-only throughput of the same kernel chain (CN FP16 on the whole stack).
    root_ms = timed_steps(torch, lambda: dr.inv_root_cn(wl.F, wl.lam, CN_ITERS, dr.FP16, ridge=RIDGE,
                                                         X=wl.Froot, ws=wl.ws_root), 2)

    # End to end: gradients from pinned host memory in, update back to pinned host memory.
    Gin = wl.G_global if wl.dp is not None else wl.G
    G_host = torch.empty(Gin.shape, dtype=Gin.dtype, pin_memory=True)
    G_host.copy_(Gin)
    U_host = torch.empty(wl.U.shape, dtype=wl.U.dtype, pin_memory=True)

    e2e_steps(torch, wl, G_host, U_host, 2)
    e2e_ms, up_ms, down_ms = e2e_steps(torch, wl, G_host, U_host, max(4, args.steps), dist)
    e2e_ms = max_over_ranks(e2e_ms, dev)
    h2d = G_host.numel() * G_host.element_size()
    d2h = U_host.numel() * U_host.element_size()
    del G_host, U_host

    # The whole optimizer step from weight-shaped gradients: every Llama weight's bf16
    # gradient packed into the block stack, accumulate, scale, CN, and the weight step
    # W <- W - lr U fused into the apply epilogue (W kept in the block layout).
    full = full_optimizer_step(torch, dr, synth, wl, dev, args.steps, dist, peaks)

    # The step with the root solver chosen per block by its condition estimate.
    tiered = None
    if not args.no_tiered:
        wl.ws_root = None
        torch.cuda.empty_cache()
        wl.ws_lmin = dr.workspace(dr.OP_LAMBDA_MIN, wl.nf, BS, dr.FP32_3XTF32, NVEC, device=dev)
        nb = min(dr.auto_workspace_size(wl.nf, BS, dr.DEFAULT_TIERS), 64 << 30)
        ws_auto = torch.empty(nb, dtype=torch.uint8, device=dev)
        lam_min = torch.empty_like(wl.lam)
        choice = wl.tiered_step(dr.DEFAULT_TIERS, ws_auto, lam_min)
        t_ms = timed_steps(torch, lambda: wl.tiered_step(dr.DEFAULT_TIERS, ws_auto, lam_min),
                           2, dist)
        counts = [choice.count(t) for t in range(len(dr.DEFAULT_TIERS))]
        tiered = {"ms_per_step": round(t_ms, 2), "blocks_per_s": round(wl.nf / (t_ms * 1e-3), 1),
                  "tiers": [dict(t) for t in dr.DEFAULT_TIERS], "blocks_per_tier": counts,
                  "what": "accumulate + power scale + lambda_min (shifted power iteration, "
                          "3xTF32) + per-block tier (inv_root_auto: gather, solve, scatter) + "
                          "apply"}
        del ws_auto, lam_min
        wl.ws_lmin = None
    wl.free()
    torch.cuda.empty_cache()

    # Same step with NDB in fp32 (3xTF32), a shorter run.
    ndb_ms = None
    if not args.no_ndb:
        wn = Workload(torch, dr, synth, dev, dr.FP32_3XTF32, ndb=True, power=args.power)
        wn.step()
        ndb_ms = timed_steps(torch, wn.step, 2, dist)
        wn.free()
        torch.cuda.empty_cache()

    line = {
        "metric": "B=1024 inverse-4th-root blocks/sec and optimizer-step ms; % tensor-core peak",
        "value": round(value, 2),
        "unit": "blocks/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {
            "workload": "llama-d2048 x24 layers: 1248 bf16 gradient blocks, (2496,1024,1024) fp32 "
                        "factor stack; step = accumulate(beta 0.95) + power scale(32 vec x10, "
                        + args.power + ") + CN fp16 x10 (roots stored TF32-rounded) + apply tf32, f=1",
            "blocks": wl.nf, "block": BS, "root": "cn-fp16", "iters": CN_ITERS,
            "l2": "inputs 10.5 GB >> 129 MB L2, no flush",
        },
        "roofline": roof,
        "kernel_shares": shares,
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": {"value": round(wl.nf * world / (e2e_ms * 1e-3), 2), "unit": "blocks/s",
                "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "h2d_ms_per_step": round(up_ms, 2), "d2h_ms_per_step": round(down_ms, 2),
                "h2d_gbs": round(h2d / (up_ms * 1e6), 1), "d2h_gbs": round(d2h / (down_ms * 1e6), 1),
                "copies": "pinned host buffers; uploads and read-backs on two copy streams, "
                          "G and U double-buffered so they overlap the neighbouring steps"},
        "root_only_blocks_per_s": round(wl.nf / (root_ms * 1e-3), 1),
        "tiered_step": tiered,
        "exchange": exchange,
        "ndb_fp32_step_ms": None if ndb_ms is None else round(ndb_ms, 2),
        "optimizer_step": full,
        "peaks_source": peaks["_source"],
    }
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------------ solver sweep


SWEEP_SIZES = ((256, 61035), (512, 15259), (1024, 3815), (2048, 954))
SWEEP_RUNS = (("cn", "fp16"), ("cn", "bf16"), ("cn", "tf32"), ("cn", "3xtf32"),
              ("ndb", "tf32"), ("ndb", "3xtf32"), ("cheb8", "3xtf32"), ("cheb16", "3xtf32"),
              ("cheb32", "3xtf32"))


def run_sweep(args):
    """Inverse-root throughput over ~16 GB Wishart stacks per block size (one JSON
    line per block size, solver and precision; not the headline line)."""
    import torch

    import matrix_inverse_roots_gb300 as dr
    import synth

    torch.cuda.set_device(0)
    dr.load_library()
    peaks = load_peaks()
    sizes = SWEEP_SIZES if not args.sweep_b else [x for x in SWEEP_SIZES if x[0] in args.sweep_b]
    for b, n in sizes:
        A = synth.wishart(n, b, seed=1005 + b, device="cuda", chunk=256)
        s = dr.spectral_scale(A, dr.SCALE_FROBENIUS)
        X = torch.empty_like(A)
        for solver, prec in SWEEP_RUNS:
            p = dr.PRECISIONS[prec]
            if solver == "cn":
                op, param = dr.OP_INV_ROOT_CN, CN_ITERS
            elif solver == "ndb":
                op, param = dr.OP_INV_ROOT_NDB, NDB_ITERS
            else:
                op, param = dr.OP_INV_ROOT_CHEB, int(solver[4:])
            ws = dr.workspace(op, n, b, p, param, max_bytes=48 << 30)
            if solver == "cn":
                fn = lambda: dr.inv_root_cn(A, s, CN_ITERS, p, X=X, ws=ws)
            elif solver == "ndb":
                fn = lambda: dr.inv_root_ndb(A, s, NDB_ITERS, p, X=X, ws=ws)
            else:
                fn = lambda: dr.inv_root_cheb(A, s, param, 1e-2, 1.05, p, X=X, ws=ws)
            fn()
            dr.trace_start(4096)
            ms = timed_steps(torch, fn, 2)
            # Tensor-core work as executed: a symmetric-half product counts only the
            # tiles it computes (the library's trace records those flops).
            executed = sum(r[1] for r in dr.trace_records() if r[0].startswith("gemm")) / 2
            dr.trace_stop()
            mm = dr.op_matmuls(op, param)
            tflops = executed / (ms * 1e-3) / 1e12
            dense = mm * 2.0 * b ** 3 * n / (ms * 1e-3) / 1e12
            base = peaks["bf16_tflops_sustained"]
            peak = base if prec in ("fp16", "bf16") else (
                base * TF32_RATIO if prec == "tf32" else base * TF32_RATIO / 3.0)
            print(json.dumps({"sweep": True, "B": b, "N": n, "solver": solver, "prec": prec,
                              "ms": round(ms, 2), "blocks_per_s": round(n / (ms * 1e-3), 1),
                              "matmuls_per_block": mm, "tflops": round(tflops, 1),
                              "dense_equivalent_tflops": round(dense, 1),
                              "peak_tflops": round(peak, 1), "frac": round(tflops / peak, 4)}),
                  flush=True)
            del ws
            torch.cuda.empty_cache()
        del A, X, s
        torch.cuda.empty_cache()


# ------------------------------------------------------------------ profiling case


def run_case(args):
    """A small untimed case for ncu captures: Wishart blocks, a scale, one root call;
    --case accumulate: one accumulate of n bf16 Llama-like gradient blocks into 2n
    factors (two GEMM launches, with mirrored stores when B is a multiple of 256);
    --case apply: one preconditioned update of n blocks (the gradient conversion, two
    GEMMs); --case pack: n stacked 2048 x 5632 bf16 gradients into blocks and back;
    --case auto: per-block solver choice on n blocks alternating between two tiers;
    --case step: two steps of the benchmark workload (profile the second)."""
    import torch

    import matrix_inverse_roots_gb300 as dr
    import synth

    torch.cuda.set_device(0)
    dr.load_library()
    n, b = args.case_n, args.case_b
    if args.case == "step":
        # One warm-up step of the benchmark workload, then the step a profiler
        # captures (skip the first step's launches).
        wl = Workload(torch, dr, synth, torch.device("cuda", 0), dr.FP16, power=args.power)
        wl.step()
        torch.cuda.synchronize()
        wl.step()
        torch.cuda.synchronize()
        print("case ok, device status", dr.device_status())
        return
    if args.case in ("apply", "pack"):
        g = torch.Generator(device="cuda").manual_seed(5)
        G = (0.1 * torch.randn((n, b, b), generator=g, device="cuda")).to(torch.bfloat16)
        if args.case == "apply":
            R = synth.wishart(2 * n, b, seed=6, device="cuda")
            dr.precondition_apply(G, R, args.case_prec)
        else:
            # n Llama MLP weights' gradients stacked (2048 n x 5632, row-major) into
            # their blocks (184 MB at n = 8: more than L2), and back.
            M = (0.1 * torch.randn((2048 * n, 5632), generator=g, device="cuda")).to(torch.bfloat16)
            P, _, _ = dr.pack_blocks(M, b)
            dr.unpack_blocks(P, M.shape[0], M.shape[1], out=torch.empty_like(M))
        torch.cuda.synchronize()
        print("case ok, device status", dr.device_status())
        return
    if args.case == "auto":
        # Per-block solver choice on blocks alternating between the two default tiers
        # (kappa 2 and 1e4): lambda_max and lambda_min in the fp32-accurate mode, then
        # each tier gathered, solved and scattered back.
        A = synth.two_cluster_blocks(n, b, 5).cuda()
        V0 = synth.start_vectors(n, b, 32, seed=6, device="cuda")
        lam = dr.spectral_scale(A, dr.SCALE_POWER, V0, POWER_ITERS)
        lmin = dr.spectral_lambda_min(A, lam, dr.SCALE_POWER, V0, POWER_ITERS)
        dr.inv_root_auto(A, lam, lmin, dr.DEFAULT_TIERS)
        torch.cuda.synchronize()
        print("case ok, device status", dr.device_status())
        return
    if args.case == "accumulate":
        g = torch.Generator(device="cuda").manual_seed(5)
        G = (0.1 * torch.randn((n, b, b), generator=g, device="cuda")).to(torch.bfloat16)
        F = torch.zeros((2 * n, b, b), dtype=torch.float32, device="cuda")
        dr.shampoo_accumulate(G, F, BETA)
        torch.cuda.synchronize()
        print("case ok, device status", dr.device_status())
        return
    A = synth.wishart(n, b, seed=5, device="cuda")
    if args.case_scale in ("power", "power-fp16"):
        mode = dr.SCALE_POWER if args.case_scale == "power" else dr.SCALE_POWER_F16
        s = dr.spectral_scale(A, mode, synth.start_vectors(n, b, 32, seed=6, device="cuda"),
                              POWER_ITERS)
    else:
        s = dr.spectral_scale(A, dr.SCALE_FROBENIUS)
    if args.case == "cn":
        dr.inv_root_cn(A, s, args.case_iters, args.case_prec)
    elif args.case == "ndb":
        dr.inv_root_ndb(A, s, args.case_iters, args.case_prec)
    else:
        dr.inv_root_cheb(A, s, args.case_iters, 1e-2, 1.05, args.case_prec)
    torch.cuda.synchronize()
    print("case ok, device status", dr.device_status())


# ------------------------------------------------------------------ reference arm


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    ng = 2
    for _ in range(args.warmup):
        cpu_sample(ng)
    times = [cpu_sample(ng) for _ in range(args.steps)]
    secs = sum(times) / len(times)
    blocks = 2 * ng
    value = blocks / secs
    # The GPU arm's stack: an L and an R factor per gradient block of the 24 layers.
    import synth

    nf = 2 * len(synth.llama_block_layout(LAYERS, BS)[0])
    line = {
        "impl": "reference",
        "metric": "B=1024 inverse-4th-root blocks/sec and optimizer-step ms; % tensor-core peak",
        "value": round(value, 4),
        "unit": "blocks/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 * nf / blocks, 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "llama-d2048 x24 layers step (as the GPU arm), timed on a sample "
                               "of %d gradient blocks per step; ms_per_step extrapolated to "
                               "2496 factor blocks" % ng,
                   "blocks": nf, "block": BS},
        "cpu_baseline": {"value": round(value, 4), "unit": "blocks/s", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": "%d gradient blocks (%d factor blocks) per step" % (ng, blocks)},
        "e2e": {"value": round(value, 4), "unit": "blocks/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="dash", choices=["dash", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-ndb", action="store_true", help="skip the NDB fp32 step")
    ap.add_argument("--no-tiered", action="store_true",
                    help="skip the step with per-block solver selection")
    ap.add_argument("--power", choices=["fp16", "bf16", "3xtf32"], default="fp16",
                    help="arithmetic of the power-iteration scaling (the pages: half precision)")
    ap.add_argument("--sweep", action="store_true",
                    help="inverse-root throughput sweep over block sizes and precisions")
    ap.add_argument("--sweep-b", type=int, nargs="*", default=None)
    ap.add_argument("--case", choices=["cn", "ndb", "cheb", "accumulate", "apply", "pack", "step",
                                       "auto"],
                    default=None,
                    help="run one small untimed case (for profiler captures)")
    ap.add_argument("--case-n", type=int, default=64)
    ap.add_argument("--case-b", type=int, default=1024)
    ap.add_argument("--case-prec", default="fp16")
    ap.add_argument("--case-iters", type=int, default=3)
    ap.add_argument("--case-scale", choices=["power", "power-fp16", "frobenius"], default="power")
    args = ap.parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ and not (args.case or args.sweep):
        # One process per GPU: relaunch this command under torch.distributed.run.
        import socket

        with socket.socket() as s:
            s.bind(("127.0.0.1", 0))
            port = s.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               "--nproc-per-node=%d" % args.gpus, "--master-addr", "127.0.0.1",
               "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
        sys.exit(subprocess.call(cmd))
    if args.case:
        run_case(args)
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
