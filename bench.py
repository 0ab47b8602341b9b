#!/usr/bin/env python
"""Benchmark: VSA (video sparse attention) forward + backward on GB300.

One step = the whole hot path on one batch: SFC reorder + cube pool, coarse
attention + Top-K, tcgen05 fine attention, gated combine (forward), then the
full backward (combine backward, coarse backward, fine backward, pool backward
+ inverse reorder), through the library's C ABI (vsa_forward / vsa_backward).

Metric: effective TFLOP/s = FLOPs the method needs at the given sparsity
(fine: 4*N*64K*d forward + 10*N*64K*d backward; coarse: 4*Nc^2*d + 10*Nc^2*d,
per batch*head) divided by the step time; reported whole-job (all ranks).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs an
independent replica of the workload (heads are independent; no collective on
the data path) and the max time over ranks is used.
"""
from __future__ import annotations

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
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "VSA fwd+bwd effective TFLOPS at 32K tokens, 70% sparsity; % of bf16 tensor peak"
UNIT = "TFLOP/s"
# libvsa kernels launched by one forward + backward step (the ncu launch list
# of the bench's step shows exactly these): permute_pool, coarse_fwd,
# pair_overlap, plan_pairs, fine_fwd, combine | inv_count, inv_scan, inv_fill,
# pair_overlap, plan_pairs, bwd_prep, coarse_bwd, fine_bwd_kv, fine_bwd_dq.
KERNELS_PER_STEP = 15
WORKLOAD = "wan1.3b"


class near_gpu_memory:
    """Within the block, this thread runs on the CPUs of the GPU's own NUMA
    node, so that pinned host buffers allocated there are first touched in
    that node's memory (the host<->device copies then take the shortest path);
    the previous CPU set is restored afterwards.  Does nothing where the
    topology cannot be read."""

    def __init__(self, device_index: int):
        self.cpus = None
        try:
            import torch
            p = torch.cuda.get_device_properties(device_index)
            bus = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
            with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
                node = int(f.read().strip())
            if node >= 0:
                with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
                    cpus = set()
                    for part in f.read().strip().split(","):
                        a, _, b = part.partition("-")
                        cpus.update(range(int(a), int(b or a) + 1))
                self.cpus = cpus & os.sched_getaffinity(0) or None
        except (OSError, ValueError, AttributeError):
            self.cpus = None

    def __enter__(self):
        self.saved = os.sched_getaffinity(0)
        if self.cpus:
            os.sched_setaffinity(0, self.cpus)
        return self

    def __exit__(self, *exc):
        os.sched_setaffinity(0, self.saved)
        return False


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over all ranks (every rank receives it); x itself at world 1."""
    if world == 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_step: float, steps: int, ms: float) -> float:
    """Replicas: every rank runs the whole workload, so the job does world x the
    work of one rank in the slowest rank's time."""
    return world * flops_per_step * steps / (ms * 1e-3) / 1e12


def step_flops(wl: synth.Workload, cubes: float = None) -> dict:
    # keys per query: the listed cubes (K, or the mean list length when the
    # lists are Top-K united with a neighbourhood) of N / Nc tokens on average
    # (64 unless the grid has partial boundary cubes)
    keys = (wl.topk if cubes is None else cubes) * wl.N / wl.Nc
    fine_fwd = 4.0 * wl.N * keys * wl.d * wl.BH
    fine_bwd = 10.0 * wl.N * keys * wl.d * wl.BH
    coarse = 14.0 * wl.Nc * wl.Nc * wl.d * wl.BH
    return dict(fine_fwd=fine_fwd, fine_bwd=fine_bwd, coarse=coarse, total=fine_fwd + fine_bwd + coarse)


def kernel_flops(wl: synth.Workload, cubes: float = None) -> dict:
    """Work each fine kernel does per launch, in products of 2*N*64K*d FLOP per
    (batch, head): forward S and PV (2); backward dK/dV kernel S^T, dP^T, dV,
    dK (4); dQ kernel S, dP, dQ (3).  The effective metric counts 2 + 5: of the
    dQ kernel only its dQ product (dq_product) is new work."""
    unit = 2.0 * wl.N * ((wl.topk if cubes is None else cubes) * wl.N / wl.Nc) * wl.d * wl.BH
    return {"fine_fwd": 2 * unit, "fine_bwd_kv": 4 * unit, "fine_bwd_dq": 3 * unit, "dq_product": unit}


def roof(flops: float, ms: float, peak: float) -> dict:
    a = flops / (ms * 1e-3) / 1e12
    return {"ms": round(ms, 4), "tflops": round(a, 2), "frac": round(a / peak, 4), "flops_per_launch": flops}


def fine_bwd_wall(per_kernel: dict) -> tuple:
    """(ms, overlapped): the fine backward's wall time per step.  vsa_backward
    runs the dK/dV kernel on a higher-priority stream of its own while the
    coarse backward and then the dQ kernel run on the caller's stream, filling
    the SMs the dK/dV kernel leaves; the coarse and dQ event pairs then follow
    one another on the caller's stream and together span the fine backward
    (the coarse backward included).  Back to back, the two kernel intervals add."""
    overlapped = per_kernel["fine_bwd_dq"] > per_kernel["fine_bwd_kv"]
    ms = (per_kernel["coarse_bwd"] + per_kernel["fine_bwd_dq"] if overlapped
          else per_kernel["fine_bwd_kv"] + per_kernel["fine_bwd_dq"])
    return ms, overlapped


def public_calls(public, per_kernel: dict, bwd_ms: float, overlapped: bool):
    """The public calls' times beside the fine stage inside the whole pass:
    vsa_fine_fwd against the fine forward kernel, vsa_fine_bwd against the
    fine backward's wall time (without the coarse backward)."""
    if not public:
        return None
    inner = {"fine_fwd": per_kernel["fine_fwd"],
             "fine_bwd": bwd_ms - per_kernel["coarse_bwd"] if overlapped else bwd_ms}
    return {n: dict(v, internal_ms=round(inner[n], 4), ratio=round(v["ms"] / inner[n], 3)) for n, v in public.items()}


def config_of(wl: synth.Workload, parallelism: str, curve: str = "raster", radius: int = -1) -> dict:
    return {
        "workload": (f"{wl.name}: B={wl.B}, heads={wl.heads}, d={wl.d}, grid (T,H,W)=({wl.T},{wl.H},{wl.W}) = "
                     f"{wl.N} tokens, {wl.Nc} cubes of (4,4,4), Top-K={wl.topk} "
                     f"({100 * wl.sparsity:.1f}% sparsity), learnable gates on"),
        "global_batch": wl.B,
        "seq_len": wl.N,
        "heads": wl.heads,
        "head_dim": wl.d,
        "topk": wl.topk,
        "parallelism": parallelism,
        "l2": "inputs larger than L2: 6 bf16 tensors of 100.7 MB per step (Q,K,V,gates,dO)",
        "inputs": "synthetic smooth field + noise (synth.py), seed base 20250519",
        "out_dtype": "bf16", "grad_dtype": "bf16",
        "cube_order": curve,
        "selection": ("Top-K" if radius < 0 else f"Top-K united with the radius-{radius} cube neighbourhood"),
    }


def load_peaks() -> dict:
    """The dense bf16 tensor peaks and the copy bandwidth: measured on this
    pool's GB300s when MEASURED_PEAKS.json is present, else the fallback.
    burst: cuBLAS timed alone at full clock; sustained: a seconds-long GEMM
    loop under the power cap (fp16 has the same nominal rate as bf16)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(burst=p["bf16_tflops"], sustained=p.get("bf16_tflops_sustained") or p["bf16_tflops"],
                    hbm=p["hbm_gbs"], source="measured (MEASURED_PEAKS.json)")
    return dict(burst=1900.0, sustained=1700.0, hbm=6800.0, source="fallback")


def pick_peak(peaks: dict, clocks: dict) -> tuple:
    """(peak, kind) for the timed region: the burst peak when its SM clock
    stayed at the maximum (median within 3%) with no power cap or slowdown
    active, as for the burst measurement; the sustained peak otherwise."""
    sm, smax, reasons = clocks.get("sm_mhz"), clocks.get("sm_max_mhz"), clocks.get("reasons") or []
    at_max = bool(sm and smax and sm >= 0.97 * smax)
    capped = any(r in reasons for r in ("sw_power_cap", "hw_slowdown", "hw_thermal_slowdown",
                                        "sw_thermal_slowdown", "no samples"))
    if at_max and not capped:
        return peaks["burst"], "burst"
    return peaks["sustained"], "sustained"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self) -> dict:
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle sample
def oracle_sample(wl: synth.Workload, budget_s: float, rows_hint: int = 0):
    """Time the CPU oracle on head 0: the coarse stage in full plus the fine
    forward and the fine backward (dQ) of a subset of query rows.  Returns
    (effective FLOPs done, seconds, rows, threads)."""
    import oracle
    oracle.build()
    q, k, v = (a.reshape(1, wl.N, wl.d) for a in synth.make_qkv(wl, heads_subset=[0]))
    dout = synth.make_dout(wl, heads_subset=[0]).reshape(1, wl.N, wl.d)
    scale = wl.d ** -0.5
    rng = np.random.default_rng(7)

    def run(rows: int):
        t0 = time.perf_counter()
        qp, kp, vp, dp = (oracle.permute(a, wl.T, wl.H, wl.W) for a in (q, k, v, dout))
        pq, pk, pv = (oracle.pool(a) for a in (qp, kp, vp))
        scores, _, _ = oracle.coarse(pq, pk, pv, scale)
        idx = oracle.topk(scores, wl.topk)
        cnt = np.full(idx.shape[:-1], wl.topk, np.int32)
        sel = np.sort(rng.choice(wl.N, rows, replace=False))
        oracle.fine_fwd_rows(qp, kp, vp, idx, cnt, scale, sel)
        oracle.fine_bwd_query_rows(qp, kp, vp, dp, idx, cnt, scale, sel)
        dt = time.perf_counter() - t0
        # per row: forward 4*64K*d; backward recompute of S, dP and dQ 6*64K*d
        flops = rows * 10.0 * 64 * wl.topk * wl.d + 4.0 * wl.Nc * wl.Nc * wl.d
        return flops, dt

    if rows_hint <= 0:
        f0, t0 = run(128)
        per_row = max(t0, 1e-3) / 128
        rows_hint = int(min(wl.N, max(64, budget_s / per_row)))
    flops, dt = run(rows_hint)
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return flops, dt, rows_hint, threads


# ----------------------------------------------------------------------------- other configurations
OTHER_CONFIGS = ["wan1.3b_k512", "wan1.3b_k256", "wan1.3b_k64", "wan14b", "long"]


def measure_other_configs(vsa, dev, args, headline_inputs, order) -> dict:
    """The sparsity sweep (Top-K 512 / 256 / 64 of 512 cubes), the 40-head
    Wan-14B-shaped layer and the 122880-token long video: each a full
    forward + backward step, timed like the headline (warm-up, then CUDA
    events around `config_steps` steps, per-kernel event pairs).  The sweep
    reuses the headline layer's inputs (same tensors, another K); the other
    two get their own seeded inputs.  Each also gets an oracle sample on the
    host cores (head 0, coarse stage in full plus sampled fine rows)."""
    import torch
    runs = {}
    with ClockSampler(dev.index or 0) as clocks:
        for name in OTHER_CONFIGS:
            wl = synth.WORKLOADS[name]
            if wl.T == synth.WORKLOADS[WORKLOAD].T and wl.heads == synth.WORKLOADS[WORKLOAD].heads and \
                    wl.H == synth.WORKLOADS[WORKLOAD].H and wl.W == synth.WORKLOADS[WORKLOAD].W:
                inputs, src = headline_inputs, f"the {WORKLOAD} layer's inputs"
            else:
                q, k, v = synth.make_qkv(wl)
                gc, gf = synth.make_gates(wl)
                dout = synth.make_dout(wl)
                inputs = tuple(torch.from_numpy(a).to(dev).to(torch.bfloat16) for a in (q, k, v, gc, gf, dout))
                del q, k, v, gc, gf, dout
                src = "own seeded inputs"
            qd, kd, vd, gcd, gfd, dod = inputs
            out = torch.empty_like(qd)
            grads = {n: torch.empty_like(qd) for n in ("dq", "dk", "dv", "dgc", "dgf")}
            fws = torch.empty(vsa.workspace_bytes(0, wl.B, wl.heads, wl.d, wl.T, wl.H, wl.W, wl.topk),
                              dtype=torch.uint8, device=dev)
            bws = torch.empty(vsa.workspace_bytes(1, wl.B, wl.heads, wl.d, wl.T, wl.H, wl.W, wl.topk),
                              dtype=torch.uint8, device=dev)
            ordr = None if order is None else vsa.cube_order(wl.T, wl.H, wl.W, args.curve, device=dev)

            def step():
                _, st = vsa.forward(qd, kd, vd, wl.T, wl.H, wl.W, wl.topk, g_coarse=gcd, g_fine=gfd, out=out,
                                    ws=fws, cube_order=ordr)
                vsa.backward(st, dod, g_coarse=gcd, g_fine=gfd, grads=grads, ws=bws)

            for _ in range(max(3, args.warmup)):
                step()
            torch.cuda.synchronize()
            assert vsa.device_status() == 0, f"device error flag set in {name}"
            vsa.timing_read()
            stream = torch.cuda.current_stream()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            vsa.timing_enable(True)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(args.config_steps):
                step()
            e1.record(stream)
            torch.cuda.synchronize()
            vsa.timing_enable(False)
            ms = e0.elapsed_time(e1) / args.config_steps
            kern = vsa.timing_read()
            assert vsa.device_status() == 0, f"device error flag set in {name}"
            per_kernel = {n: t / max(c, 1) for n, (t, c) in kern.items()}
            fl = step_flops(wl)
            bwd_ms, _ = fine_bwd_wall(per_kernel)
            runs[name] = {
                "workload": config_of(wl, "single GPU", args.curve)["workload"],
                "inputs": src, "steps": args.config_steps, "ms_per_step": round(ms, 3),
                "tflops": round(fl["total"] / (ms * 1e-3) / 1e12, 2),
                "fine_fwd_ms": round(per_kernel["fine_fwd"], 4),
                "fine_bwd_ms": round(bwd_ms, 4),
                "per_kernel": per_kernel, "kflops": kernel_flops(wl),
            }
            del out, grads, fws, bws, inputs, qd, kd, vd, gcd, gfd, dod
            torch.cuda.empty_cache()
    if not args.no_cpu_baseline:
        for name in OTHER_CONFIGS:
            flops, dt, rows, threads = oracle_sample(synth.WORKLOADS[name], args.config_cpu_seconds)
            runs[name]["cpu_oracle"] = {"tflops": round(flops / dt / 1e12, 6), "cores": threads,
                                        "sample": f"head 0: coarse stage in full + fine fwd/bwd (dQ) of {rows} rows"}
    return {"clocks": clocks.summary(), "runs": runs,
            "note": "fractions against the same peak as the headline; each config's own timed steps"}


# ----------------------------------------------------------------------------- GPU arm
def run_ours(args, rank: int, world: int):
    import torch
    import block_sparse_video_sfc_gb300 as vsa

    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = synth.WORKLOADS[args.config]

    q, k, v = synth.make_qkv(wl)
    gc, gf = synth.make_gates(wl)
    dout = synth.make_dout(wl)
    with near_gpu_memory(local):
        host = [torch.from_numpy(a).to(torch.bfloat16).pin_memory() for a in (q, k, v, gc, gf, dout)]
    dq_, dk_, dv_, dgc_, dgf_, ddo = (h.to(dev) for h in host)
    out = torch.empty_like(dq_)
    grads = dict(dq=torch.empty_like(dq_), dk=torch.empty_like(dq_), dv=torch.empty_like(dq_),
                 dgc=torch.empty_like(dq_), dgf=torch.empty_like(dq_))
    fws = torch.empty(vsa.workspace_bytes(0, wl.B, wl.heads, wl.d, wl.T, wl.H, wl.W, wl.topk, args.radius),
                      dtype=torch.uint8, device=dev)
    bws = torch.empty(vsa.workspace_bytes(1, wl.B, wl.heads, wl.d, wl.T, wl.H, wl.W, wl.topk, args.radius),
                      dtype=torch.uint8, device=dev)
    order = None if args.curve == "raster" else vsa.cube_order(wl.T, wl.H, wl.W, args.curve, device=dev)

    def step(qd, kd, vd, gcd, gfd, dod, res_out=None, res_grads=None):
        _, st = vsa.forward(qd, kd, vd, wl.T, wl.H, wl.W, wl.topk, g_coarse=gcd, g_fine=gfd,
                            out=out if res_out is None else res_out, ws=fws, cube_order=order, radius=args.radius)
        vsa.backward(st, dod, g_coarse=gcd, g_fine=gfd, grads=grads if res_grads is None else res_grads, ws=bws)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step(dq_, dk_, dv_, dgc_, dgf_, ddo)
    torch.cuda.synchronize()
    assert vsa.device_status() == 0, "device error flag set during warm-up"
    # Listed cubes per query cube: K, or with a neighbourhood radius the mean
    # length of the lists the forward selected (the work the method does).
    cubes = None
    if args.radius >= 0:
        _, st0 = vsa.forward(dq_, dk_, dv_, wl.T, wl.H, wl.W, wl.topk, g_coarse=dgc_, g_fine=dgf_, out=out, ws=fws,
                             cube_order=order, radius=args.radius)
        cubes = float(st0.saved()["cnt"].float().mean())
    fl = step_flops(wl, cubes)
    vsa.timing_read()

    # ---- timed region: inputs resident in HBM
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    vsa.timing_enable(True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        e0.record(stream)
        for _ in range(args.steps):
            step(dq_, dk_, dv_, dgc_, dgf_, ddo)
        e1.record(stream)
        torch.cuda.synchronize()
    barrier()
    vsa.timing_enable(False)
    ms = e0.elapsed_time(e1)
    kern = vsa.timing_read()
    status = vsa.device_status()
    assert status == 0, f"device error flag {status}"
    ms = max_over_ranks(ms, world, dev)

    # ---- forward alone: vsa_forward (which also writes the state the
    # backward needs) and vsa_forward_inference (the fine stage reads the
    # native layout through 5-D TMA boxes; no reordered copies).  Reported
    # beside the headline; not part of it.
    fwd_only = None
    if world == 1 and not args.no_forward_only:
        iws = torch.empty(vsa.workspace_bytes(3, wl.B, wl.heads, wl.d, wl.T, wl.H, wl.W, wl.topk, args.radius),
                          dtype=torch.uint8, device=dev)
        runs = {
            "forward": lambda: vsa.forward(dq_, dk_, dv_, wl.T, wl.H, wl.W, wl.topk, g_coarse=dgc_, g_fine=dgf_,
                                           out=out, ws=fws, cube_order=order, radius=args.radius),
            "forward_inference": lambda: vsa.forward_inference(dq_, dk_, dv_, wl.T, wl.H, wl.W, wl.topk,
                                                               g_coarse=dgc_, g_fine=dgf_, out=out, ws=iws,
                                                               cube_order=order, radius=args.radius),
        }
        fwd_only = {}
        for name, fn in runs.items():
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(args.steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            fms = e0.elapsed_time(e1) / args.steps
            fwd_only[name] = {"ms": round(fms, 4),
                              "tflops": round((fl["fine_fwd"] + fl["coarse"] * 4 / 14) / (fms * 1e-3) / 1e12, 2)}
        assert vsa.device_status() == 0, "device error flag set in the forward-only runs"
        del iws

    # ---- the public single-stage calls, vsa_fine_fwd and vsa_fine_bwd with
    # their workspaces, on the layer's inputs in cube order and the lists the
    # forward selected; compared with the same kernels inside vsa_forward /
    # vsa_backward.  Reported beside the headline; not part of it.
    public = None
    if world == 1 and not args.no_forward_only:
        _, st = vsa.forward(dq_, dk_, dv_, wl.T, wl.H, wl.W, wl.topk, g_coarse=dgc_, g_fine=dgf_, out=out, ws=fws,
                            cube_order=order, radius=args.radius)
        sv = st.saved()
        lists = (sv["idx"], sv["cnt"])
        qp, kp, vp, dop = (vsa.permute(t, wl.T, wl.H, wl.W, cube_order=order).view(wl.BH, -1, wl.d)
                           for t in (dq_, dk_, dv_, ddo))
        fres = {}

        def pub_fwd():
            fres["of"], fres["lse"] = vsa.fine_fwd(qp, kp, vp, *lists)

        def pub_bwd():
            vsa.fine_bwd(qp, kp, vp, fres["of"], fres["lse"], dop, *lists)

        public = {}
        for name, fn in (("fine_fwd", pub_fwd), ("fine_bwd", pub_bwd)):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(args.steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            public[name] = {"ms": round(e0.elapsed_time(e1) / args.steps, 4)}
        assert vsa.device_status() == 0, "device error flag set in the public-call runs"
        del qp, kp, vp, dop, fres

    # ---- end to end through the public API with host buffers.  Every step
    # copies its six inputs from pinned host memory and its six results back;
    # the copies run on two copy streams, double-buffered, so that step i+1's
    # uploads and step i-1's downloads overlap step i's kernels.
    e2e = None
    if not args.no_e2e:
        with near_gpu_memory(local):
            host_out = [torch.empty(out.shape, dtype=torch.bfloat16).pin_memory() for _ in range(6)]
        dev_in = [[dq_, dk_, dv_, dgc_, dgf_, ddo], [torch.empty_like(dq_) for _ in range(6)]]
        res = [dict(out=out, **grads),
               dict(out=torch.empty_like(out), **{n: torch.empty_like(t) for n, t in grads.items()})]
        order_res = ["out", "dq", "dk", "dv", "dgc", "dgf"]
        h2d = sum(h.numel() * h.element_size() for h in host)
        d2h = sum(res[0][n].numel() * res[0][n].element_size() for n in order_res)
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        in_ready, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        up.wait_event(e0)
        down.wait_event(e0)
        for i in range(args.steps):
            b = i & 1
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(comp_done[b])          # step i-2 has finished reading these inputs
                for d, h in zip(dev_in[b], host):
                    d.copy_(h, non_blocking=True)
                in_ready[b].record(up)
            stream.wait_event(in_ready[b])
            if i >= 2:
                stream.wait_event(out_done[b])           # step i-2's results have been read out
            g = res[b]
            step(*dev_in[b], res_out=g["out"], res_grads={n: g[n] for n in order_res[1:]})
            comp_done[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(comp_done[b])
                for h, n in zip(host_out, order_res):
                    h.copy_(g[n], non_blocking=True)
                out_done[b].record(down)
        stream.wait_stream(up)
        stream.wait_stream(down)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ems = e0.elapsed_time(e1)
        ems = max_over_ranks(ems, world, dev)
        e2e = {"value": round(whole_job_tflops(world, fl["total"], args.steps, ems), 2), "unit": UNIT,
               "ms_per_step": round(ems / args.steps, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    configs = None
    if world == 1 and not args.no_configs:
        configs = measure_other_configs(vsa, dev, args, (dq_, dk_, dv_, dgc_, dgf_, ddo), order)

    if rank != 0:
        return
    peaks = load_peaks()
    csum = clocks.summary()
    peak, peak_kind = pick_peak(peaks, csum)
    value = whole_job_tflops(world, fl["total"], args.steps, ms)
    per_kernel = {n: round(t / max(c, 1), 4) for n, (t, c) in kern.items()}
    launches = {n: c for n, (t, c) in kern.items()}
    kflops = kernel_flops(wl, cubes)
    # The roofline is reported for the kernel with the most work per step.
    dominant = max(("fine_fwd", "fine_bwd_kv", "fine_bwd_dq"), key=lambda n: kflops[n])
    traffic = None  # DRAM bytes per launch from the committed ncu capture (profiles/traffic.txt)
    tpath = os.path.join(ROOT, "profiles", "traffic.txt")
    if os.path.exists(tpath) and args.config == WORKLOAD and args.curve == "raster":  # the captured case only
        with open(tpath) as f:
            for ln in f:
                parts = ln.split()
                if len(parts) == 2 and not ln.startswith("#") and parts[0] == dominant:
                    traffic = int(parts[1])
    bwd_ms, overlapped = fine_bwd_wall(per_kernel)
    dom = roof(kflops[dominant], per_kernel[dominant], peak)
    dq_roof = roof(kflops["fine_bwd_dq"], per_kernel["fine_bwd_dq"], peak)
    dq_eff = roof(kflops["dq_product"], per_kernel["fine_bwd_dq"], peak)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded smooth field + noise; Wan2.1 activations are not available)",
        "config": config_of(wl, "replicas" if world > 1 else "single GPU", args.curve, args.radius),
        "pct_of_peak": round(100 * value / world / peak, 2),
        "roofline": {"bound": "tensor", "kernel": dominant, "achieved": dom["tflops"], "peak": peak,
                     "unit": "TFLOP/s", "frac": dom["frac"], "traffic": traffic,
                     "peak_kind": peak_kind, "peak_burst": peaks["burst"], "peak_sustained": peaks["sustained"],
                     "frac_burst": round(dom["tflops"] / peaks["burst"], 4),
                     "frac_sustained": round(dom["tflops"] / peaks["sustained"], 4),
                     "peak_source": (peaks["source"] + f", dense bf16 {peak_kind} (fp16 has the same nominal rate); "
                                     "burst when the timed region held the maximum SM clock with no power cap"),
                     "flops_per_launch": kflops[dominant]},
        "fine_fwd": roof(kflops["fine_fwd"], per_kernel["fine_fwd"], peak),
        "fine_bwd_kv": roof(kflops["fine_bwd_kv"], per_kernel["fine_bwd_kv"], peak),
        "fine_bwd_dq": dict(dq_roof, effective_tflops=dq_eff["tflops"], effective_frac=dq_eff["frac"],
                            note=("interval on the caller's stream, beside fine_bwd_kv (shares the SMs of its last "
                                  "wave); effective = the dQ product alone, 2*N*64K*d per head"
                                  if overlapped else "effective = the dQ product alone, 2*N*64K*d per head")),
        "fine_bwd_effective": {"ms": round(bwd_ms, 4),
                               "tflops": round(fl["fine_bwd"] / (bwd_ms * 1e-3) / 1e12, 2),
                               "frac": round(fl["fine_bwd"] / (bwd_ms * 1e-3) / 1e12 / peak, 4)},
        "kernel_ms_per_step": per_kernel,
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "kernel_launches_timed": launches,
        "forward_only": fwd_only,
        "public_calls": public_calls(public, per_kernel, bwd_ms, overlapped),
        "clocks": csum,
        "e2e": e2e,
    }
    if configs is not None:
        for c in configs.get("runs", {}).values():
            if "per_kernel" in c:
                pk = c.pop("per_kernel")
                cf = c.pop("kflops")
                c["fine_fwd_frac"] = roof(cf["fine_fwd"], pk["fine_fwd"], peak)["frac"]
                c["fine_bwd_kv_frac"] = roof(cf["fine_bwd_kv"], pk["fine_bwd_kv"], peak)["frac"]
                c["pct_of_peak"] = round(100 * c["tflops"] / peak, 2)
        line["configs"] = configs
    if not args.no_cpu_baseline and world == 1:
        flops, dt, rows, threads = oracle_sample(wl, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": (f"head 0 of {wl.heads}: coarse stage in full, fine forward and fine backward (dQ) of "
                       f"{rows} random query rows; {dt:.1f} s; FLOPs counted per row 10*64K*d")}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.config]
    budget = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    _, _, rows, threads = oracle_sample(wl, budget)
    for _ in range(args.warmup):
        oracle_sample(wl, budget, rows_hint=rows)
    tot_f, tot_t = 0.0, 0.0
    for _ in range(args.steps):
        f, t, _, _ = oracle_sample(wl, budget, rows_hint=rows)
        tot_f += f
        tot_t += t
    value = tot_f / tot_t / 1e12
    sample = (f"per step: head 0 of {wl.heads}, coarse stage in full + fine forward and backward (dQ) of {rows} "
              f"query rows on the CPU oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot_t / args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded smooth field + noise)", "config": config_of(wl, "single process, host cores"),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-forward-only", action="store_true", help="skip the forward-only timings")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other workloads (sparsity sweep, Wan-14B layer, long video)")
    ap.add_argument("--config-steps", type=int, default=5, help="timed steps per other workload")
    ap.add_argument("--config-cpu-seconds", type=float, default=3.0, help="oracle sample per other workload")
    ap.add_argument("--curve", choices=["raster", "hilbert"], default="raster",
                    help="cube order of the space-filling-curve reordering")
    ap.add_argument("--radius", type=int, default=-1,
                    help="unite each Top-K list with the radius-r cube neighbourhood (-1: Top-K alone)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
