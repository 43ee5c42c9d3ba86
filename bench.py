#!/usr/bin/env python
"""Benchmark of the flexible-mask attention hot path on GB300.

One step = the whole path on one batch: the slice planner, the forward
(out, lse) and the backward (dq, dk, dv), on the 64K-token heterogeneous
mask (a shared 4096-token prefix plus 23 documents of mixed mask types,
47 slices, 16 heads, head_dim 128, bf16).  The metric is effective TFLOPS
over the unmasked area: forward 4*D*area*Hq, backward 2.5x that.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ffa|reference]

Under torchrun every rank runs its own replica of the workload (the path
has no cross-GPU exchange), ranks meet at a barrier around the timed loop,
and rank 0 prints one JSON line with the max time over ranks.
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective TFLOPS (unmasked area) fwd/bwd on 1 GB300; % of BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ffa", "reference"], default="ffa")
    ap.add_argument("--config", default="heterogeneous")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling runs)")
    ap.add_argument("--sink", type=int, default=0,
                    help="attention-sink logits per query head (seeded fp32 [n, Hq]); 0 = none")
    ap.add_argument("--softcap", type=float, default=0.0, help="score cap c (0 = none)")
    return ap.parse_args()


def dist_setup(use_cuda: bool):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend="nccl" if use_cuda else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.skip = 0  # samples taken before the timed region

    def _lines(self) -> int:
        try:
            with open(self.path) as fh:
                return sum(1 for _ in fh)
        except OSError:
            return 0

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # nvidia-smi takes a while to start: wait for its first sample, then
        # count only the samples taken from here on (the timed region)
        import time
        t0 = time.monotonic()
        while self._lines() == 0 and time.monotonic() - t0 < 3.0 and self.proc.poll() is None:
            time.sleep(0.01)
        self.skip = self._lines()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        lines = open(self.path).read().splitlines()
        if len(lines) > self.skip:  # else keep the last sample before the region
            lines = lines[self.skip:]
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons, "samples": len(rows)}


def kernel_source_hash() -> str:
    """Hash of the CUDA sources with comments and blank lines removed, so
    that a capture stays matched to its kernels across comment edits."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "flexible_mask_attention_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(f.encode() + code.encode())
    return h.hexdigest()[:16]


def traffic_from_profile(kernel: str):
    """DRAM bytes per launch recorded by an ncu capture of the current kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash()
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and parts[0] == kernel and parts[1] == want:
            return float(parts[2])
    return None


def row_counts(wl):
    """Visible keys of every query row (one head), from the slice table."""
    import numpy as np

    from oracle import planner
    counts = np.zeros(wl.total_q, dtype=np.int64)
    qr, kr, ty = (np.asarray(a, dtype=np.int64) for a in (wl.q_ranges, wl.k_ranges,
                                                          wl.mask_types))
    full = (ty == 0) & (qr[:, 1] > qr[:, 0]) & (kr[:, 1] > kr[:, 0])
    diff = np.zeros(wl.total_q + 1, dtype=np.int64)  # full slices: one add per range end
    np.add.at(diff, qr[full, 0], kr[full, 1] - kr[full, 0])
    np.add.at(diff, qr[full, 1], -(kr[full, 1] - kr[full, 0]))
    counts += np.cumsum(diff)[:-1]
    for (qs, qe), (ks, ke), t in zip(qr[~full], kr[~full], ty[~full]):
        if qe > qs and ke > ks:
            rows, lo, hi = planner.row_intervals(int(qs), int(qe), int(ks), int(ke), int(t))
            counts[rows] += np.clip(hi - lo, 0, None)
    return counts


# Metric credit of the oracle legs the CPU baseline runs, per visible (q, k,
# head) in units of D: the forward's two products (4) and, of the backward's
# five, the dQ product (2).  The oracle's dK/dV leg is not run (it would
# recompute every row's lse for each sampled key), so it is not credited.
ORACLE_CREDIT = 6.0


def oracle_sample(wl, q, k, v, do, seconds: float, seed: int = 0):
    """Time the fp64 oracle on a seeded row sample: forward (out, lse) and dq
    of those rows, credited 4*D + 2*D per visible pair and head (the work it
    ran, in the metric's units)."""
    import numpy as np

    import oracle
    rng = np.random.default_rng(seed)
    D, Hq = wl.head_dim, wl.num_heads_q
    counts = row_counts(wl)
    # calibrate on a small sample, then size the real one
    probe = rng.choice(wl.total_q, 8, replace=False)
    t0 = time.perf_counter()
    oracle.fwd(q, k, v, wl.q_ranges, wl.k_ranges, wl.mask_types, rows=probe)
    oracle.bwd(q, k, v, do, wl.q_ranges, wl.k_ranges, wl.mask_types, dq_rows=probe, dkv_keys=[])
    dt = max(time.perf_counter() - t0, 1e-4)
    per_pair = dt / max(1, counts[probe].sum())
    n = int(np.clip(seconds / max(per_pair * counts.mean(), 1e-9), 8, wl.total_q))
    rows = np.sort(rng.choice(wl.total_q, n, replace=False))
    t0 = time.perf_counter()
    oracle.fwd(q, k, v, wl.q_ranges, wl.k_ranges, wl.mask_types, rows=rows)
    oracle.bwd(q, k, v, do, wl.q_ranges, wl.k_ranges, wl.mask_types, dq_rows=rows, dkv_keys=[])
    t = time.perf_counter() - t0
    flops = ORACLE_CREDIT * D * Hq * float(counts[rows].sum())
    return {"value": flops / t / 1e12, "unit": "TFLOPS", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": (f"{n} seeded query rows of {wl.total_q} x all {Hq} heads: fp64 forward "
                       f"and dq of those rows, credited 6*D per visible pair and head (fwd 4*D "
                       f"+ the dQ product 2*D; dK/dV not run, not credited); "
                       f"{t:.1f} s on the host")}, t


# GB300 L2 (129 MB); a workload whose step inputs (q, k, v, dout) fit in twice
# that is timed with L2 flushed between steps (FLUSH_BYTES written).
L2_BYTES = 129e6
FLUSH_BYTES = 512 << 20


def input_bytes(wl) -> int:
    return 2 * wl.head_dim * 2 * (wl.total_q * wl.num_heads_q + wl.total_k * wl.num_heads_kv)


def needs_flush(wl) -> bool:
    return input_bytes(wl) < 2 * L2_BYTES


def workload_config(args, wl, area, world):
    """The `config` object of the JSON line (identical for both arms)."""
    Tq, Hq, Hkv, D = wl.total_q, wl.num_heads_q, wl.num_heads_kv, wl.head_dim
    sizes = (f"q and dout {Tq * Hq * D * 2 / 1e6:.0f} MB each, "
             f"k and v {wl.total_k * Hkv * D * 2 / 1e6:.0f} MB each")
    l2 = (f"L2 flushed between timed steps ({FLUSH_BYTES >> 20} MB written, outside the "
          f"timed steps): inputs {sizes}" if needs_flush(wl)
          else f"inputs larger than L2: {sizes}, no flush")
    return {"workload": wl.name, "slices": wl.num_slices, "tokens": Tq,
            "heads_q": Hq, "heads_kv": Hkv, "head_dim": D,
            "sink": args.sink, "softcap": args.softcap,
            "visible_pairs_per_head": int(area), "parallelism": f"replicas x{world}",
            "l2": l2}


def run_reference(args, wl, world, rank):
    """The oracle as the reference arm: each step a bounded CPU sample."""
    import torch
    if rank != 0:
        return
    q, k, v, do = __import__("flexible_mask_attention_gb300.workloads",
                             fromlist=["x"]).make_tensors(wl, with_dout=True)
    per_step = max(1.0, min(args.cpu_seconds, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(wl, q, k, v, do, per_step / 4, seed=1)
    vals, total_t = [], 0.0
    last = None
    for s in range(args.steps):
        last, t = oracle_sample(wl, q, k, v, do, per_step, seed=100 + s)
        vals.append(last["value"])
        total_t += t
    value = statistics.mean(vals)
    line = {"metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": workload_config(args, wl, int(row_counts(wl).sum()), world),
            "cpu_baseline": dict(last, value=value),
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ffa(args, wl, world, rank, local):
    import numpy as np
    import torch

    import flexible_mask_attention_gb300 as ffa
    from flexible_mask_attention_gb300 import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q, k, v, do = W.make_tensors(wl, with_dout=True)
    host = [t.pin_memory() for t in (q, k, v, do)]
    qd, kd, vd, dod = (t.to(dev) for t in host)
    qr = torch.as_tensor(wl.q_ranges, dtype=torch.int32)
    kr = torch.as_tensor(wl.k_ranges, dtype=torch.int32)
    ty = torch.as_tensor(wl.mask_types, dtype=torch.int32)
    qr_d, kr_d, ty_d = qr.to(dev), kr.to(dev), ty.to(dev)
    Tq, Tk, Hq, Hkv, D = wl.total_q, wl.total_k, wl.num_heads_q, wl.num_heads_kv, wl.head_dim
    out = torch.empty_like(qd)
    lse = torch.empty(Hq, Tq, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    plan0 = ffa.ffa_plan_create(qr_d, kr_d, ty_d, Tq, Tk, Hq, Hkv, D)
    info = ffa.ffa_plan_info(plan0)
    ws_f = torch.empty(max(16, ffa.ffa_fwd_workspace_size(plan0)), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(max(16, ffa.ffa_bwd_workspace_size(plan0)), dtype=torch.uint8, device=dev)
    plan0.destroy()
    area = info["area"]
    sink = dsink = None
    if args.sink > 0:
        g = torch.Generator().manual_seed(wl.seed + 1000)
        sink = (2.0 * torch.randn(args.sink, Hq, generator=g)).float().to(dev)
        dsink = torch.empty_like(sink)
    extended = sink is not None or args.softcap > 0
    f_fwd = 4.0 * D * area * Hq
    f_bwd = 2.5 * f_fwd
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    def step(qa, ka, va, doa, record=None, outs=None, after_plan=None):
        # outs: (out, lse, dq, dk, dv) to write; after_plan: called between the
        # plan and the forward (the planner reads only the slice table).
        o_, l_, dq_, dk_, dv_ = outs if outs is not None else (out, lse, dq, dk, dv)
        if record is not None:
            record[0].record(stream)
        plan = ffa.ffa_plan_create(qr_d, kr_d, ty_d, Tq, Tk, Hq, Hkv, D)
        if record is not None:
            ffa.ffa_plan_set_events(plan, record[4:10])
            record[1].record(stream)
        if after_plan is not None:
            after_plan()
        if extended:
            ffa.ffa_fwd_ex(plan, qa, ka, va, sink=sink, out=o_, lse=l_, softcap=args.softcap,
                           workspace=ws_f)
        else:
            ffa.ffa_fwd(plan, qa, ka, va, out=o_, lse=l_, workspace=ws_f)
        if record is not None:
            record[2].record(stream)
        if extended:
            ffa.ffa_bwd_ex(plan, qa, ka, va, o_, doa, l_, sink=sink, dq=dq_, dk=dk_, dv=dv_,
                           dsink=dsink, softcap=args.softcap, workspace=ws_b)
        else:
            ffa.ffa_bwd(plan, qa, ka, va, o_, doa, l_, dq=dq_, dk=dk_, dv=dv_, workspace=ws_b)
        if record is not None:
            record[3].record(stream)
        return plan

    for _ in range(args.warmup):
        step(qd, kd, vd, dod).destroy()
    torch.cuda.synchronize()
    # correctness guard: no device error, finite results
    p = step(qd, kd, vd, dod)
    torch.cuda.synchronize()
    err = ffa.ffa_get_last_device_error(p)
    p.destroy()
    if err != (0, 0):
        raise RuntimeError(f"device error {err}")

    sampler = ClockSampler(local)
    launches0 = ffa.ffa_kernel_launch_count()
    t_plan, t_fwd, t_bwd = [], [], []
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if needs_flush(wl) else None
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    plans = []
    for _ in range(args.steps):
        if flush is not None:  # outside the step's events; the steps' own times are summed
            flush.zero_()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(10)]
        plans.append((step(qd, kd, vd, dod, evs), evs))
    end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier(world)
    launches = ffa.ffa_kernel_launch_count() - launches0
    elapsed_ms = start.elapsed_time(end)
    if flush is not None:
        elapsed_ms = sum(evs[0].elapsed_time(evs[3]) for _, evs in plans)
        del flush
    t_kern = {"ffa_fwd_kernel": [], "ffa_bwd_pre_kernel": [], "ffa_bwd_dkdv_kernel": [],
              "ffa_bwd_dq_kernel": []}
    for pl, evs in plans:
        t_plan.append(evs[0].elapsed_time(evs[1]))
        t_fwd.append(evs[1].elapsed_time(evs[2]))
        t_bwd.append(evs[2].elapsed_time(evs[3]))
        t_kern["ffa_fwd_kernel"].append(evs[4].elapsed_time(evs[5]))
        t_kern["ffa_bwd_pre_kernel"].append(evs[6].elapsed_time(evs[7]))
        t_kern["ffa_bwd_dkdv_kernel"].append(evs[7].elapsed_time(evs[8]))
        t_kern["ffa_bwd_dq_kernel"].append(evs[8].elapsed_time(evs[9]))
        pl.destroy()
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, world, dev, stream, step, host, out, lse, dq, dk, dv, qr,
                      f_fwd + f_bwd)
    peaks, peak_src = load_peaks()
    return finish(args, wl, world, rank, elapsed_ms, t_plan, t_fwd, t_bwd, f_fwd, f_bwd, area,
                  launches, clocks, e2e, peaks, peak_src, q, k, v, do, t_kern)


def run_e2e(args, world, dev, stream, step, host, out, lse, dq, dk, dv, qr, flops):
    """Steps through the public API from pinned host buffers, as a serving loop
    runs them: each step's inputs are copied host -> device and its results
    (out, lse, dq, dk, dv) device -> host, on one copy stream per direction,
    double-buffered so that step s+1's inputs and step s-1's results move
    while step s computes.  The timed region runs from before the first input
    copy to after the last result copy, on the compute stream."""
    import torch
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    din = [[torch.empty_like(t, device=dev) for t in host] for _ in range(2)]
    dres = [tuple(torch.empty_like(t) for t in (out, lse, dq, dk, dv)) for _ in range(2)]
    hres = [tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dres[0])
            for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host) + 3 * qr.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in hres[0])

    def pipeline(n):
        """n steps through the double-buffered pipeline; returns the device
        time from before the first input copy to after the last result copy."""
        ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(n)] for _ in range(3))
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_s.wait_event(e0)
        plans = []  # freed after the timed region: cudaFree would synchronize the device
        for s_ in range(n):
            p = s_ % 2
            with torch.cuda.stream(h2d_s):  # inputs of step s (buffer free once step s-2 computed)
                if s_ >= 2:
                    h2d_s.wait_event(ev_comp[s_ - 2])
                for d_, h_ in zip(din[p], host):
                    d_.copy_(h_, non_blocking=True)
                ev_in[s_].record(h2d_s)

            def inputs_ready(s_=s_):
                stream.wait_event(ev_in[s_])
                if s_ >= 2:  # results of step s-2 copied out of this buffer
                    stream.wait_event(ev_out[s_ - 2])

            pl = step(*din[p], outs=dres[p], after_plan=inputs_ready)
            ev_comp[s_].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_comp[s_])
                for h_, d_ in zip(hres[p], dres[p]):
                    h_.copy_(d_, non_blocking=True)
                ev_out[s_].record(d2h_s)
            plans.append(pl)
        stream.wait_event(ev_out[n - 1])
        e1.record(stream)
        torch.cuda.synchronize()
        for pl in plans:
            pl.destroy()
        return e0.elapsed_time(e1)

    pipeline(max(args.warmup, 2))  # untimed: first use of the streams, buffers and events
    n = args.steps
    ms = pipeline(n)
    e2e_ms = max_over_ranks(ms, world, dev)
    e2e_value = world * n * flops / (e2e_ms / 1e3) / 1e12
    return {"value": e2e_value, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "note": "pinned host buffers, one copy stream per direction, double-buffered"}


# FLOP credited to each tensor-core kernel per visible (q, k, head), in units
# of D: the forward's two products; of the backward's five (S, dP, dV, dK, dQ)
# the dK/dV pass computes four and the dQ pass one (it also recomputes S and
# dP, which is not credited).
KERNEL_CREDIT = {"ffa_fwd_kernel": 4.0, "ffa_bwd_dkdv_kernel": 8.0, "ffa_bwd_dq_kernel": 2.0}


def finish(args, wl, world, rank, elapsed_ms, t_plan, t_fwd, t_bwd, f_fwd, f_bwd, area,
           launches, clocks, e2e, peaks, peak_src, q, k, v, do, t_kern):
    Tq, Hq, Hkv, D = wl.total_q, wl.num_heads_q, wl.num_heads_kv, wl.head_dim
    ms_step = elapsed_ms / args.steps
    value = world * args.steps * (f_fwd + f_bwd) / (elapsed_ms / 1e3) / 1e12
    fwd_ms, bwd_ms, plan_ms = (statistics.mean(x) for x in (t_fwd, t_bwd, t_plan))
    kern_ms = {k: statistics.mean(v) for k, v in t_kern.items()}
    dom = max(KERNEL_CREDIT, key=lambda k: kern_ms[k])
    dom_flops = KERNEL_CREDIT[dom] * D * area * Hq
    achieved = dom_flops / (kern_ms[dom] / 1e3) / 1e12
    # The burst peak applies to a kernel timed in a loop shorter than the few
    # seconds it takes the power cap to settle; the sustained one to longer loops.
    timed_s = elapsed_ms / 1e3
    peak_kind = "bf16_tflops_sustained" if timed_s >= 3.0 else "bf16_tflops"
    peak = peaks[peak_kind]
    traffic = traffic_from_profile(dom)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic, "kernel": dom,
                "kernel_ms": kern_ms[dom],
                "credited_flop_per_visible_pair_head": f"{KERNEL_CREDIT[dom]:.0f}*D",
                "peak_source": f"{peak_src} {peak_kind} (timed loop {timed_s:.2f} s)",
                "frac_of_burst_peak": achieved / peaks["bf16_tflops"],
                "frac_of_sustained_peak": achieved / peaks["bf16_tflops_sustained"]}
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(args, wl, area, world),
        "phases_ms": {"plan": plan_ms, "fwd": fwd_ms, "bwd": bwd_ms},
        "kernels_ms": kern_ms,
        "fwd_tflops": f_fwd / (fwd_ms / 1e3) / 1e12,
        "bwd_tflops": f_bwd / (bwd_ms / 1e3) / 1e12,
        "fwd_frac_of_peak": f_fwd / (fwd_ms / 1e3) / 1e12 / peak,
        "bwd_frac_of_peak": f_bwd / (bwd_ms / 1e3) / 1e12 / peak,
        "peak_used": peak_kind,
        "fwd_frac_of_burst": f_fwd / (fwd_ms / 1e3) / 1e12 / peaks["bf16_tflops"],
        "bwd_frac_of_burst": f_bwd / (bwd_ms / 1e3) / 1e12 / peaks["bf16_tflops"],
        "fwd_frac_of_sustained": f_fwd / (fwd_ms / 1e3) / 1e12 / peaks["bf16_tflops_sustained"],
        "bwd_frac_of_sustained": f_bwd / (bwd_ms / 1e3) / 1e12 / peaks["bf16_tflops_sustained"],
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"], _ = oracle_sample(wl, q, k, v, do, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    from flexible_mask_attention_gb300 import workloads as W
    wl = W.CONFIGS[args.config]()
    if args.impl == "reference":
        world, rank, _ = dist_setup(use_cuda=False)
        run_reference(args, wl, world, rank)
    else:
        world, rank, local = dist_setup(use_cuda=True)
        run_ffa(args, wl, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
