#!/usr/bin/env python
"""GDPA forward + backward throughput on GB300 (useful TFLOP/s).

One step = the whole hot path over one batch of synthetic input, through the
C-ABI: gdpa_fwd (work list, forward kernel) then gdpa_bwd (work list and dQ
clear in one launch, backward kernel, dQ convert). The workload is the jagged
self-attention scenario of the gdpa/README.md page's benchmark section
("Self Attention, sparsity=0.5"): B=64 sequences with lengths uniform in
[1, 2048], 4 heads, head dim 128, bf16, GELU, non-causal.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdpa|reference]

N > 1 runs under torchrun as independent replicas (one per GPU, same
workload, no collective on the data path); the JSON line reports the
aggregate over all ranks. `--impl reference` times the float64 CPU oracle on
a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import glob
import json
import math
import os
import random
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# More hardware work queues than CUDA's default 8, so that the end-to-end
# leg's two copy streams (host->device, device->host) and the compute stream
# are less likely to share one queue and serialise behind each other. Read at
# CUDA initialisation, so it has to be set before torch touches the GPU; a
# value already in the environment wins.
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")

import torch  # noqa: E402

METRIC = "GDPA fwd & bwd TFLOP/s (useful, jagged) and % of GB300 dense tensor-core peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gdpa", "reference"], default="gdpa")
    ap.add_argument("--workload", default="jagged_self")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_sources_digest(kernel: str) -> str:
    """Short hash of the sources a main kernel is built from: its own files
    (fwd* or bwd*) and the shared headers. Ties recorded ncu counters to them."""
    own = "fwd" if "fwd" in kernel else "bwd"
    h = hashlib.sha1()
    for p in sorted(glob.glob(os.path.join(ROOT, "generalized_attention_recsys_gb300", "csrc", "*"))):
        name = os.path.basename(p)
        if not os.path.isfile(p) or not name.endswith((".cu", ".cuh", ".h")):
            continue
        if name.startswith(("fwd", "bwd")) and not name.startswith(own):
            continue
        if name == "api.cu":
            continue
        with open(p, "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:12]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (matching digest); else None."""
    digest = kernel_sources_digest(kernel)
    for p in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        with open(p) as f:
            for line in f:
                m = re.match(r"\s*traffic:\s*kernel=(\S+)\s+workload=(\S+)\s+bytes_per_launch=(\d+)\s+csrc=(\w+)",
                             line)
                if m and m.group(1) == kernel and m.group(2) == workload and m.group(4) == digest:
                    return int(m.group(3))
    return None


# ---------------------------------------------------------------- cross-rank aggregation (replicas)

def reduce_max(value: float, dist=None, device=None) -> float:
    """Max of a per-rank value over all ranks (the slowest replica sets the time)."""
    t = torch.tensor([value], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(flops_per_step: float, steps: int, world: int, slowest_ms: float) -> float:
    """Whole-job TFLOP/s: every replica runs `steps` steps of the same workload."""
    return flops_per_step * steps * world / (slowest_ms * 1e-3) / 1e12


# ---------------------------------------------------------------- clocks during the timed region

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines: list[str] = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()
        time.sleep(0.6)  # first samples before the timed region opens

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which: str):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        for ts, line in self.lines:
            if self.t0 is not None and not (self.t0 - 0.15 <= ts <= self.t1 + 0.15):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle sample

def oracle_sample(inp, budget_s: float, seed: int = 0):
    """Times the float64 oracle (forward + backward) on (sequence, head) units
    in seeded random order until the time budget is used; returns
    (useful TFLOP/s, units done, total units, seconds, threads)."""
    import oracle  # test infrastructure: timed here as the CPU baseline only
    from generalized_attention_recsys_gb300 import flops

    wl = inp.wl
    q, k, v, do = inp.values("q"), inp.values("k"), inp.values("v"), inp.dout.double()
    cu_q, cu_k = inp.cu_seqlens_q, inp.cu_seqlens_k
    units = [(b, h) for b in range(wl.batch) for h in range(wl.h_q)]
    random.Random(seed).shuffle(units)
    done, fl, t_used = 0, 0.0, 0.0
    for b, h in units:
        lq, lk = int(inp.lengths_q[b]), int(inp.lengths_k[b])
        t0 = time.perf_counter()
        oracle.gdpa_fwd(q, k, v, cu_q, cu_k, wl.batch, wl.max_q, wl.max_k, wl.act, wl.softmax_scale,
                        wl.causal, wl.window, units=[(b, h)])
        oracle.gdpa_bwd(q, k, v, do, cu_q, cu_k, wl.batch, wl.max_q, wl.max_k, wl.act, wl.softmax_scale,
                        wl.causal, wl.window, units=[(b, h)])
        t_used += time.perf_counter() - t0
        f = 2.0 * flops.allowed_pairs([lq], [lk], wl.causal, wl.window) * (wl.d_qk + wl.d_v)
        fl += 3.5 * f
        done += 1
        if t_used >= budget_s:
            break
    return fl / t_used / 1e12, done, len(units), t_used, torch.get_num_threads()


def run_reference(args, wl):
    """Reference arm: the float64 CPU oracle on a bounded sample per step."""
    from generalized_attention_recsys_gb300 import flops, inputs

    inp = inputs.make_inputs(wl, seed=args.seed)
    q, k, v = inp.values("q"), inp.values("k"), inp.values("v")
    do = inp.dout.double() if inp.dout is not None else None
    import oracle

    units = [(b, h) for b in range(wl.batch) for h in range(wl.h_q)]
    random.Random(args.seed).shuffle(units)
    # a fixed sample per step of about 0.5-1 s of CPU work (two mid-length units)
    step_units = units[:2]
    fl = sum((1.0 if do is None else 3.5) * 2.0 *
             flops.allowed_pairs([int(inp.lengths_q[b])], [int(inp.lengths_k[b])], wl.causal, wl.window) *
             (wl.d_qk + wl.d_v) for b, _ in step_units)

    def step():
        oracle.gdpa_fwd(q, k, v, inp.cu_seqlens_q, inp.cu_seqlens_k, wl.batch, wl.max_q, wl.max_k, wl.act,
                        wl.softmax_scale, wl.causal, wl.window, units=step_units)
        if do is not None:
            oracle.gdpa_bwd(q, k, v, do, inp.cu_seqlens_q, inp.cu_seqlens_k, wl.batch, wl.max_q, wl.max_k, wl.act,
                            wl.softmax_scale, wl.causal, wl.window, units=step_units)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = fl * args.steps / dt / 1e12
    sample = (f"{len(step_units)} of {len(units)} (sequence, head) units per step (lengths "
              f"{[int(inp.lengths_q[b]) for b, _ in step_units]}), float64 forward"
              f"{'' if do is None else ' + backward'}")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name + ": " + wl.notes, "useful_flops_per_step": fl},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": torch.get_num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

def main():
    args = parse_args()
    from generalized_attention_recsys_gb300 import inputs

    wl = inputs.WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, wl)
        return

    import __graft_entry__

    __graft_entry__.build()
    from generalized_attention_recsys_gb300 import _lib, flops

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def barrier():
        if dist is not None:
            dist.barrier()

    inp = inputs.make_inputs(wl, seed=args.seed)
    f_fwd, f_bwd = flops.useful_flops(inp)
    fwd_only = wl.fwd_only  # forward-only workloads (FP8, and the softmax cross-check at the same shapes)
    if fwd_only:
        f_bwd = 0.0
    dev = torch.device("cuda", local_rank)
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    do = inp.dout.to(dev) if inp.dout is not None else None
    cu_q, cu_k = inp.cu_seqlens_q.to(dev), inp.cu_seqlens_k.to(dev)
    mq, mk = inp.max_q, inp.max_k
    desc = torch.tensor(inp.descale, dtype=torch.float32, device=dev) if inp.descale is not None else None
    mxs = tuple(t.to(dev) for t in inp.mx) if inp.mx is not None else None  # MXFP8 block scales of q, k, v
    out_dtype = torch.bfloat16 if wl.dtype in ("e4m3", "mxe4m3") else q.dtype
    out = torch.empty(q.shape[0], q.shape[1], v.shape[2], dtype=out_dtype, device=dev)
    lse = torch.empty(q.shape[1], q.shape[0], dtype=torch.float32, device=dev) if wl.act == "softmax" else None
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    shape = _lib.make_shape(q, k, v, wl.batch)
    # the MXFP8 forward also stages its scale atoms in the workspace
    ws_f = torch.empty(_lib.gdpa_workspace_bytes(shape, mq, mk, 3 if mxs is not None else 0), dtype=torch.uint8,
                       device=dev)
    ws_b = torch.empty(_lib.gdpa_workspace_bytes(shape, mq, mk, True), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    a = (wl.act, wl.softmax_scale, wl.causal, wl.window)

    def fwd_call(qq, kk, vv, cq, ck, o, l, sc):
        if sc is not None:
            _lib.gdpa_fwd_mxfp8(qq, kk, vv, *sc, cq, ck, mq, mk, *a, out=o, lse=l, batch=wl.batch, workspace=ws_f)
        else:
            _lib.gdpa_fwd(qq, kk, vv, cq, ck, mq, mk, *a, descale_qkv=desc, out=o, lse=l, batch=wl.batch,
                          workspace=ws_f)

    def step(qq=q, kk=k, vv=v, dd=do, cq=cu_q, ck=cu_k, ev=None, o=None):
        o = out if o is None else o
        if ev is not None:
            _lib.gdpa_set_profile_events(ev[0], ev[1])
        fwd_call(qq, kk, vv, cq, ck, o, lse, mxs)
        if not fwd_only:
            if ev is not None:
                _lib.gdpa_set_profile_events(ev[2], ev[3])
            _lib.gdpa_bwd(qq, kk, vv, cq, ck, mq, mk, *a, o, lse, dd, dq=dq, dk=dk, dv=dv, batch=wl.batch,
                          workspace=ws_b)
        if ev is not None:
            _lib.gdpa_set_profile_events(None, None)

    for _ in range(max(args.warmup, 3)):
        step()
    if _lib.gdpa_get_status() != 0:
        raise RuntimeError("device status not ok after warm-up")

    K = args.steps
    mk_ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev_step = [(mk_ev(), mk_ev()) for _ in range(K)]
    ev_main = [tuple(mk_ev() for _ in range(4)) for _ in range(K)]
    for e in ev_main:
        for x in e:
            x.record()  # create the CUDA events before the timed region
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t0")
    for i in range(K):
        flush.zero_()  # L2 flush between timed steps, outside the step's events
        ev_step[i][0].record()
        step(ev=ev_main[i])
        ev_step[i][1].record()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t1")
    barrier()
    clocks = sampler.stop() if sampler else None
    if _lib.gdpa_get_status() != 0:
        raise RuntimeError("device status not ok after the timed steps")

    step_ms = sum(s.elapsed_time(e) for s, e in ev_step)
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in ev_main) / K
    bwd_ms = sum(e[2].elapsed_time(e[3]) for e in ev_main) / K if not fwd_only else 0.0
    step_ms_max = reduce_max(step_ms, dist, dev)
    value = replica_throughput(f_fwd + f_bwd, K, world, step_ms_max)

    # ---- end to end through the C-ABI with host buffers (pinned), copies inside the timed region.
    # Pipelined as a host-buffer caller would run it: step i+1's inputs are copied in on one copy
    # stream and step i-1's results copied out on another while step i's kernels run; device
    # buffers are double-buffered. The timed region spans all steps with all of their copies.
    e2e = None
    if not args.no_e2e:
        # inputs q, k, v, (dO), cu_seqlens; results out, (lse), (dq, dk, dv)
        ins = ([inp.q, inp.k, inp.v] + ([inp.dout] if not fwd_only else []) + [inp.cu_seqlens_q, inp.cu_seqlens_k] +
               (list(inp.mx) if inp.mx is not None else []))
        n_mx = 3 if inp.mx is not None else 0
        host_in = [t.pin_memory() for t in ins]
        dev_in = [[torch.empty_like(t, device=dev) for t in host_in] for _ in range(2)]
        res = [out] + ([lse] if lse is not None else []) + ([dq, dk, dv] if not fwd_only else [])
        dev_out = [[torch.empty_like(t) for t in res] for _ in range(2)]
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in res]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        comp = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_ready, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

        def e2e_steps(n):
            for e in comp_done + out_done:
                e.record(comp)
            for i in range(n):
                b = i % 2
                s_in.wait_event(comp_done[b])  # step i-2 finished reading these inputs
                with torch.cuda.stream(s_in):
                    for hsrc, ddst in zip(host_in, dev_in[b]):
                        ddst.copy_(hsrc, non_blocking=True)
                in_ready[b].record(s_in)
                comp.wait_event(in_ready[b])
                comp.wait_event(out_done[b])  # step i-2's results have left these buffers
                qq, kk, vv = dev_in[b][:3]
                dd = dev_in[b][3] if not fwd_only else None
                nin = len(dev_in[b]) - n_mx
                cq, ck = dev_in[b][nin - 2:nin]
                r = dev_out[b]
                o_, l_ = r[0], (r[1] if lse is not None else None)
                fwd_call(qq, kk, vv, cq, ck, o_, l_, tuple(dev_in[b][nin:]) if n_mx else None)
                if not fwd_only:
                    dq_, dk_, dv_ = r[-3:]
                    _lib.gdpa_bwd(qq, kk, vv, cq, ck, mq, mk, *a, o_, l_, dd, dq=dq_, dk=dk_, dv=dv_,
                                  batch=wl.batch, workspace=ws_b)
                comp_done[b].record(comp)
                s_out.wait_event(comp_done[b])
                with torch.cuda.stream(s_out):
                    for dsrc, hdst in zip(dev_out[b], host_out):
                        hdst.copy_(dsrc, non_blocking=True)
                out_done[b].record(s_out)
            comp.wait_stream(s_out)
            comp.wait_stream(s_in)

        e2e_steps(max(args.warmup, 3))
        ke = max(K // 2, 20)  # enough steps to average out copy-overlap variance
        e0, e1 = mk_ev(), mk_ev()
        barrier()
        torch.cuda.synchronize()
        e0.record(comp)
        e2e_steps(ke)
        e1.record(comp)
        torch.cuda.synchronize()
        barrier()
        e_ms = reduce_max(e0.elapsed_time(e1), dist, dev)
        e2e = {"value": replica_throughput(f_fwd + f_bwd, ke, world, e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": ke,
               "pipeline": "double-buffered: H2D of step i+1 and D2H of step i-1 overlap step i's kernels"}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    peak_label = f"{peak_src} bf16 dense (burst)"
    if wl.dtype in ("e4m3", "mxe4m3"):  # the contraction's dtype: measured bf16 x the nominal e4m3 / bf16 ratio (4.5 / 2.25)
        peak *= 2.0
        peak_label = f"{peak_src} bf16 dense (burst) x 2, the nominal e4m3 / bf16 ratio"
    fwd_tflops = f_fwd / (fwd_ms * 1e-3) / 1e12
    bwd_tflops = f_bwd / (bwd_ms * 1e-3) / 1e12 if not fwd_only else None
    dominant = "gdpa_bwd_kernel" if bwd_ms >= fwd_ms else "gdpa_fwd_kernel"
    dom_flops, dom_ms = (f_bwd, bwd_ms) if dominant == "gdpa_bwd_kernel" else (f_fwd, fwd_ms)
    # algorithmic HBM bytes of one launch: every input read once, every result written once
    esz = lambda t: t.numel() * t.element_size()  # noqa: E731
    fwd_bytes = esz(q) + esz(k) + esz(v) + esz(out) + (esz(lse) if lse is not None else 0)
    bwd_bytes = (esz(q) + esz(k) + esz(v) + (esz(do) if do is not None else 0) + esz(dq) + esz(dk) + esz(dv) +
                 (esz(out) + esz(lse) if lse is not None else 0))
    dom_bytes = bwd_bytes if dominant == "gdpa_bwd_kernel" else fwd_bytes
    hbm = float(peaks["hbm_gbs"])
    # each main kernel against both ceilings: algorithmic bytes (and FLOPs) per launch / its event time
    kernels = {"gdpa_fwd_kernel": {"ms": fwd_ms, "tflops": fwd_tflops, "gbs": fwd_bytes / (fwd_ms * 1e-3) / 1e9,
                                   "hbm_frac": fwd_bytes / (fwd_ms * 1e-3) / 1e9 / hbm,
                                   "algorithmic_bytes": fwd_bytes}}
    if not fwd_only:
        kernels["gdpa_bwd_kernel"] = {"ms": bwd_ms, "tflops": bwd_tflops, "gbs": bwd_bytes / (bwd_ms * 1e-3) / 1e9,
                                      "hbm_frac": bwd_bytes / (bwd_ms * 1e-3) / 1e9 / hbm,
                                      "algorithmic_bytes": bwd_bytes}
    if dom_flops / dom_bytes < peak * 1e12 / (hbm * 1e9):  # below the ridge point: bound by HBM
        achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                    "traffic": recorded_traffic(dominant, wl.name), "kernel": dominant,
                    "peak_source": f"{peak_src} HBM copy bandwidth", "algorithmic_bytes_per_launch": dom_bytes,
                    "avg_launch_ms": dom_ms, "tflops": dom_flops / (dom_ms * 1e-3) / 1e12}
    else:
        achieved = dom_flops / (dom_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": recorded_traffic(dominant, wl.name),
                    "kernel": dominant, "peak_source": peak_label,
                    "algorithmic_flops_per_launch": dom_flops, "avg_launch_ms": dom_ms}

    cpu = None
    if world == 1 and not args.no_cpu_baseline and not fwd_only:
        tf, done, total, secs, thr = oracle_sample(inp, args.cpu_seconds, args.seed)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
               "sample": f"{done} of {total} (sequence, head) units in seeded random order, float64 forward + "
                         f"backward, {secs:.1f} s"}

    in_mb = (esz(q) + esz(k) + esz(v) + (esz(do) if do is not None else 0)) / 2**20
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name + ": " + wl.notes, "total_tokens": inp.total_q, "max_len": wl.max_q,
                   "seed": args.seed, "useful_flops_fwd": f_fwd, "useful_flops_bwd": f_bwd,
                   "l2": "flushed (256 MB write) before every timed step, outside the step's events; "
                         f"inputs ({in_mb:.0f} MB) {'also exceed' if in_mb > 129 else 'are within'} L2 (129 MB)",
                   "parallelism": f"replicas x{world}"},
        "fwd_tflops": fwd_tflops, "bwd_tflops": bwd_tflops,
        "fwd_pct_of_peak": 100.0 * fwd_tflops / peak,
        "bwd_pct_of_peak": 100.0 * bwd_tflops / peak if bwd_tflops is not None else None,
        "peak_bf16_tflops": {"burst": peak, "sustained": float(peaks.get("bf16_tflops_sustained", 0.0)),
                             "source": peak_src},
        "roofline": roofline,
        "kernels": kernels,
        "cpu_baseline": cpu,
        "e2e": e2e,
        # per step: work list + forward kernel (MXFP8: + the scale-atom staging); backward: work list
        # (which also clears the dQ accumulator), prep (softmax rowsum, or direct dQ's unwritten rows),
        # main kernel and (unless dQ is written directly) the dQ convert
        "gpu_launches": (2 + (1 if mxs is not None else 0)
                         + (0 if fwd_only else 2 + (1 if (wl.act == "softmax" or mk <= 128) else 0)
                            + (1 if mk > 128 else 0))) * K,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
