#!/usr/bin/env python
"""Benchmark of the blocked GQA flash-attention hot path (forward + backward).

One step = fa_fwd + fa_bwd (every kernel of the path) over one batch of the
seeded synthetic workload, inputs already resident in HBM.  Prints ONE JSON
line (rank 0).  Metric: attention fwd+bwd TFLOP/s, mask-adjusted, i.e.
4*B*K*G*H*(kept query/key pairs) for the forward and 2.5x that for the
backward, over the device time of the step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU fp64 oracle, same metric

Multi-GPU (torchrun): every rank runs its own copy of the workload (the
(batch, kv head) units are independent, so there is no data exchange); the
only collectives are the timing barrier and the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np
import torch

from flash_attention_gqa_gb300 import inputs

METRIC = "attention fwd+bwd TFLOP/s (mask-adjusted) on 1 GB300; % of bf16 dense peak"
DEFAULT_WORKLOAD = "gqa_causal_h256_t8192"
L2_BYTES = 129 * 2**20

# DRAM traffic per launch of the roofline kernel from one ncu capture, keyed
# by workload and kernel label (as kernel_names() gives it); valid only while
# the kernel source's code (its comments aside) hashes to `src_sha`.  Each
# entry names the capture it comes from in `note`.
_CAPTURE = ("one --metrics capture on one GB300 (medians of 15 launches; profiles/"
            "launches_gqa_causal_h256_t8192.md); DRAM traffic of the same code varies "
            "box to box with L2 residency")
NCU_TRAFFIC: dict = {
    "gqa_causal_h256_t8192": {
        "fa_fwd_kernel<256>": {"bytes_per_launch": 108200000, "src": "fwd.cu",
                               "src_sha": "083071e8dc022dc9", "note": _CAPTURE},
        "fa_bwd_dkdv1_kernel<256, 64, 0, 0>": {"bytes_per_launch": 170500000, "src": "bwd.cu",
                                               "src_sha": "dcda10fcedc593e6", "note": _CAPTURE},
        "fa_bwd_dq_kernel<256, 64, 0>": {"bytes_per_launch": 188400000, "src": "bwd.cu",
                                         "src_sha": "dcda10fcedc593e6", "note": _CAPTURE},
    },
    "gqa_packed_docs_h128_t4096": {
        "fa_bwd_dkdv_kernel<128, 128, 0, 1>": {
            "bytes_per_launch": 426100000, "src": "bwd.cu", "src_sha": "dcda10fcedc593e6",
            "note": ("one ncu --set full capture of one launch on one GB300 "
                     "(profiles/full_packed_docs_h128_t4096.md); DRAM traffic of the same code "
                     "varies box to box with L2 residency")},
    },
}


def kernel_names(w: inputs.Workload, n_splits: int, masked: bool) -> dict:
    """Labels of the launches one step makes, as ncu names the kernels
    (template arguments included), from the rules the library applies: the
    persistent forward for H <= 128 without split-KV when the Q tiles
    outnumber the SMs; the backward's KV tile size and dK/dV split from
    fa_bwd_plan."""
    from flash_attention_gqa_gb300 import binding
    sms = binding.fa_device_sm_count()
    items = -(-w.T // (128 // w.G)) * w.B * w.K
    if n_splits > 1:
        fwd = f"fa_fwd_kernel<{w.H}> (split-KV x{n_splits}) + split_combine_kernel<{w.H}>"
    elif w.H <= 128 and items > sms:
        fwd = f"fa_fwd_persistent_kernel<{w.H}>"
    else:
        fwd = f"fa_fwd_kernel<{w.H}>"
    names = {"fwd": fwd}
    if w.backward:
        rc, kvr, qs = binding.fa_bwd_plan(w.B, w.K, w.G, w.T, w.S, w.H, w.causal,
                                          masked or w.segments, sms)
        assert rc == binding.FA_OK, binding.status_string(rc)
        split, segs = int(qs > 1), int(w.segments)
        dkdv = (f"fa_bwd_dkdv1_kernel<256, {kvr}, {split}, {segs}>" if w.H == 256
                else f"fa_bwd_dkdv_kernel<{max(w.H, 128)}, {kvr}, {split}, {segs}>")
        dq = f"fa_bwd_dq_kernel<{max(w.H, 128)}, {kvr}, {segs}>"
        pre = f"bwd_preprocess_kernel<{w.H}>" + (" + seg_ranges_kernel x2" if w.segments else "")
        names.update(pre=pre, dkdv=dkdv, dq=dq, bwd=f"fa_bwd_masked: {pre} + {dkdv} + {dq}")
    return names


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-rows", type=int, default=2048,
                   help="query positions in the oracle's timed sample")
    return p.parse_args()


# ------------------------------------------------------------- bookkeeping

def flop_counts(w: inputs.Workload, seg: np.ndarray | None, dense_mask=None):
    if dense_mask is not None:   # the mask already encodes causality and the window
        pairs = int(dense_mask.sum()) * w.B
    else:
        pairs = inputs.unmasked_pairs(w.T, w.S, w.causal, seg, seg, B=w.B)
    fwd = 4.0 * w.K * w.G * w.H * pairs
    return fwd, (2.5 * fwd if w.backward else 0.0), pairs / (w.B * w.T * w.S)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), d.get("hbm_gbs"), "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


def src_sha(name: str) -> str:
    """Hash of a kernel source's code: `//` comments, surrounding blanks and empty
    lines are dropped, so a comment edit keeps the counters taken for the code."""
    with open(os.path.join(ROOT, "flash_attention_gqa_gb300", "csrc", name), encoding="utf-8") as f:
        code = [line.split("//", 1)[0].strip() for line in f]
    return hashlib.sha256("\n".join(c for c in code if c).encode()).hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        out = os.environ.get("FA_BENCH_OUT", os.path.join(ROOT, "bench_out"))
        self.path = os.path.join(out, f"clocks_rank{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
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
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- oracle

def oracle_sample(w: inputs.Workload, x: inputs.Tensors, rows: int, dense_mask=None):
    """The first `rows` query positions of the workload (with the keys they can
    see when causal) as a self-contained sub-problem for the CPU oracle."""
    rows = min(rows, w.T)
    sl = lambda t, ax, n: t.narrow(ax, 0, n)
    nkeys = rows if w.causal else w.S
    sub = dict(q=sl(x.q, 3, rows), k=sl(x.k, 2, nkeys), v=sl(x.v, 2, nkeys),
               dO=None if x.dO is None else sl(x.dO, 3, rows),
               seg_q=None if x.seg_q is None else sl(x.seg_q, 1, rows),
               seg_kv=None if x.seg_kv is None else sl(x.seg_kv, 1, nkeys))
    segq = None if sub["seg_q"] is None else sub["seg_q"].numpy()
    segk = None if sub["seg_kv"] is None else sub["seg_kv"].numpy()
    if w.kind == "decode":
        nkeys = w.S   # one query against the whole cache
        sub.update(k=x.k, v=x.v)
    sub["mask"] = None
    if dense_mask is not None:
        sub["mask"] = dense_mask[:, :rows, :nkeys]
        pairs = int(sub["mask"].sum()) * w.B
    else:
        pairs = inputs.unmasked_pairs(rows, nkeys, w.causal, segq, segk, B=w.B)
    fwd = 4.0 * w.K * w.G * w.H * pairs
    flop = fwd * (3.5 if w.backward else 1.0)
    desc = (f"first {rows} of {w.T} query positions x all {w.B * w.K * w.G} heads "
            f"against {'the keys they can see' if w.causal else 'all keys'}; "
            f"{'forward + backward' if w.backward else 'forward'}")
    return sub, flop, desc


def run_oracle_step(w, sub):
    import oracle  # the CPU oracle: only the baseline / reference legs use it
    kw = dict(causal=w.causal, seg_q=sub["seg_q"], seg_kv=sub["seg_kv"], mask=sub["mask"])
    oracle.attention_forward(sub["q"], sub["k"], sub["v"], **kw)
    if w.backward:
        oracle.attention_backward(sub["q"], sub["k"], sub["v"], sub["dO"], **kw)


def cpu_baseline(w, x, rows, dense_mask=None):
    sub, flop, desc = oracle_sample(w, x, rows, dense_mask)
    t = time.perf_counter()
    run_oracle_step(w, sub)
    dt = time.perf_counter() - t
    return {"value": round(flop / dt / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": desc + f"; numpy fp64, BLAS pool of {os.cpu_count()} threads"}


# ------------------------------------------------------------------ arms

def reduce_max(x: float, device=None) -> float:
    """Max of a per-rank timing over all ranks (identity without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group(backend="nccl")
    return world, rank, local


def reference_arm(args, world, rank):
    if rank != 0:
        return
    w = inputs.WORKLOADS[args.workload]
    x = inputs.make_workload(w)
    dense_mask = inputs.window_mask(w.T, w.S, w.window) if w.kind == "window" else None
    # Size the sample so the whole run stays within about two and a half
    # minutes: time a 256-row sample once (untimed) and scale by the causal
    # (quadratic) or linear growth of the work with the number of rows.
    budget = 150.0 / max(1, args.steps + args.warmup)
    probe, _, _ = oracle_sample(w, x, 256, dense_mask)
    t = time.perf_counter()
    run_oracle_step(w, probe)
    t256 = max(time.perf_counter() - t, 1e-3)
    growth = 0.5 if w.causal else 1.0
    rows = int(256 * (budget / t256) ** growth) // 128 * 128
    rows = max(1, min(max(rows, 128), 2048, w.T))
    sub, flop, desc = oracle_sample(w, x, rows, dense_mask)
    for _ in range(args.warmup):
        run_oracle_step(w, sub)
    t = time.perf_counter()
    for _ in range(args.steps):
        run_oracle_step(w, sub)
    dt = (time.perf_counter() - t) / max(args.steps, 1)
    value = round(flop / dt / 1e12, 6)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1), bf16-rounded)",
        "config": {"workload": w.name, "B": w.B, "K": w.K, "G": w.G, "T": w.T, "S": w.S,
                   "H": w.H, "causal": w.causal, "segments": w.segments,
                   "sample": desc},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def ours_arm(args, world, rank, local):
    from flash_attention_gqa_gb300 import binding
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = binding.load()
    w = inputs.WORKLOADS[args.workload]
    x = inputs.make_workload(w)
    seg_np = None if x.seg_q is None else x.seg_q.numpy()
    dense_mask = inputs.window_mask(w.T, w.S, w.window) if w.kind == "window" else None
    fwd_flop, bwd_flop, frac = flop_counts(w, seg_np, dense_mask)
    step_flop = fwd_flop + bwd_flop
    meta = None
    if dense_mask is not None:
        meta = binding.block_mask_from_dense(dense_mask, device=dev)
    n_splits = 1
    if w.kind == "decode":
        n_splits = binding.fa_fwd_splitkv_default_splits(w.B, w.K, w.G, w.T, w.S, w.H)

    q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
    dO = x.dO.to(dev) if w.backward else None
    sq = None if x.seg_q is None else x.seg_q.to(dev)
    skv = None if x.seg_kv is None else x.seg_kv.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.K, w.G, w.T), dtype=torch.float32, device=dev)
    if w.backward:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(max(256, binding.fa_bwd_workspace_size(w.B, w.K, w.G, w.T, w.S, w.H)),
                         dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    if n_splits > 1:
        ws_split = torch.empty(binding.fa_fwd_splitkv_workspace_size(w.B, w.K, w.G, w.T, w.S, w.H,
                                                                     n_splits),
                               dtype=torch.uint8, device=dev)
    n_kernels = 1 + (1 if n_splits > 1 else 0) + \
        ((1 + (2 if sq is not None else 0) + 2) if w.backward else 0)
    n_ev = 5 if w.backward else 2

    # device buffers of one step: inputs (q, k, v, dO, seg ids) and outputs
    bufs0 = {"q": q, "k": k, "v": v, "dO": dO, "sq": sq, "skv": skv, "o": o, "lse": lse}
    if w.backward:
        bufs0.update(dq=dq, dk=dk, dv=dv)

    def step(evs=None, bufs=None):
        B_ = bufs0 if bufs is None else bufs
        q_, k_, v_, dO_, sq_, skv_ = (B_[n] for n in ("q", "k", "v", "dO", "sq", "skv"))
        o_, lse_ = B_["o"], B_["lse"]
        if evs is not None:
            evs[0].record(stream)
        if meta is not None:
            binding.fa_fwd_masked(q_, k_, v_, sq_, skv_, w.causal, meta, o_, lse_, stream)
        elif n_splits > 1:
            binding.fa_fwd_splitkv(q_, k_, v_, sq_, skv_, w.causal, o_, lse_, n_splits, ws_split,
                                   stream)
        else:
            binding.fa_fwd(q_, k_, v_, sq_, skv_, w.causal, o_, lse_, stream)
        if evs is not None:
            evs[1].record(stream)
        if not w.backward:
            return
        dq_, dk_, dv_ = B_["dq"], B_["dk"], B_["dv"]
        if meta is not None:
            # the masked backward runs its stages back to back (one call)
            binding.fa_bwd_masked(q_, k_, v_, o_, lse_, dO_, sq_, skv_, w.causal, meta, dq_, dk_,
                                  dv_, ws, stream)
            if evs is not None:
                for i in (2, 3, 4):
                    evs[i].record(stream)
        elif evs is None:
            # one call: the dQ grid may overlap the tail of the dK/dV grid
            binding.fa_bwd(q_, k_, v_, o_, lse_, dO_, sq_, skv_, w.causal, dq_, dk_, dv_, ws, stream)
        else:
            # stage by stage with events between them: per-kernel durations
            for st in range(3):
                binding.fa_bwd_stage(st, q_, k_, v_, o_, lse_, dO_, sq_, skv_, w.causal, dq_, dk_,
                                     dv_, ws, stream)
                evs[2 + st].record(stream)

    # Inputs and outputs smaller than L2: write a buffer of twice L2 between
    # timed steps (outside their events) so that no step starts L2-warm.
    in_bytes = sum(t.numel() * t.element_size() for t in bufs0.values() if t is not None)
    small = in_bytes <= L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if small else None

    def flush():
        if flush_buf is not None:
            flush_buf.fill_(1)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert binding.fa_check_status(stream) == binding.FA_OK

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # every step between its own pair of events; the reported step time is the
    # median over the timed steps (the mean is reported beside it)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    t_start.record(stream)
    for i in range(args.steps):
        flush()
        step_ev[i][0].record(stream)
        step()
        step_ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    status = binding.fa_check_status(stream)
    assert status == binding.FA_OK, binding.status_string(status)
    step_ms = [a_.elapsed_time(b_) for a_, b_ in step_ev]
    ms = reduce_max(statistics.median(step_ms), dev)
    ms_mean = reduce_max(statistics.mean(step_ms), dev)
    span_ms = reduce_max(t_start.elapsed_time(t_end), dev)

    # per-kernel device time: a second loop, stage by stage with CUDA events
    # between the launches (which also keeps dQ from overlapping dK/dV there)
    n_k = max(3, min(args.steps, 20))
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(n_k)]
    for i in range(n_k):
        flush()
        step(events[i])
    torch.cuda.synchronize()
    med = lambda i, j: statistics.median(e[i].elapsed_time(e[j]) for e in events)
    names = kernel_names(w, n_splits, meta is not None)
    per = {names["fwd"]: med(0, 1)}
    # algorithmic FLOPs each launch performs: fwd = S and O products; dK/dV = S,
    # dP, dV, dK products (2x fwd); dQ = S, dP, dQ products (1.5x fwd); the
    # backward as a whole counts 2.5x fwd
    kflop = {names["fwd"]: fwd_flop}
    if w.backward and meta is None:
        per[names["pre"]] = med(1, 2)
        per[names["dkdv"]] = med(2, 3)
        per[names["dq"]] = med(3, 4)
        kflop.update({names["dkdv"]: 2.0 * fwd_flop, names["dq"]: 1.5 * fwd_flop})
    elif w.backward:   # the masked backward is one call: timed and counted as a whole
        per[names["bwd"]] = med(1, 4)
        kflop[names["bwd"]] = bwd_flop
    top = max((n for n in per if n in kflop), key=lambda n: per[n])
    burst, sustained, hbm, src = measured_peaks()
    timed_s = span_ms / 1e3
    peak = burst if timed_s < 1.0 else sustained
    tr = NCU_TRAFFIC.get(w.name, {}).get(top)
    traffic = tr["bytes_per_launch"] if tr and tr.get("src_sha") == src_sha(tr["src"]) else None
    # forward algorithmic bytes: q, k, v, o and lse move once
    fbytes = 2 * (x.k.numel() + x.v.numel() + 2 * x.q.numel()) + 4 * lse.numel()
    ridge = peak * 1e12 / (hbm * 1e9)   # FLOP per byte where the two roofs meet
    if w.kind == "decode" or (not w.backward and fwd_flop / fbytes < ridge):
        # below the ridge: the roofline bound is HBM
        achieved = fbytes / (per[names["fwd"]] * 1e-3) / 1e9
        kname = names["fwd"]
        roofline = {"bound": "hbm", "kernel": kname,
                    "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(achieved / hbm, 4), "traffic": None,
                    "algorithmic_bytes": fbytes, "intensity_flop_per_byte": round(fwd_flop / fbytes, 1),
                    "ridge_flop_per_byte": round(ridge, 1), "peak_source": f"{src} HBM copy",
                    "per_kernel_ms": {n: round(t, 4) for n, t in per.items()}}
    else:
        achieved = kflop[top] / (per[top] * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": top, "achieved": round(achieved, 1),
                    "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "traffic": traffic,
                    "traffic_source": (tr["note"] if traffic is not None else
                                       "no ncu capture of this kernel's current code"),
                    "algorithmic_flop": kflop[top],
                    "peak_source": f"{src} bf16 {'burst' if peak == burst else 'sustained'}",
                    "per_kernel_ms": {n: round(t, 4) for n, t in per.items()},
                    "per_kernel_ms_stat": f"median of {n_k} steps, events between launches"}

    # end to end through the C ABI with host buffers: H2D inputs, D2H outputs
    host_in = [t.pin_memory() for t in (x.q, x.k, x.v) + ((x.dO,) if w.backward else ())]
    seg_host = [] if x.seg_q is None else [x.seg_q.pin_memory(), x.seg_kv.pin_memory()]
    dev_in = [q, k, v] + ([dO] if w.backward else [])
    dev_seg = [] if sq is None else [sq, skv]
    outs = [o, lse] + ([dq, dk, dv] if w.backward else [])
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in host_in + seg_host)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    # as many steps as the device-timed loop: the pipelined mode's fill (first
    # H2D) and drain (last D2H) are spread over the same run length
    e2e_steps = max(3, args.steps)

    def e2e_step():
        for h, d in zip(host_in + seg_host, dev_in + dev_seg):
            d.copy_(h, non_blocking=True)
        step()
        for h, d in zip(host_out, outs):
            h.copy_(d, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = reduce_max(e0.elapsed_time(e1) / e2e_steps, dev)

    # Pipelined: two device buffer sets; step i's inputs are copied in on one
    # stream and step i-1's results copied out on another while step i-1 / i
    # compute, as a training loop with prefetch would.  Every step still moves
    # its inputs from pinned host memory and its results back.
    in_names = [n for n in ("q", "k", "v", "dO", "sq", "skv") if bufs0[n] is not None]
    out_names = ["o", "lse"] + (["dq", "dk", "dv"] if w.backward else [])
    bufs1 = {n: (torch.empty_like(t) if t is not None else None) for n, t in bufs0.items()}
    sets = [bufs0, bufs1]
    host_src = dict(zip(["q", "k", "v"] + (["dO"] if w.backward else []), host_in))
    if seg_host:
        host_src.update(sq=seg_host[0], skv=seg_host[1])
    host_dst = [dict(zip(out_names, host_out)),
                {n: torch.empty(bufs0[n].shape, dtype=bufs0[n].dtype, pin_memory=True)
                 for n in out_names}]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_pipelined(n_steps):
        ev = [{k_: torch.cuda.Event() for k_ in ("h2d", "comp", "d2h")} for _ in range(n_steps)]
        start = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for i in range(n_steps):
            b_ = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev[i - 2]["comp"])  # inputs of set b_ were read
                for n in in_names:
                    sets[b_][n].copy_(host_src[n], non_blocking=True)
                ev[i]["h2d"].record(s_in)
            stream.wait_event(ev[i]["h2d"])
            if i >= 2:
                stream.wait_event(ev[i - 2]["d2h"])  # outputs of set b_ were read back
            step(bufs=sets[b_])
            ev[i]["comp"].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev[i]["comp"])
                for n in out_names:
                    host_dst[b_][n].copy_(sets[b_][n], non_blocking=True)
                ev[i]["d2h"].record(s_out)
        stream.wait_event(ev[n_steps - 1]["d2h"])
        stream.wait_event(ev[n_steps - 1]["h2d"])
        end = torch.cuda.Event(enable_timing=True)
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / n_steps

    e2e_pipelined(2)
    e2e_ms = reduce_max(e2e_pipelined(e2e_steps), dev)
    # both are end to end (every step's inputs in, results out); report the faster
    if e2e_ms <= e2e_serial_ms:
        e2e_best, e2e_mode = e2e_ms, ("pipelined: H2D of step i and D2H of step i-1 on two copy "
                                      "streams overlap the kernels (two device buffer sets)")
    else:
        e2e_best, e2e_mode = e2e_serial_ms, "serial: H2D, kernels, D2H in order on one stream"
    torch.cuda.synchronize()
    status = binding.fa_check_status(stream)
    assert status == binding.FA_OK, binding.status_string(status)

    line = {
        "metric": METRIC,
        "value": round(world * step_flop / (ms * 1e-3) / 1e12, 2),
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "ms_per_step_stat": f"median of {args.steps} steps",
        "ms_per_step_mean": round(ms_mean, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16-rounded; q pre-scaled by H^-1/2)",
        "config": {"workload": w.name, "B": w.B, "K": w.K, "G": w.G, "T": w.T, "S": w.S,
                   "H": w.H, "causal": w.causal, "segments": w.segments,
                   "unmasked_frac": round(frac, 6), "fwd_flop": fwd_flop, "bwd_flop": bwd_flop,
                   "fwd_tflops": round(fwd_flop / (per[names["fwd"]] * 1e-3) / 1e12, 1),
                   "bwd_tflops": (round(bwd_flop / ((ms - per[names["fwd"]]) * 1e-3) / 1e12, 1)
                                  if w.backward else None),
                   "kind": w.kind, "split_kv": n_splits if n_splits > 1 else None,
                   "window": w.window or None,
                   "pct_of_peak": round(100 * step_flop / (ms * 1e-3) / 1e12 / peak, 2),
                   "l2": f"inputs+outputs {in_bytes / 2**20:.0f} MiB vs L2 {L2_BYTES / 2**20:.0f} MiB"
                         + (" (larger: no flush)" if not small else
                            f" (smaller: {2 * L2_BYTES / 2**20:.0f} MiB written between timed steps, "
                            "outside the steps' events)"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roofline,
        "e2e": {"value": round(world * step_flop / (e2e_best * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_best, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "mode": e2e_mode,
                "pipelined_ms_per_step": round(e2e_ms, 4),
                "serial_ms_per_step": round(e2e_serial_ms, 4), "steps": e2e_steps},
        "gpu_launches": n_kernels * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, x, args.cpu_rows, dense_mask)
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            reference_arm(args, world, rank)
        else:
            ours_arm(args, world, rank, local)
    finally:
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
