#!/usr/bin/env python
"""KDA forward benchmark on GB300.

Default workload: long_context (B=1, T=65536, H=32, K=V=128, fp32 initial and
final state, seed 3) -- the configuration the headline metric is quoted on.
A step is one full forward pass (chunk schedule, chunk kernel, recurrence
kernel) over that workload with inputs resident in HBM; inputs (2.7 GB per
step) are far larger than L2 (129 MB), so no explicit flush is needed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun, one process per GPU; each rank runs an
independent replica of the workload (the pass has no cross-GPU exchange), so
scaling is weak and value = all ranks' head-tokens / max-over-ranks time.
``--impl reference`` times the fp64 CPU oracle (the reference arm: there is
no runnable reference implementation) on a bounded sample of the workload.
``--pass bwd`` times the backward pass (``kda_bwd``: all eight gradients from
resident inputs and output gradients) instead, with the same launch, JSON
line and reference arm (the fp64 reverse-mode oracle).
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA fwd head-tokens/s at T=65536,H=32; % of roofline (bf16 TC vs HBM)"
UNIT = "head-tokens/s"
D = 128
BYTES_PER_HEAD_TOKEN = 4 * 2 * D + 2 + 2 * D   # q, k, v, g reads + beta + out write = 1282


# ----------------------------------------------------------------------------- counted work

def seq_lengths(p):
    if p["cu_seqlens"] is None:
        return [p["T"]] * p["B"]
    cu = p["cu_seqlens"].tolist()
    return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]


def chunk_flops(c):
    """Counted FLOPs of one chunk of length c for one head (5c^2D + 6cD^2 + c^3/3)."""
    return 5 * c * c * D + 6 * c * D * D + c ** 3 / 3.0


def counted_work(p):
    H = p["H"]
    flops = 0.0
    for L in seq_lengths(p):
        full, rem = divmod(L, 64)
        flops += full * chunk_flops(64) + (chunk_flops(rem) if rem else 0.0)
    flops *= H
    head_tokens = p["B"] * p["T"] * H
    state_bytes = 0
    sd = p["state_dtype"]
    if sd is not None:
        es = 4 if str(sd) == "torch.float32" else 2
        state_bytes = 2 * p["N"] * H * D * D * es   # read initial + write final
    return head_tokens, flops, head_tokens * BYTES_PER_HEAD_TOKEN + state_bytes


def l2_note(alg_bytes, what):
    """How the timed steps stand to the 129 MB L2 (no explicit flush is made)."""
    if alg_bytes > 129e6:
        return "%s larger than L2 (%.2f GB per step vs 129 MB)" % (what, alg_bytes / 1e9)
    return "%s fit in L2 (%.1f MB per step): cache-resident steps, no flush" % (
        what, alg_bytes / 1e6)


def workload_config(w, p, alg_bytes, head_tokens, flops, world):
    return {"workload": w.name, "B": p["B"], "T": p["T"], "H": p["H"], "K": D, "V": D,
            "seed": w.seed, "state_dtype": str(p["state_dtype"]).replace("torch.", ""),
            "parallelism": "replicas" if world > 1 else "single-gpu",
            "l2": l2_note(alg_bytes, "inputs"),
            "head_tokens_per_step": head_tokens, "counted_flop_per_step": flops,
            "counted_bytes_per_step": alg_bytes}


# sources that make up each timed kernel (the hash ties ncu counters to a build)
KERNEL_SOURCES = {
    "chunk": ("kda_prep.cu", "kda_prep.cuh"),
    "recurrence/sliced": ("kda_recur.cu",),
    "recurrence/transposed": ("kda_recur_t.cu", "kda_recur_t.cuh"),
    "fused": ("kda_fused.cu", "kda_prep.cuh", "kda_recur_t.cuh"),
    "decode": ("kda_decode.cu",),
    "recurrence/segmented": ("kda_recur.cu",),
    "maps": ("kda_recur.cu", "kda_segmented.cu"),
    "scan": ("kda_segmented.cu",),
    "bwd": ("kda_bwd.cu", "kda_bwd_status.h"),
}
# kernels one forward pass launches, per path
LAUNCHES = {"sliced": 3, "transposed": 3, "fused": 2, "decode": 1, "segmented": 6}


# shared headers each kernel's sources include (the forward kernels all include tc.cuh)
SHARED_HEADERS = {"bwd": ("kda_internal.h",)}


def kernel_source_hash(kernel):
    """Hash of a kernel's sources and the headers they include, with comments and
    whitespace removed (a comment edit does not make stored counters stale)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel] + SHARED_HEADERS.get(kernel, ("tc.cuh", "kda_internal.h")):
        with open(os.path.join(ROOT, "gated_delta_rule_30_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(re.sub(r"\s+", "", text).encode())
    return h.hexdigest()[:16]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for nm, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- oracle timing

def oracle_sample(p, target_s, max_tokens=None, fixed=None):
    """Time the fp64 oracle (as it stands) on a prefix of S tokens of every head: of the
    packed token stream cut into whole sequences, of the first sequence when a dense
    batch's sequences are longer than S, else of the first S // T whole sequences."""
    import torch

    import oracle
    oracle.build()
    dense = p["cu_seqlens"] is None
    T = p["B"] * p["T"] if dense else int(p["cu_seqlens"][-1])
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    H = p["H"]
    nseq = [1]  # sequences in the last sample

    def run(S):
        if not dense:
            cu = p["cu_seqlens"].tolist()
            n = max(1, max(i for i in range(len(cu)) if cu[i] <= S))
            S = cu[n]
            cu_s = torch.tensor(cu[:n + 1], dtype=torch.int32)
            h0 = None if p["initial_state"] is None else p["initial_state"][:n]
            sl = [x[:1, :S].contiguous() for x in (p["q"], p["k"], p["v"], p["g"], p["beta"])]
        else:
            cu_s = None
            n, L = (1, S) if S <= p["T"] else (min(p["B"], S // p["T"]), p["T"])
            S = n * L
            h0 = None if p["initial_state"] is None else p["initial_state"][:n]
            sl = [x[:n, :L].contiguous() for x in (p["q"], p["k"], p["v"], p["g"], p["beta"])]
        nseq[0] = n
        t0 = time.perf_counter()
        oracle.recurrent(*sl, p["scale"], p["A_log"], p["dt_bias"], p["lower_bound"],
                         initial_state=h0, cu_seqlens=cu_s, nthreads=cores)
        return time.perf_counter() - t0, S * H

    if fixed is not None:
        S = fixed
        dt, ht = run(S)
    else:
        S = min(T, 512)
        dt, ht = run(S)
        S2 = int(min(T, max_tokens or T, S * max(1.0, target_s / max(dt, 1e-3))))
        if S2 > S:
            dt, ht = run(S2)
            S = S2
    threads = min(cores, H * nseq[0])
    return {"value": ht / dt, "unit": UNIT, "cores": threads, "kind": "oracle", "tokens": ht // H,
            "sample": f"first {ht // H} tokens ({nseq[0]} sequence(s)) x {H} heads of the "
                      f"workload ({ht} head-tokens), fp64 C oracle, OpenMP over (sequence, "
                      f"head), {dt:.1f} s"}


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(x, world, device):
    """The largest of each rank's x (replicas: the job takes as long as the slowest)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, seconds):
    """Whole-job rate: every rank processes its own replica of the workload."""
    return units_per_rank * world / seconds


# ----------------------------------------------------------------------------- backward pass

METRIC_BWD = "KDA bwd head-tokens/s (all eight gradients, fp32)"
# bytes per head-token the backward pass must move: q, k, v, g, dout (bf16) and beta
# read; dq, dk, dv, dg (fp32) and dbeta written
BWD_BYTES_PER_HEAD_TOKEN = 5 * 2 * D + 2 + 4 * 4 * D + 4
# fp32 operations per head-token of one forward token step (decay, r = S~^T k,
# rank-1 update: 3 D^2) and one reverse step (dq, dS += q dO^T, du, two for dk,
# dS += k dr^T, da, dS *= a: 8 D^2), a fused multiply-add counting as one
BWD_OPS_PER_HEAD_TOKEN = 11 * D * D
# fp32 lanes x maximum SM clock: 152 SMs x 128 lanes x 2.07 GHz, in Gop/s
FP32_LANE_PEAK_GOPS = 152 * 128 * 2.07


def bwd_oracle_sample(p, ct, target_s, max_tokens=4096, fixed=None):
    """Time the fp64 reverse-mode oracle (as it stands) on the first S tokens of every
    head of the first sequence (it keeps every state of a pair, so S is capped)."""
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    H = p["H"]
    L0 = seq_lengths(p)[0]

    def run(S):
        # sequence 0 starts at token 0 of batch row 0 (dense or packed)
        S = max(1, min(S, L0))
        sl = [x[:1, :S].contiguous() for x in (p["q"], p["k"], p["v"], p["g"], p["beta"])]
        do = ct["dout"][:1, :S].contiguous()
        h0 = None if p["initial_state"] is None else p["initial_state"][:1]
        t0 = time.perf_counter()
        oracle.recurrent_bwd(*sl, p["scale"], p["A_log"], p["dt_bias"], p["lower_bound"], do,
                             initial_state=h0, dfinal_state=ct["dfinal_state"][:1],
                             nthreads=cores)
        return time.perf_counter() - t0, S

    if fixed is not None:
        dt, S = run(fixed)
    else:
        dt, S = run(256)
        S2 = int(min(max_tokens, S * max(1.0, target_s / max(dt, 1e-3))))
        if S2 > S:
            dt, S = run(S2)
    return {"value": S * H / dt, "unit": UNIT, "cores": min(cores, H), "kind": "oracle",
            "tokens": S,
            "sample": f"first {S} tokens of sequence 0 x {H} heads ({S * H} head-tokens), fp64 "
                      f"reverse-mode C oracle, OpenMP over heads, {dt:.1f} s"}


def bench_bwd(args, warmup, rank, world, local_rank, w):
    """The backward pass (kda_bwd) on the workload: device-timed value, an end-to-end
    figure through kda.bwd with pinned host buffers, and the oracle beside it."""
    from gated_delta_rule_30_gb300 import inputs
    p = inputs.make(w)
    ct = inputs.cotangents(p, w.seed)
    head_tokens = p["B"] * p["T"] * p["H"]
    es = 0 if p["state_dtype"] is None else (4 if str(p["state_dtype"]) == "torch.float32" else 2)
    state_bytes = p["N"] * p["H"] * D * D * (es + 4 + 4)  # h0 and dfinal read, dh0 written
    alg_bytes = head_tokens * BWD_BYTES_PER_HEAD_TOKEN + state_bytes
    ops = head_tokens * BWD_OPS_PER_HEAD_TOKEN
    cfg = {"workload": w.name, "B": p["B"], "T": p["T"], "H": p["H"], "K": D, "V": D,
           "seed": w.seed, "cotangent_seed": w.seed + 1000,
           "state_dtype": str(p["state_dtype"]).replace("torch.", ""),
           "parallelism": "replicas" if world > 1 else "single-gpu",
           "l2": l2_note(alg_bytes, "inputs and gradients"),
           "head_tokens_per_step": head_tokens, "counted_ops_per_step": ops,
           "counted_bytes_per_step": alg_bytes, "low_memory": bool(args.low_memory)}
    if args.impl == "reference":
        if rank != 0:
            return 0
        res = bwd_oracle_sample(p, ct, target_s=2.0, max_tokens=1024)
        rates = []
        for i in range(warmup + args.steps):
            r = bwd_oracle_sample(p, ct, 0.0, fixed=res["tokens"])
            if i >= warmup:
                rates.append(r["value"])
        val = statistics.median(rates)
        line = {"impl": "reference", "metric": METRIC_BWD, "value": val, "unit": UNIT,
                "n_gpus": 1, "steps": args.steps, "warmup": warmup, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": cfg,
                "cpu_baseline": {"value": val, "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                                 "sample": r["sample"]},
                "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    import torch.distributed as dist

    import gated_delta_rule_30_gb300 as kda
    from gated_delta_rule_30_gb300 import build as kbuild
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    kbuild.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    dout = ct["dout"].to(dev)
    dhT = ct["dfinal_state"].to(dev)
    ws = torch.empty(kda.bwd_workspace_size(p["B"], p["T"], p["H"],
                                            p["N"] if p["cu_seqlens"] is not None else 0,
                                            p["cu_seqlens"] is not None,
                                            low_memory=args.low_memory),
                     dtype=torch.uint8, device=dev)
    cfg["workspace_bytes"] = ws.numel()

    def step(x, dout_, dhT_):
        return kda.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["A_log"],
                       x["dt_bias"], x["lower_bound"], dout_, initial_state=x["initial_state"],
                       dfinal_state=dhT_, cu_seqlens=x["cu_seqlens"], workspace=ws,
                       low_memory=args.low_memory)

    for _ in range(warmup):
        step(d, dout, dhT)
    torch.cuda.synchronize(dev)
    kda.device_status(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    clocks = ClockSampler(dev.index if world == 1 else local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record(stream)
    for i in range(args.steps):
        step(d, dout, dhT)
        ev[i + 1].record(stream)
    barrier()
    clk = clocks.stop()
    kda.device_status(dev)
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    ms_step = max_over_ranks(ev[0].elapsed_time(ev[-1]) / args.steps, world, dev)

    # end to end: pinned host inputs in, kda.bwd, every gradient back to pinned host
    # memory.  Pipelined like a training loop: two device input sets, one copy
    # stream per input tensor, a copy-out stream; step i+1's copies overlap step i's
    # backward pass and its gradients' readback.
    host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    host["dout"], host["dfinal_state"] = ct["dout"].pin_memory(), ct["dfinal_state"].pin_memory()
    in_keys = [k for k in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state",
                           "cu_seqlens", "dout", "dfinal_state") if host.get(k) is not None]
    h2d = sum(host[k].numel() * host[k].element_size() for k in in_keys)
    d["dout"], d["dfinal_state"] = dout, dhT
    res = step(d, dout, dhT)
    grad_keys = [k for k, v in res.items() if v is not None]
    outs_h = [{k: torch.empty(res[k].shape, dtype=res[k].dtype, pin_memory=True)
               for k in grad_keys} for _ in range(2)]
    d2h = sum(v.numel() * v.element_size() for v in outs_h[0].values())
    del res
    bufs = [d, {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}]
    s_in = [torch.cuda.Stream(dev) for _ in in_keys]
    s_out = torch.cuda.Stream(dev)
    ev_free = [torch.cuda.Event() for _ in range(2)]   # the pass reading buffer set b finished
    ev_read = [torch.cuda.Event() for _ in range(2)]   # gradients of set b read back
    for e in ev_free + ev_read:
        e.record(stream)

    def e2e_step(i):
        b = i & 1
        landed = []
        for j, k in enumerate(in_keys):
            s_in[j].wait_event(ev_free[b])
            with torch.cuda.stream(s_in[j]):
                bufs[b][k].copy_(host[k], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_in[j])
            landed.append(e)
        for e in landed:
            stream.wait_event(e)
        x = bufs[b]
        r = step(x, x["dout"], x["dfinal_state"])
        ev_free[b].record(stream)
        s_out.wait_event(ev_free[b])
        s_out.wait_event(ev_read[b])   # the host buffers of set b are free again
        with torch.cuda.stream(s_out):
            for k in grad_keys:
                r[k].record_stream(s_out)
                outs_h[b][k].copy_(r[k], non_blocking=True)
            ev_read[b].record(s_out)

    e2e_steps = max(1, args.e2e_steps)
    for i in range(2):
        e2e_step(i)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for st_ in s_in + [s_out]:
        st_.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_event(ev_read[(e2e_steps - 1) & 1])
    stream.wait_event(ev_read[e2e_steps & 1])
    e1.record(stream)
    barrier()
    kda.device_status(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)

    ops_rate = ops / (ms_step * 1e-3) / 1e9
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath) and not args.low_memory:
        with open(tpath) as f:
            tr = json.load(f).get("bwd", {})
        if tr.get("source_sha256_16") == kernel_source_hash("bwd") and \
                tr.get("workload") == args.workload:
            traffic = tr.get("bytes_per_launch")
    line = {
        "metric": METRIC_BWD, "value": job_throughput(head_tokens, world, ms_step * 1e-3),
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic", "config": cfg,
        "roofline": {"bound": "alu", "kernel": "bwd", "achieved": ops_rate,
                     "peak": FP32_LANE_PEAK_GOPS, "unit": "Gop/s",
                     "frac": ops_rate / FP32_LANE_PEAK_GOPS, "traffic": traffic,
                     "peak_kind": "derived: 152 SMs x 128 fp32 lanes x 2.07 GHz",
                     "hbm_frac": alg_bytes / (ms_step * 1e-3) / 1e9 / peaks()[0],
                     "note": "achieved = counted fp32 operations of one forward and one reverse "
                             "token step per head-token / step time; the step is the backward "
                             "kernel plus a 1-block parameter reduction"},
        "step_ms_min_max": [min(per), max(per)],
        "e2e": {"value": job_throughput(head_tokens, world, e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "note": "pinned host buffers; copies of step i+1 overlap step i's backward pass "
                        "and readback (two device input sets, one copy stream per input tensor)"},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = bwd_oracle_sample(p, ct, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_context")
    ap.add_argument("--e2e-steps", type=int, default=10,
                    help="steps of the pipelined end-to-end window (fill and drain amortised over it)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="which", choices=["fwd", "bwd"], default="fwd",
                    help="fwd (default): the forward pass; bwd: its backward pass (kda_bwd)")
    ap.add_argument("--low-memory", action="store_true",
                    help="with --pass bwd: the backward pass's low-memory mode (KDA_BWD_LOW_MEMORY)")
    ap.add_argument("--path", default="auto",
                    choices=["auto", "sliced", "transposed", "fused", "segmented"],
                    help="recurrence selection (default: the library's automatic choice)")
    args = ap.parse_args()
    warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    from gated_delta_rule_30_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    if args.which == "bwd":
        return bench_bwd(args, warmup, rank, world, local_rank, w)

    if args.impl == "reference":
        if rank != 0:
            return 0
        p = inputs.make(w)
        # each step: the oracle on a fixed bounded sample (first tokens of every head)
        res = oracle_sample(p, target_s=2.0, max_tokens=2048)
        S_tokens = res["tokens"]
        rates = []
        for i in range(warmup + args.steps):
            r = oracle_sample(p, target_s=0.0, max_tokens=S_tokens, fixed=S_tokens)
            if i >= warmup:
                rates.append(r["value"])
        val = statistics.median(rates)
        res = r
        head_tokens, flops, alg_bytes = counted_work(p)
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": 1,
                "steps": args.steps, "warmup": warmup, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": workload_config(w, p, alg_bytes, head_tokens, flops, 1),
                "cpu_baseline": {"value": val, "unit": UNIT, "cores": res["cores"],
                                 "kind": "oracle", "sample": res["sample"]},
                "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    import torch.distributed as dist

    import gated_delta_rule_30_gb300 as kda
    from gated_delta_rule_30_gb300 import build as kbuild
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    kbuild.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    kda.set_recurrence_kernel(args.path)  # before the workspace size query

    p = inputs.make(w)
    head_tokens, flops, alg_bytes = counted_work(p)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    out = torch.empty_like(d["v"])
    hT = None if d["initial_state"] is None else torch.empty_like(d["initial_state"])
    ws = torch.empty(kda.workspace_size(p["B"], p["T"], p["H"], p["N"] if p["cu_seqlens"] is not None
                                        else 0, p["cu_seqlens"] is not None),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], out, d["A_log"],
                d["dt_bias"], d["lower_bound"], initial_state=d["initial_state"], final_state=hT,
                cu_seqlens=d["cu_seqlens"], workspace=ws)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    kda.device_status(dev)
    path = kda.last_path()  # "sliced" / "transposed": chunk kernel + recurrence; "fused": one launch

    # stage events: per-kernel durations measured on the launch stream
    n_ev = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_ev)]
    for row in evs:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    clocks = ClockSampler(dev.index if world == 1 else local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        kda.set_stage_events(evs[i])
        step()
    t_end.record(stream)
    barrier()
    kda.set_stage_events(None)
    clk = clocks.stop()
    kda.device_status(dev)
    ms_total = t_start.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total, world, dev)
    ms_step = ms_total / args.steps
    # events: [0] before the schedule kernel, [1] after it, [2] after the chunk
    # kernel (fused path: after the fused kernel), [3] after the recurrence
    # (single-token path: [0] before and [1] after its one kernel; segmented
    # path: [3] after the map pass, [4] after the scan, [5] after the recurrence)
    names = {"fused": ("schedule", "fused"), "decode": ("decode",),
             "segmented": ("schedule", "chunk", "maps", "scan", "recurrence")}.get(
        path, ("schedule", "chunk", "recurrence"))
    stage_ms = {k: [] for k in names}
    for row in evs:
        for j, k in enumerate(names):
            stage_ms[k].append(row[j].elapsed_time(row[j + 1]))
    stage_avg = {k: sum(v) / len(v) for k, v in stage_ms.items()}

    # end to end: pinned host inputs -> device -> fwd -> outputs back to pinned host
    host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in p.items()}
    out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    hT_h = None if hT is None else torch.empty(hT.shape, dtype=hT.dtype, pin_memory=True)
    in_keys = [k for k in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state",
                           "cu_seqlens") if host.get(k) is not None]
    h2d = sum(host[k].numel() * host[k].element_size() for k in in_keys)
    d2h = out.numel() * out.element_size() + (0 if hT is None else hT.numel() * hT.element_size())

    # Pipelined like a serving loop: two device input sets, one copy stream per
    # input tensor (parallel copy engines), a copy-out stream.  Every step still
    # copies all of its inputs in from pinned host memory and reads its output
    # (and final state) back; step i+1's copies overlap step i's compute.
    bufs = [d, {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}]
    outs = [out, torch.empty_like(out)]
    hTs = [hT, None if hT is None else torch.empty_like(hT)]
    wss = [ws, torch.empty_like(ws)]
    s_in = [torch.cuda.Stream(dev) for _ in in_keys]
    s_out = torch.cuda.Stream(dev)
    ev_free = [torch.cuda.Event() for _ in range(2)]   # compute on buffer set b finished
    ev_read = [torch.cuda.Event() for _ in range(2)]   # output b read back to the host
    for e in ev_free + ev_read:
        e.record(stream)

    def e2e_step(i):
        b = i & 1
        landed = []
        for j, k in enumerate(in_keys):
            s_in[j].wait_event(ev_free[b])
            with torch.cuda.stream(s_in[j]):
                bufs[b][k].copy_(host[k], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_in[j])
            landed.append(e)
        for e in landed:
            stream.wait_event(e)
        stream.wait_event(ev_read[b])
        x = bufs[b]
        kda.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], outs[b], x["A_log"],
                x["dt_bias"], x["lower_bound"], initial_state=x["initial_state"],
                final_state=hTs[b], cu_seqlens=x["cu_seqlens"], workspace=wss[b])
        ev_free[b].record(stream)
        s_out.wait_event(ev_free[b])
        with torch.cuda.stream(s_out):
            out_h.copy_(outs[b], non_blocking=True)
            if hT is not None:
                hT_h.copy_(hTs[b], non_blocking=True)
            ev_read[b].record(s_out)

    for i in range(2):
        e2e_step(i)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for st_ in s_in + [s_out]:
        st_.wait_event(e0)
    for i in range(args.e2e_steps):
        e2e_step(i)
    stream.wait_event(ev_read[(args.e2e_steps - 1) & 1])
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    kda.device_status(dev)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)

    hbm_peak, bf16_peak, peak_kind = peaks()
    dominant = max((k for k in names if k != "schedule"), key=lambda k: stage_avg[k])
    dom_ms = stage_avg[dominant]
    dom_kernel = dominant if dominant != "recurrence" else "recurrence/" + path
    achieved = alg_bytes / (dom_ms * 1e-3) / 1e9
    roofline_s = max(flops / (bf16_peak * 1e12), alg_bytes / (hbm_peak * 1e9))
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        h = kernel_source_hash(dom_kernel)
        with open(tpath) as f:
            tr = json.load(f).get(dom_kernel, {})
        if tr.get("source_sha256_16") == h and tr.get("workload") == args.workload:
            traffic = tr.get("bytes_per_launch")

    line = {
        "metric": METRIC, "value": job_throughput(head_tokens, world, ms_step * 1e-3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(w, p, alg_bytes, head_tokens, flops, world),
        "tflops": flops / (ms_step * 1e-3) / 1e12,
        "roofline_fraction_step": roofline_s / (ms_step * 1e-3),
        "stage_ms": stage_avg,
        "path": path,
        "roofline": {"bound": "hbm", "kernel": dom_kernel, "achieved": achieved, "peak": hbm_peak,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": traffic,
                     "peak_kind": peak_kind,
                     "note": "achieved = counted bytes of the whole pass / dominant kernel time"},
        "e2e": {"value": job_throughput(head_tokens, world, e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "note": "pinned host buffers; copies of step i+1 overlap step i (two device "
                        "input sets, one copy stream per input tensor)"},
        "gpu_launches": LAUNCHES[path] * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_sample(p, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
