#!/usr/bin/env python
"""Causal MHA/GQA attention forward + backward throughput on GB300.

One step = attn_fwd_ws (the forward with its RoPE pass over Q/K into a
workspace) + attn_bwd_rot (the backward with its prologue kernel, reading the
forward's rotated Q/K) over one batch of the synthetic workload, through the
library's C ABI.  Prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload gqa_block|long_context_gqa|gpt2_124m_mha]

Metric: causal attention fwd+bwd TFLOP/s with the algorithmic causal FLOP
count (pairs = T(T+1)/2, fwd = 4*B*NH*hd*pairs, bwd = 2.5*fwd).  Under
torchrun (N > 1) rank r runs its own shard of a global batch of N*B rows (the
workload's shapes, its own seeded batch rows: the path shards over batch rows
and kv groups with no exchange); the value is the work of all ranks divided by
the slowest rank's time.

The default run also times the long-context GQA workload (`--also`, at most
`--also-steps` steps) in the same process and reports it under `per_config`,
so both GQA bf16 configurations are measured by one command.  Fractions are
priced against the measured burst bf16 peak (a short cuBLAS loop at full
clocks) unless a timed region lasts at least two seconds, when the sustained
(power-capped) figure applies; the line names the peak it used.  Next to the
per-kernel roofline, `bwd_combined` gives the backward's five algorithmic GEMM
units over the summed time of its two tensor-core kernels.

`--impl reference` times the float64 CPU oracle instead (rank 0 only), on a
bounded sample of the same workload: one kv group of one batch row per step.

`--proj B,T,Cm,NH,NKV,hd` times attn_qkv_proj (the QKV projection GEMM with
the rotated Q/K copy in its epilogue, and without the copy), with cuBLAS
(torch.matmul) on the same GEMM for context, and prints one JSON line.

`--fp8` times attn_fwd_fp8 (the e4m3 forward, its quantization pass
included) next to attn_fwd_ws on the workload and prints one JSON line
(forward TFLOP/s against the FP8 peak = 2 x the measured bf16 peak, the
nominal dense fp8/bf16 ratio).

`--rope-interleaved` runs the same step with interleaved (GPT-J) RoPE pairs.

`--decode B,L,NH,NKV,hd` times attn_decode (one new token per batch row
against a bf16 KV cache of L rows) instead and prints one JSON line with its
HBM throughput (cache bytes read per call / device time; L2 flushed between
calls) against the measured copy bandwidth.
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

METRIC = "causal attn fwd+bwd TFLOP/s on 1 GB300; % of BF16 tensor peak"
FLUSH_BYTES = 256 << 20          # > 129 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {
    "fwd_tc05": "attn_fwd2_sm103.cu", "bwd_dkdv_tc05": "attn_bwd_sm103.cu", "bwd_dq_tc05": "attn_bwd_sm103.cu",
    "bwd_row_dot": "attn_prep.cu", "rope_qk": "attn_prep.cu", "bwd_prologue": "attn_prep.cu",
    "fwd_split": "attn_split_sm103.cu", "bwd_dkdv_split": "attn_split_sm103.cu", "bwd_dq_split": "attn_split_sm103.cu",
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gqa_block")
    ap.add_argument("--also", default="long_context_gqa",
                    help="second workload timed in the same run and reported under per_config ('' for none)")
    ap.add_argument("--also-steps", type=int, default=200)
    ap.add_argument("--dtype", choices=["bf16", "tf32"], default="bf16",
                    help="tf32: float32 tensors through ATTN_DTYPE_TF32 (the split tensor-core path at head size 64)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode", default=None, metavar="B,L,NH,NKV,hd")
    ap.add_argument("--proj", default=None, metavar="B,T,Cm,NH,NKV,hd")
    ap.add_argument("--fp8", action="store_true")
    ap.add_argument("--rope-interleaved", action="store_true")
    return ap.parse_args()


# --------------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def config_of(w, extra=None):
    cfg = {"workload": w.name, "B": w.B, "T": w.T, "C": w.C, "NH": w.NH, "NKV": w.NKV, "hd": w.hd,
           "rope_theta": w.rope_theta, "qkv_std": w.qkv_std, "dout_std": w.dout_std, "seed": w.seed}
    cfg.update(extra or {})
    return cfg


def flops_per_step(w):
    return w.flops_fwd() + w.flops_bwd()


def oracle_sample(w):
    """One kv group of batch row 0 as a standalone problem (NH = grp, NKV = 1)."""
    import numpy as np
    from causal_attention_gqa_gb300.workloads import make_inputs
    qkv, dout = make_inputs(w, "bf16")
    hd, grp = w.hd, w.NH // w.NKV
    q = qkv[:1, :, :grp * hd]
    k = qkv[:1, :, w.C:w.C + hd]
    v = qkv[:1, :, w.C + w.NKV * hd:w.C + w.NKV * hd + hd]
    sub_qkv = np.ascontiguousarray(np.concatenate([q, k, v], axis=2))
    sub_dout = np.ascontiguousarray(dout[:1, :, :grp * hd])
    sub = w.replace(B=1, C=grp * hd, NH=grp, NKV=1)
    return sub, sub_qkv, sub_dout


def time_oracle(w, min_seconds=10.0, max_reps=50):
    """Time the oracle's forward+backward on the bounded sample; TFLOP/s."""
    import oracle
    sub, qkv, dout = oracle_sample(w)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.attention_backward(qkv, dout, sub.C, sub.NH, sub.NKV, sub.rope_theta, return_aux=True)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {
        "value": flops_per_step(sub) * reps / el / 1e12,
        "unit": "TFLOP/s",
        "cores": cores,
        "kind": "oracle",
        "sample": f"float64 NumPy oracle fwd+bwd of one kv group ({sub.NH} query heads, T={sub.T}, "
                  f"hd={sub.hd}) of batch row 0, x{reps} in {el:.1f} s",
        "seconds": el,
    }


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        idx = vis.split(",")[local_rank] if vis else str(local_rank)
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons)}


def traffic_for(kernel, workload=None):
    """DRAM bytes per launch from the committed ncu summary of this kernel on
    this workload, if the kernel's source is unchanged since the capture;
    else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    rec = table.get(f"{kernel}@{workload}") or table.get(kernel)
    if not rec or (workload is not None and rec.get("workload") != workload):
        return None
    # A record may name its own source file (the same event name covers
    # different kernels at different head sizes).
    src = os.path.join(ROOT, "causal_attention_gqa_gb300", "csrc", rec.get("source") or KERNEL_SOURCES.get(kernel, ""))
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    return rec.get("bytes_per_launch") if rec.get("source_sha256") == sha else None


def kernel_algorithmic_flops(name, w):
    """Algorithmic FLOPs one launch of `name` processes (causal pairs only).
    One GEMM-unit = 2*B*NH*hd*pairs; the forward is 2 units (QK^T, PV); the
    dK/dV kernel covers 4 (S, dP, dV, dK); the dQ kernel 1 (dQ; its S and dP
    recomputation is extra work, not counted)."""
    unit = 2.0 * w.B * w.NH * w.hd * w.causal_pairs
    return {"fwd_tc05": 2 * unit, "bwd_dkdv_tc05": 4 * unit, "bwd_dq_tc05": 1 * unit,
            "fwd_split": 2 * unit, "bwd_dkdv_split": 4 * unit, "bwd_dq_split": 1 * unit}.get(name)


# --------------------------------------------------------------------------- arms
def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    sub, qkv, dout = oracle_sample(w)
    for _ in range(args.warmup):
        oracle.attention_backward(qkv, dout, sub.C, sub.NH, sub.NKV, sub.rope_theta, return_aux=True)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention_backward(qkv, dout, sub.C, sub.NH, sub.NKV, sub.rope_theta, return_aux=True)
    el = time.perf_counter() - t0
    value = flops_per_step(sub) * args.steps / el / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, {"sample": "one kv group of batch row 0 per step"}),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"float64 NumPy oracle fwd+bwd of one kv group ({sub.NH} query heads, "
                                   f"T={sub.T}, hd={sub.hd}) of batch row 0 per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def max_over_ranks(values, device):
    """Element-wise maximum of per-rank numbers over the process group (the
    slowest rank's times); the values themselves when there is no group."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


SUSTAINED_AFTER_S = 2.0     # a timed region at least this long is priced against the sustained peak


TF32_PER_BF16 = 1.1 / 2.25   # nominal dense TF32 / bf16 tensor rates of a GB300


def choose_peak(peaks, peak_src, timed_seconds, dtype="bf16"):
    """The peak a timed region is priced against: the measured bf16 burst
    figure (a short cuBLAS loop at full clocks) unless the region lasted long
    enough for the power cap to pull the clocks down, then the sustained one;
    for float32 tensors on the TF32 dtype, that figure times the nominal
    TF32/bf16 ratio."""
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    if timed_seconds >= SUSTAINED_AFTER_S:
        tf, desc = sustained, f"{peak_src} bf16_tflops_sustained ({timed_seconds:.2f} s timed region)"
    else:
        tf, desc = burst, f"{peak_src} bf16_tflops (burst: {timed_seconds:.3f} s timed region < {SUSTAINED_AFTER_S} s)"
    if dtype == "tf32":
        return tf * TF32_PER_BF16, desc + " x 1.1/2.25 (nominal dense TF32/bf16)"
    return tf, desc


def roofline_of(prof, w, peak_tf, peak_desc):
    """Dominant kernel's roofline (algorithmic FLOPs per launch / mean launch
    time) and the backward's combined figure: the five backward GEMM units
    over the summed time of the dK/dV and dQ kernels (the per-kernel split
    credits the S/dP recomputation of the dQ kernel to neither)."""
    kernel_ms = {k: v[1] for k, v in prof.items()}
    dom = max(kernel_ms, key=kernel_ms.get)
    n_launch, tot_ms = prof[dom]
    kfl = kernel_algorithmic_flops(dom, w)
    roof = None
    if kfl is not None:
        achieved = kfl / (tot_ms / n_launch * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": achieved / peak_tf, "traffic": traffic_for(dom, w.name), "peak_source": peak_desc,
                "avg_launch_ms": tot_ms / n_launch, "algorithmic_flop_per_launch": kfl}
    bwd = [k for k in ("bwd_dkdv_tc05", "bwd_dq_tc05", "bwd_dkdv_split", "bwd_dq_split") if k in prof]
    combined = None
    if bwd:
        t = sum(prof[k][1] / prof[k][0] for k in bwd)
        achieved = w.flops_bwd() / (t * 1e-3) / 1e12
        combined = {"kernels": bwd, "algorithmic_flop_per_step": w.flops_bwd(), "ms": t,
                    "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s", "frac": achieved / peak_tf}
    return roof, combined


def time_workload(args, w, dev, world, steps, e2e):
    """Time `steps` fwd+bwd steps of workload `w` (this rank's shard) with
    inputs resident in HBM; then a per-kernel event pass; then (if `e2e`) the
    end-to-end loop with host buffers.  Returns raw per-rank numbers."""
    import torch
    import torch.distributed as dist
    from causal_attention_gqa_gb300 import binding
    from causal_attention_gqa_gb300.workloads import make_inputs

    B, T, C, NH, NKV = w.B, w.T, w.C, w.NH, w.NKV
    tf32 = args.dtype == "tf32"
    tdt, esz = (torch.float32, 4) if tf32 else (torch.bfloat16, 2)
    qkv_np, dout_np = make_inputs(w, "f32" if tf32 else "bf16")
    qkv_host = torch.from_numpy(qkv_np).to(tdt).pin_memory()
    dout_host = torch.from_numpy(dout_np).to(tdt).pin_memory()
    del qkv_np, dout_np
    qkv = qkv_host.to(dev)
    dout = dout_host.to(dev)
    out = torch.empty((B, T, C), dtype=tdt, device=dev)
    lse = torch.empty((B, NH, T), dtype=torch.float32, device=dev)
    dqkv = torch.empty_like(qkv)
    dqkv_host = torch.empty(dqkv.shape, dtype=tdt).pin_memory()
    base = binding.DTYPE_TF32 if tf32 else binding.DTYPE_BF16
    ws_bytes = binding.attn_bwd_workspace_bytes(B, T, C, NH, NKV, base)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    fws_bytes = binding.attn_fwd_workspace_bytes(B, T, C, NH, NKV, base)
    fws = torch.empty(max(fws_bytes, 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    code = base | (binding.FLAG_ROPE_INTERLEAVED if args.rope_interleaved else 0)

    def step(qkv=qkv, dout=dout, dqkv=dqkv):
        binding.attn_fwd_ws(out, lse, qkv, B, T, C, NH, NKV, w.rope_theta, code, fws, fws_bytes, sptr)
        binding.attn_bwd_rot(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, w.rope_theta, code, fws, ws, ws_bytes,
                             sptr)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    barrier()
    if binding.attn_device_status() != 0:
        raise RuntimeError("device-side error recorded during warm-up")

    # ---- device-resident timed region: K steps, L2 flushed between steps.
    # No per-kernel events here: events between the backward's programmatically
    # dependent launches would serialise them.
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    sampler = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    time.sleep(0.15)
    barrier()
    wall0 = time.perf_counter()
    for k in range(steps):
        flush.zero_()
        starts[k].record(stream)
        step()
        ends[k].record(stream)
    barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    ms_steps = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    ms_per_step = sum(ms_steps) / steps
    if binding.attn_device_status() != 0:
        raise RuntimeError("device-side error recorded during the timed region")

    # ---- the same steps again with the library's per-kernel CUDA events on
    # the launching stream: kernel breakdown, dominant kernel, roofline.
    n_prof = max(1, min(steps, 50))
    binding.attn_profile_start()
    for _ in range(n_prof):
        flush.zero_()
        step()
    barrier()
    prof = binding.attn_profile_stop()
    res = {"ms_per_step": ms_per_step, "timed_s": sum(ms_steps) * 1e-3, "wall": wall, "clocks": clocks,
           "prof": prof, "n_prof": n_prof, "steps": steps}
    if not e2e:
        return res

    # ---- end to end through the C ABI with host buffers.  Every step copies
    # its qkv and dout from pinned host memory and reads its dqkv back; the
    # copies run on their own streams into/out of two device buffer sets, so
    # step k's inputs arrive and step k-1's gradients leave while step k-1 /
    # step k compute (events order each buffer's writer after its readers).
    bufs = [(qkv, dout, dqkv), (torch.empty_like(qkv), torch.empty_like(dout), torch.empty_like(dqkv))]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e2e_steps = max(2, min(steps, 50))
    barrier()
    e_start.record(stream)
    s_in.wait_event(e_start)
    for k in range(e2e_steps):
        i = k % 2
        q_d, o_d, g_d = bufs[i]
        if k >= 2:
            s_in.wait_event(ev_done[i])          # step k-2 has read this buffer set
        with torch.cuda.stream(s_in):
            q_d.copy_(qkv_host, non_blocking=True)
            o_d.copy_(dout_host, non_blocking=True)
            ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        if k >= 2:
            stream.wait_event(ev_out[i])         # step k-2's gradients have left
        step(q_d, o_d, g_d)
        ev_done[i].record(stream)
        s_out.wait_event(ev_done[i])
        with torch.cuda.stream(s_out):
            dqkv_host.copy_(g_d, non_blocking=True)
            ev_out[i].record(s_out)
    stream.wait_event(ev_out[0])
    stream.wait_event(ev_out[1])
    e_end.record(stream)
    barrier()
    res.update({"e2e_ms": e_start.elapsed_time(e_end) / e2e_steps, "e2e_steps": e2e_steps,
                "h2d_bytes": (qkv_host.numel() + dout_host.numel()) * esz, "d2h_bytes": dqkv_host.numel() * esz})
    return res


def summarise(w, world, r, peaks, peak_src, dtype="bf16"):
    """Whole-job throughput, peak fraction, kernel table and roofline of one
    timed workload (r from time_workload, times already max-reduced)."""
    prof = r["prof"]
    fl = flops_per_step(w)
    value = world * fl / (r["ms_per_step"] * 1e-3) / 1e12
    peak_tf, peak_desc = choose_peak(peaks, peak_src, r["timed_s"], dtype)
    roof, combined = roofline_of(prof, w, peak_tf, peak_desc)
    kernel_ms = {k: v[1] for k, v in prof.items()}
    return {
        "value": value, "ms_per_step": r["ms_per_step"], "steps": r["steps"],
        f"peak_{dtype}_frac": value / world / peak_tf, f"peak_{dtype}_tflops": peak_tf, "peak_source": peak_desc,
        "wall_s_timed_region": r["wall"], "clocks": r["clocks"],
        "kernels": {k: {"launches": v[0], "avg_ms": v[1] / v[0], "share": v[1] / sum(kernel_ms.values())}
                    for k, v in prof.items()},
        "gpu_launches": int(round(sum(v[0] for v in prof.values()) / r["n_prof"] * r["steps"])),
        "roofline": roof, "bwd_combined": combined,
    }


def run_ours(args, w):
    import torch
    import torch.distributed as dist
    from causal_attention_gqa_gb300 import binding
    from causal_attention_gqa_gb300.workloads import WORKLOADS, rank_shard

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    binding.load()

    # The headline workload, then (default run) the long-context GQA workload
    # in the same process: the two GQA bf16 configurations.
    ws = rank_shard(w, rank, world)     # this rank's batch rows of the global batch
    head = time_workload(args, ws, dev, world, args.steps, e2e=True)
    extra = {}
    if args.also and args.also != w.name and args.dtype == "bf16":
        wa = WORKLOADS[args.also]
        extra[wa.name] = (wa, time_workload(args, rank_shard(wa, rank, world), dev, world,
                                            min(args.steps, args.also_steps), e2e=False))
    head["ms_per_step"], head["e2e_ms"] = max_over_ranks([head["ms_per_step"], head["e2e_ms"]], dev)
    for name, (wa, r) in extra.items():
        (r["ms_per_step"],) = max_over_ranks([r["ms_per_step"]], dev)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    s = summarise(ws, world, head, peaks, peak_src, args.dtype)
    fl = flops_per_step(ws)
    e2e_value = world * fl / (head["e2e_ms"] * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": s["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": s["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 (TF32 path: three bf16 products per float32 product)"
        if args.dtype == "tf32" else "bf16", "data": "synthetic",
        "config": config_of(ws, {"parallelism": f"batch rows sharded over {world} ranks, no collective"
                                 if world > 1 else "single GPU", "global_batch": world * ws.B,
                                 "rope_pairs": "interleaved (GPT-J)" if args.rope_interleaved else "NEOX",
                                 "l2": "flushed between timed steps (256 MiB write outside the timed events)",
                                 "kernel_breakdown": f"separate pass of {head['n_prof']} steps with per-kernel "
                                                     "events",
                                 f"peak_{args.dtype}_frac": s[f"peak_{args.dtype}_frac"],
                                 f"peak_{args.dtype}_tflops": s[f"peak_{args.dtype}_tflops"],
                                 "peak_source": s["peak_source"],
                                 "measured_peaks": {k: peaks.get(k) for k in
                                                    ("bf16_tflops", "bf16_tflops_sustained", "hbm_gbs")},
                                 "wall_s_timed_region": s["wall_s_timed_region"]}),
        "clocks": s["clocks"],
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": head["h2d_bytes"],
                "d2h_bytes_per_step": head["d2h_bytes"], "ms_per_step": head["e2e_ms"],
                "steps": head["e2e_steps"],
                "copies": "pinned host buffers; h2d and d2h on two copy streams overlapping the neighbouring "
                          "steps' kernels (two device buffer sets); L2 not flushed"},
        "gpu_launches": s["gpu_launches"],
        "kernels": s["kernels"],
        "roofline": s["roofline"],
        "bwd_combined": s["bwd_combined"],
    }
    if extra:
        line["per_config"] = {}
        for name, (wa, r) in extra.items():
            sa = summarise(rank_shard(wa, rank, world), world, r, peaks, peak_src)
            sa["config"] = config_of(rank_shard(wa, rank, world))
            line["per_config"][name] = sa
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = {k: v for k, v in time_oracle(ws).items() if k != "seconds"}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_decode(args):
    """attn_decode on a seeded bf16 cache (all rows visible); HBM GB/s."""
    import torch
    from causal_attention_gqa_gb300 import binding
    from causal_attention_gqa_gb300.workloads import make_decode_inputs
    B, L, NH, NKV, hd = (int(x) for x in args.decode.split(","))
    torch.cuda.set_device(0)
    binding.load()
    q_np, k_np, v_np = make_decode_inputs(B, NH, NKV, hd, L, "bf16", seed=2024)
    q = torch.from_numpy(q_np).to("cuda", torch.bfloat16)
    k = torch.from_numpy(k_np).to("cuda", torch.bfloat16)
    v = torch.from_numpy(v_np).to("cuda", torch.bfloat16)
    del q_np, k_np, v_np
    lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    nbytes = binding.attn_decode_workspace_bytes(B, NH, NKV, hd, L, binding.DTYPE_BF16)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((B, NH), dtype=torch.float32, device="cuda")
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def call():
        binding.attn_decode(out, lse, q, k, v, lens, B, NH, NKV, hd, L, binding.DTYPE_BF16, ws, nbytes)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    steps = min(args.steps, 200)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(0)
    for a, b in ev:
        flush.zero_()
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    cache_bytes = 2 * B * L * NKV * hd * 2
    io_bytes = cache_bytes + 2 * B * NH * hd * 2 + B * NH * 4
    peaks, src = load_peaks()
    gbs = io_bytes / (ms * 1e-3) / 1e9
    line = {
        "metric": "decode attention HBM GB/s on 1 GB300", "value": gbs, "unit": "GB/s", "n_gpus": 1,
        "steps": steps, "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "decode", "B": B, "L": L, "NH": NH, "NKV": NKV, "hd": hd,
                   "l2": "flushed between calls (256 MiB write outside the timed events)",
                   "timing": "median of per-call CUDA events"},
        "clocks": clocks,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                     "peak_source": f"{src} hbm_gbs (copy)", "algorithmic_bytes_per_launch": io_bytes},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_proj(args):
    """attn_qkv_proj on seeded bf16 inputs; TFLOP/s of the GEMM."""
    import torch
    from causal_attention_gqa_gb300 import binding
    from causal_attention_gqa_gb300.workloads import make_proj_inputs
    B, T, Cm, NH, NKV, hd = (int(v) for v in args.proj.split(","))
    torch.cuda.set_device(0)
    binding.load()
    M, N = B * T, (NH + 2 * NKV) * hd
    x_np, w_np = make_proj_inputs(M, Cm, N, seed=2025)
    x = torch.from_numpy(x_np).to("cuda", torch.bfloat16)
    w = torch.from_numpy(w_np).to("cuda", torch.bfloat16)
    qkv = torch.empty((B, T, N), dtype=torch.bfloat16, device="cuda")
    rot = torch.empty((M * (NH + NKV) * hd * 2 + 256,), dtype=torch.uint8, device="cuda")
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    calls = {
        "fused_rope_copy": lambda: binding.attn_qkv_proj(qkv, rot, x, w, B, T, Cm, NH, NKV, hd, 1e6, 0),
        "gemm_only": lambda: binding.attn_qkv_proj(qkv, None, x, w, B, T, Cm, NH, NKV, hd, 0.0, 0),
        "cublas_context": lambda: torch.matmul(x, w.t(), out=qkv.view(M, N)),
    }
    steps = min(args.steps, 100)
    res = {}
    for name, fn in calls.items():
        for _ in range(max(3, args.warmup)):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in ev:
            flush.zero_()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        ms = statistics.median(a.elapsed_time(b) for a, b in ev)
        res[name] = {"ms": ms, "tflops": 2.0 * M * N * Cm / (ms * 1e-3) / 1e12}
    peaks, src = load_peaks()
    v = res["fused_rope_copy"]["tflops"]
    line = {
        "metric": "QKV projection (+ rotated Q/K copy) TFLOP/s on 1 GB300", "value": v, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": steps, "warmup": max(3, args.warmup), "ms_per_step": res["fused_rope_copy"]["ms"],
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "qkv_projection", "B": B, "T": T, "Cm": Cm, "NH": NH, "NKV": NKV, "hd": hd,
                   "l2": "flushed between calls (256 MiB write outside the timed events)"},
        "variants": res,
        "roofline": {"bound": "tensor", "achieved": v, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": v / peaks["bf16_tflops"],
                     "traffic": traffic_for("proj", "qkv_projection_" + args.proj.replace(",", "_")),
                     "peak_source": f"{src} bf16_tflops (burst)"},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_fp8(args, w):
    """attn_fwd_fp8 vs attn_fwd_ws on the workload; forward TFLOP/s."""
    import torch
    from causal_attention_gqa_gb300 import binding
    from causal_attention_gqa_gb300.workloads import make_inputs
    torch.cuda.set_device(0)
    binding.load()
    B, T, C, NH, NKV = w.B, w.T, w.C, w.NH, w.NKV
    qkv_np, _ = make_inputs(w, "bf16")
    qkv = torch.from_numpy(qkv_np).to("cuda", torch.bfloat16)
    del qkv_np
    out = torch.empty((B, T, C), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, NH, T), dtype=torch.float32, device="cuda")
    code = binding.DTYPE_BF16
    nb8 = binding.attn_fwd_fp8_workspace_bytes(B, T, C, NH, NKV, code)
    ws8 = torch.empty(nb8, dtype=torch.uint8, device="cuda")
    nbw = binding.attn_fwd_workspace_bytes(B, T, C, NH, NKV, code)
    wsw = torch.empty(nbw, dtype=torch.uint8, device="cuda")
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    calls = {
        "fp8": lambda: binding.attn_fwd_fp8(out, lse, qkv, B, T, C, NH, NKV, w.rope_theta, code, ws8, nb8),
        "bf16_ws": lambda: binding.attn_fwd_ws(out, lse, qkv, B, T, C, NH, NKV, w.rope_theta, code, wsw, nbw),
    }
    steps = min(args.steps, 200)
    res = {}
    for name, fn in calls.items():
        for _ in range(max(3, args.warmup)):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in ev:
            flush.zero_()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        ms = statistics.median(a.elapsed_time(b) for a, b in ev)
        res[name] = {"ms": ms, "tflops": w.flops_fwd() / (ms * 1e-3) / 1e12}
    binding.attn_profile_start()
    for _ in range(20):
        flush.zero_()
        calls["fp8"]()
    torch.cuda.synchronize()
    prof = binding.attn_profile_stop()
    peaks, src = load_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    v = res["fp8"]["tflops"]
    kern = {k: {"launches": n, "avg_ms": t / n} for k, (n, t) in prof.items()}
    fk = kern.get("fwd_fp8", {}).get("avg_ms")
    line = {
        "metric": "causal attn forward TFLOP/s with e4m3 operands on 1 GB300", "value": v, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": steps, "warmup": max(3, args.warmup), "ms_per_step": res["fp8"]["ms"],
        "higher_is_better": True, "dtype": "e4m3 (bf16 in/out)", "data": "synthetic",
        "config": config_of(w, {"l2": "flushed between calls (256 MiB write outside the timed events)",
                                "timing": "median of per-call CUDA events"}),
        "variants": res, "kernels": kern,
        "roofline": {"bound": "tensor", "kernel": "fwd_fp8",
                     "achieved": (w.flops_fwd() / (fk * 1e-3) / 1e12) if fk else None, "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": (w.flops_fwd() / (fk * 1e-3) / 1e12 / fp8_peak) if fk else None,
                     "traffic": None, "peak_source": f"2 x {src} bf16_tflops (burst), the nominal fp8/bf16 ratio"},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.fp8:
        from causal_attention_gqa_gb300.workloads import WORKLOADS
        return run_fp8(args, WORKLOADS[args.workload])
    if args.decode:
        return run_decode(args)
    if args.proj:
        return run_proj(args)
    from causal_attention_gqa_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
