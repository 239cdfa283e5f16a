#!/usr/bin/env python
"""MoDA benchmark: one step = the whole hot path (forward + backward) on one batch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints ONE JSON line (rank 0).  Our arm times K steps of moda_fwd + moda_bwd on
device-resident synthetic inputs with CUDA events (max over ranks), then the same
step end to end through the C ABI with pinned host buffers (H2D of the inputs,
D2H of every output, inside the timed region).  The reference arm times the
float64 CPU oracle on a bounded sample of the same workload.

Under torchrun each rank runs an independent replica on its own GPU (the units,
(batch, kv-head) problems, are independent: no data-path collective), so the
reported value is the aggregate over ranks ("weak" scaling).
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
sys.path.insert(0, ROOT)

METRIC = "MoDA fwd/bwd TFLOP/s and fraction of roofline (tensor peak vs HBM), 1×GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- counts
def flops(shape):
    """Algorithmic FLOPs: causal sequence part 4*B*H*d*T(T+1)/2 (QK^T and PV over the
    visible triangle), depth part 4*B*H*T*S*d; backward counted as 2.5x forward."""
    B, H, T, d, S = shape.B, shape.H, shape.T, shape.d, shape.S
    seq = 4.0 * B * H * d * T * (T + 1) / 2
    depth = 4.0 * B * H * T * S * d
    return {"fwd_seq": seq, "fwd_depth": depth, "fwd": seq + depth, "bwd_seq": 2.5 * seq,
            "bwd_depth": 2.5 * depth, "bwd": 2.5 * (seq + depth)}


def bwd_kernel_name(kind, d):
    """Name of the tensor-core backward kernel of `kind` ("dkdv" or "dq") for head size d
    (the d = 64 kernels use 128-wide tiles and have kernels of their own)."""
    return f"moda_bwd_{kind}64_kernel" if d == 64 else f"moda_bwd_{kind}_kernel"


def kernel_counts(shape):
    """Algorithmic FLOPs (tensor-core contractions over the causal triangle; one GEMM is
    2*B*H*d*T(T+1)/2) and HBM bytes (each tensor read or written once) per launch of each
    kernel of the step."""
    e = 2 if shape.dtype_name == "bf16" else 4
    B, H, Hkv, T, d, S = shape.B, shape.H, shape.Hkv, shape.T, shape.d, shape.S
    gemm = 2.0 * B * H * d * T * (T + 1) / 2
    q = B * H * T * d * e
    kv = B * Hkv * T * d * e
    dkv = B * Hkv * T * S * d * e
    row = B * H * T * 4
    qf32 = B * H * T * d * 4
    counts = {
        "moda_fwd_tc_kernel": {"flops": 2 * gemm, "bytes": q + 2 * kv + 2 * dkv + q + row},
        "bwd_delta_kernel": {"flops": 0.0, "bytes": 2 * q + 3 * row},
        # with depth slots the depth kernel also forms Delta = dO . O and the row statistics
        # (reads o and lse, writes {-lse*log2 e, Delta}); there is no separate Delta kernel
        "moda_bwd_depth_kernel": {"flops": 0.0, "bytes": 4 * dkv + 3 * q + 3 * row + qf32},
        bwd_kernel_name("dkdv", d): {"flops": 4 * gemm, "bytes": 2 * kv + 2 * q + 2 * row + 2 * kv},
        bwd_kernel_name("dq", d): {"flops": 3 * gemm, "bytes": 2 * q + 2 * kv + 2 * row + qf32 + q},
    }
    if S > 0:
        del counts["bwd_delta_kernel"]
    else:
        del counts["moda_bwd_depth_kernel"]
    return counts


def bytes_moved(shape):
    """Algorithmic HBM bytes: every tensor read or written once (depth KV once per kv head)."""
    e = 2 if shape.dtype_name == "bf16" else 4
    B, H, Hkv, T, d, S = shape.B, shape.H, shape.Hkv, shape.T, shape.d, shape.S
    q = B * H * T * d * e
    kv = 2 * B * Hkv * T * d * e
    dkv = 2 * B * Hkv * T * S * d * e
    dkv_mem = 2 * B * Hkv * T * shape.S_mem * d * e  # dkd/dvd cover every slot in memory
    lse = B * H * T * 4
    fwd = q + kv + dkv + q + lse  # read q, k, v, kd, vd (the S slots read); write o, lse
    bwd = (q + kv + dkv + q + q + lse) + (q + kv + dkv_mem)  # read q,k,v,kd,vd,o,dout,lse; write dq..dvd
    return {"fwd": fwd, "bwd": bwd, "inputs": q + kv + dkv_mem + q, "outputs": q + lse + q + kv + dkv_mem}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def traffic_record(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged
    since the counters were taken (lines: kernel workload bytes source-sha256-prefix)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    for line in lines:
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload:
            if parts[3] == source_digest(kernel):
                return float(parts[2])
    return None


KERNEL_SOURCES = {"moda_fwd_tc_kernel": ["moda_fwd_sm103.cu", "sm103_ptx.cuh"],
                  "bwd_delta_kernel": ["moda_simt.cu"],
                  "moda_bwd_depth_kernel": ["moda_bwd_sm103.cu", "sm103_ptx.cuh"],
                  "moda_bwd_dkdv_kernel": ["moda_bwd_sm103.cu", "sm103_ptx.cuh"],
                  "moda_bwd_dq_kernel": ["moda_bwd_sm103.cu", "sm103_ptx.cuh"],
                  "moda_bwd_dkdv64_kernel": ["moda_bwd_sm103.cu", "sm103_ptx.cuh"],
                  "moda_bwd_dq64_kernel": ["moda_bwd_sm103.cu", "sm103_ptx.cuh"],
                  "moda_depth_project_kernel": ["moda_depth_write_sm103.cu", "sm103_ptx.cuh"],
                  "moda_depth_store_kernel": ["moda_depth_write_sm103.cu"]}


def source_digest(kernel):
    h = hashlib.sha256()
    for fn in KERNEL_SOURCES.get(kernel, []):
        p = os.path.join(ROOT, "joint_sequence_depth_gb300", "csrc", fn)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


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
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle
def oracle_sample(shape, T_sample):
    """Bounded sample of the workload for the CPU oracle: batch 0, kv head 0 (its G query
    heads), the first T_sample positions -- itself a valid MoDA problem."""
    import numpy as np
    import torch

    from joint_sequence_depth_gb300.inputs import make_inputs, scaled

    sub = scaled(shape, B=1, H=shape.G, Hkv=1, T=T_sample, slot_capacity=0)  # the S slots read
    x = make_inputs(sub, seed=101, device="cpu", with_dout=True)
    host = [x[n].view(torch.int16).numpy().view(np.uint16) if x[n].dtype == torch.bfloat16 else x[n].numpy()
            for n in ("q", "k", "v", "kd", "vd", "dout")]
    return sub, host


def time_oracle_steps(shape, T_sample, steps):
    import oracle

    oracle.build()
    sub, host = oracle_sample(shape, T_sample)
    f = flops(sub)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.forward(*host[:5])
        oracle.backward(*host)
        times.append(time.perf_counter() - t0)
    per = statistics.mean(times)
    return {"value": (f["fwd"] + f["bwd"]) / per / 1e12, "seconds_per_step": per, "cores": oracle.cores(),
            "sample": f"batch 0, kv head 0 ({sub.H} query heads), positions 0..{T_sample - 1}, "
                      f"S={sub.S}, d={sub.d}: forward + backward ({(f['fwd'] + f['bwd']) / 1e9:.1f} GFLOP)"}


# ----------------------------------------------------------------------------- main
def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="bf16_train")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=8)
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(workload, rank):
    """Each rank draws its own batch: replicas work on independent problems."""
    from joint_sequence_depth_gb300.inputs import SEEDS

    return SEEDS[workload] + 1000 * rank


def max_over_ranks(values, device):
    """Element-wise maximum over all ranks (the slowest rank sets every time)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def aggregate_tflops(step_flops, ms_per_step, world):
    """Whole-job throughput: every rank processed step_flops per step in ms_per_step."""
    return world * step_flops / (ms_per_step * 1e-3) / 1e12


def run_reference(args, shape):
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    steps, warm = max(1, args.steps), max(0, args.warmup)
    T_sample = 1024
    time_oracle_steps(shape, T_sample, warm) if warm else None
    r = time_oracle_steps(shape, T_sample, steps)
    line = {"impl": "reference", "metric": METRIC, "value": r["value"], "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": steps, "warmup": warm, "ms_per_step": r["seconds_per_step"] * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(shape),
            "cpu_baseline": {"value": r["value"], "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle",
                             "sample": r["sample"]},
            "e2e": {"value": r["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(shape):
    ring = f" read of {shape.S_mem} in memory (bounded slot buffer)" if shape.slot_capacity else ""
    cfg = {"workload": f"{shape.name}: B={shape.B} H={shape.H} Hkv={shape.Hkv} T={shape.T} d={shape.d} "
                       f"S={shape.S}{ring} {shape.dtype_name}, causal, forward+backward",
           "global_batch": shape.B, "seq_len": shape.T, "depth_slots": shape.S,
           "l2": "inputs larger than L2 (no flush)"}
    if shape.slot_capacity:
        cfg["slot_capacity"] = shape.slot_capacity
    return cfg


DECODE_METRIC = "MoDA decode step GB/s and fraction of the HBM roofline, 1\u00d7GB300"


def decode_bytes(shape):
    """Algorithmic HBM bytes of one decode step: the sequence cache (K, V) and the depth
    slots read once for the G heads of their kv head, q read, o and lse written."""
    e = 2
    B, H, Hkv, T, d, S = shape.B, shape.H, shape.Hkv, shape.T, shape.d, shape.S
    return 2 * B * Hkv * T * d * e + 2 * B * Hkv * S * d * e + 2 * B * H * d * e + 4 * B * H


def decode_config(shape):
    return {"workload": f"{shape.name}: B={shape.B} H={shape.H} Hkv={shape.Hkv} cached T={shape.T} d={shape.d} "
                        f"S={shape.S} {shape.dtype_name}, one decode step",
            "global_batch": shape.B, "seq_len": shape.T, "depth_slots": shape.S,
            "l2": "K/V cache larger than L2 (no flush)"}


def time_oracle_decode(shape, groups):
    """The float64 oracle on `groups` (batch, kv head) groups of the decode step."""
    import numpy as np
    import oracle
    import torch
    from joint_sequence_depth_gb300.inputs import DECODE_SEEDS, Shape, make_decode_inputs

    sub = Shape(shape.name, 1, shape.G, 1, shape.T, shape.d, shape.S, shape.dtype)
    x = make_decode_inputs(sub, seed=DECODE_SEEDS[shape.name])
    host = [x[n].view(torch.int16).numpy().view(np.uint16) for n in ("q", "k", "v", "kd", "vd")]
    t0 = time.perf_counter()
    for _ in range(groups):
        oracle.decode(*host)
    per_group = (time.perf_counter() - t0) / groups
    by = decode_bytes(sub)
    return {"value": by / per_group / 1e9, "seconds_per_group": per_group, "cores": 1,
            "sample": f"{groups} (batch, kv head) groups of {shape.G} query heads, T={shape.T}, S={shape.S}, "
                      f"d={shape.d} ({by / 1e6:.1f} MB each); numpy float64 on one core"}


def run_decode(args, shape):
    """Decode-step benchmark: device time of moda_decode with the cache resident in HBM;
    e2e adds the step's own inputs (q, kd, vd) from pinned host memory and its outputs
    (o, lse) back, the cache staying on the device."""
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        if rank != 0:
            return 0
        steps = max(1, args.steps)
        r = time_oracle_decode(shape, steps)
        ms = r["seconds_per_group"] * shape.B * shape.Hkv * 1e3
        line = {"impl": "reference", "metric": DECODE_METRIC, "value": r["value"], "unit": "GB/s",
                "n_gpus": args.gpus, "steps": steps, "warmup": 0, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": decode_config(shape),
                "cpu_baseline": {"value": r["value"], "unit": "GB/s", "cores": r["cores"], "kind": "oracle",
                                 "sample": r["sample"]},
                "e2e": {"value": r["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0
    import torch
    import torch.distributed as dist

    from joint_sequence_depth_gb300 import binding
    from joint_sequence_depth_gb300 import build as mbuild
    from joint_sequence_depth_gb300.inputs import DECODE_SEEDS, make_decode_inputs

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mbuild.build()
    binding.load_library()
    x = make_decode_inputs(shape, seed=DECODE_SEEDS[shape.name] + 1000 * rank, device=dev)
    o = torch.empty_like(x["q"])
    lse = torch.empty(shape.B, shape.H, dtype=torch.float32, device=dev)
    desc = binding.make_desc(shape.B, shape.H, shape.Hkv, shape.T, shape.S, shape.d, shape.dtype)
    ws = torch.empty(binding.moda_decode_workspace_bytes(desc), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        binding.moda_decode(x["q"], x["k"], x["v"], x["kd"], x["vd"], o=o, lse=lse, workspace=ws)

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    K = args.steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    launches0 = binding.moda_launch_count()
    ev[0].record(stream)
    for i in range(K):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    launches = binding.moda_launch_count() - launches0
    clk = clocks.stop()
    total_ms = ev[0].elapsed_time(ev[K])
    status = binding.moda_device_status()
    if status != 0:
        raise RuntimeError(f"device status {binding.STATUS_NAMES.get(status, status)} after the timed steps")
    # end to end: the step's own inputs in from pinned host memory, outputs back
    names = ("q", "kd", "vd")
    host_in = {n: x[n].cpu().pin_memory() for n in names}
    host_o = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    host_l = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    E = max(3, args.e2e_steps)
    for _ in range(2):
        for n in names:
            x[n].copy_(host_in[n], non_blocking=True)
        step()
        host_o.copy_(o, non_blocking=True)
        host_l.copy_(lse, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E):
        for n in names:
            x[n].copy_(host_in[n], non_blocking=True)
        step()
        host_o.copy_(o, non_blocking=True)
        host_l.copy_(lse, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / E
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_o.numel() * host_o.element_size() + host_l.numel() * host_l.element_size()
    ms_per_step, e2e_ms = max_over_ranks([total_ms / K, e2e_ms], dev)
    by = decode_bytes(shape)
    value = world * by / (ms_per_step * 1e-3) / 1e9
    peaks, peak_kind = load_peaks()
    roof = {"bound": "hbm", "achieved": by / (ms_per_step * 1e-3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof.update({"traffic": None, "kernel": "moda_decode_kernel (+ moda_decode_merge_kernel)",
                 "peak_source": f"{peak_kind} (copy)", "algorithmic": {"flops": 0.0, "bytes": by},
                 "ms": ms_per_step})
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = time_oracle_decode(shape, 4)
        cpu = {"value": r["value"], "unit": "GB/s", "cores": r["cores"], "kind": "oracle", "sample": r["sample"]}
    if rank == 0:
        line = {"metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
                "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": shape.dtype_name, "data": "synthetic",
                "config": decode_config(shape), "clocks": clk,
                "e2e": {"value": world * by / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
                "gpu_launches": launches, "roofline": roof, "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


WRITE_METRIC = "MoDA depth-KV write (slot store + FFN-input projection) TFLOP/s and fraction of roofline, 1\u00d7GB300"


def write_counts(shape):
    """Algorithmic work of one layer's depth-KV write: the attention K, V copied into one
    slot, and x [B,T,Dm] projected by wk, wv [Dm,Hkv*d] into another."""
    from joint_sequence_depth_gb300.inputs import d_model

    e = 2
    B, Hkv, T, d = shape.B, shape.Hkv, shape.T, shape.d
    Dm = d_model(shape)
    n = Hkv * d
    return {"flops": 2.0 * 2 * B * T * Dm * n,
            "store_bytes": 4.0 * B * Hkv * T * d * e,
            "project_bytes": float(B * T * Dm * e + 2 * Dm * n * e + 2 * B * T * n * e)}


def write_config(shape):
    from joint_sequence_depth_gb300.inputs import d_model

    return {"workload": f"{shape.name}: B={shape.B} Hkv={shape.Hkv} T={shape.T} d={shape.d} S={shape.S} "
                        f"d_model={d_model(shape)} {shape.dtype_name}, one layer's depth-KV write "
                        f"(store into slot S-1, projection into slot S/2)",
            "global_batch": shape.B, "seq_len": shape.T, "depth_slots": shape.S,
            "l2": "L2 flushed between steps (256 MiB write, then 256 MiB read, outside the timed events)"}


def time_oracle_write(shape, T_sample, steps):
    """The float64 oracle's store + projection on batch 0, positions 0..T_sample-1."""
    import numpy as np
    import torch

    import oracle
    from joint_sequence_depth_gb300.inputs import WRITE_SEEDS, make_write_inputs, scaled

    sub = scaled(shape, B=1, T=T_sample)
    x = make_write_inputs(sub, seed=WRITE_SEEDS[shape.name])
    h = {n: t.view(torch.int16).numpy().view(np.uint16) for n, t in x.items()}
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.depth_store(h["k"], h["v"], h["kd"], h["vd"], shape.S - 1)
        oracle.depth_project(h["x"], h["wk"], h["wv"], h["kd"], h["vd"], shape.S // 2)
    per = (time.perf_counter() - t0) / steps
    f = write_counts(sub)["flops"]
    return {"value": f / per / 1e12, "seconds_per_step": per, "cores": os.cpu_count() or 1,
            "sample": f"batch 0, positions 0..{T_sample - 1}, all {shape.Hkv} kv heads, S={shape.S}: "
                      f"store + projection ({f / 1e9:.2f} GFLOP); numpy float64, BLAS may use every host core"}


def run_write(args, shape):
    """Depth-KV write benchmark: one step = moda_depth_store_kv + moda_depth_project_kv on
    device-resident inputs, L2 flushed between steps; e2e adds the layer's own inputs
    (k, v, x) from pinned host memory and reads back the written slots of the last position."""
    world, rank, local = dist_setup(args)
    T_sample = max(128, shape.T // 32)
    if args.impl == "reference":
        if rank != 0:
            return 0
        steps = max(1, args.steps)
        r = time_oracle_write(shape, T_sample, steps)
        ms = r["seconds_per_step"] * shape.B * (shape.T / T_sample) * 1e3
        line = {"impl": "reference", "metric": WRITE_METRIC, "value": r["value"], "unit": "TFLOP/s",
                "n_gpus": args.gpus, "steps": steps, "warmup": 0, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": write_config(shape),
                "cpu_baseline": {"value": r["value"], "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle",
                                 "sample": r["sample"]},
                "e2e": {"value": r["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0
    import torch
    import torch.distributed as dist

    from joint_sequence_depth_gb300 import binding
    from joint_sequence_depth_gb300 import build as mbuild
    from joint_sequence_depth_gb300.inputs import WRITE_SEEDS, make_write_inputs

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mbuild.build()
    binding.load_library()
    x = make_write_inputs(shape, seed=WRITE_SEEDS[shape.name] + 1000 * rank, device=dev)
    S = shape.S
    slot_store, slot_proj = S - 1, S // 2
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    clean = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def flush_l2():
        # write 256 MiB (evicts the inputs), then read 256 MiB of another buffer so that the
        # flush's own dirty lines are written back here and not inside the next timed kernel
        flush.zero_()
        clean.sum()

    def step():
        binding.moda_depth_store_kv(x["k"], x["v"], x["kd"], x["vd"], slot_store)
        binding.moda_depth_project_kv(x["x"], x["wk"], x["wv"], x["kd"], x["vd"], slot_proj)

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(max(3, args.warmup)):
        flush_l2()
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    launches0 = binding.moda_launch_count()
    for i in range(K):
        flush_l2()
        ev[i][0].record(stream)
        binding.moda_depth_store_kv(x["k"], x["v"], x["kd"], x["vd"], slot_store)
        ev[i][1].record(stream)
        binding.moda_depth_project_kv(x["x"], x["wk"], x["wv"], x["kd"], x["vd"], slot_proj)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    launches = binding.moda_launch_count() - launches0
    clk = clocks.stop()
    store_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    proj_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    status = binding.moda_device_status()
    if status != 0:
        raise RuntimeError(f"device status {binding.STATUS_NAMES.get(status, status)} after the timed steps")
    names = ("k", "v", "x")
    host_in = {n: x[n].cpu().pin_memory() for n in names}
    host_kd = torch.empty(shape.B, shape.Hkv, 2, shape.d, dtype=x["kd"].dtype, pin_memory=True)
    host_vd = torch.empty_like(host_kd, pin_memory=True)
    slots = [slot_proj, slot_store]

    def e2e_step():
        for n in names:
            x[n].copy_(host_in[n], non_blocking=True)
        step()
        host_kd.copy_(x["kd"][:, :, shape.T - 1, slots], non_blocking=True)
        host_vd.copy_(x["vd"][:, :, shape.T - 1, slots], non_blocking=True)

    E = max(3, args.e2e_steps)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / E
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = 2 * host_kd.numel() * host_kd.element_size()
    ms_per_step, e2e_ms, proj_ms, store_ms = max_over_ranks([store_ms + proj_ms, e2e_ms, proj_ms, store_ms], dev)
    c = write_counts(shape)
    value = world * c["flops"] / (ms_per_step * 1e-3) / 1e12
    peaks, peak_kind = load_peaks()
    roof = {"bound": "tensor", "achieved": c["flops"] / (proj_ms * 1e-3) / 1e12, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof.update({"traffic": traffic_record("moda_depth_project_kernel", shape.name),
                 "kernel": "moda_depth_project_kernel", "peak_source": f"{peak_kind} bf16 burst (cuBLAS)",
                 "algorithmic": {"flops": c["flops"], "bytes": c["project_bytes"]}, "ms": proj_ms,
                 "store_kernel": {"kernel": "moda_depth_store_kernel", "ms": store_ms, "bound": "hbm",
                                  "achieved": c["store_bytes"] / (store_ms * 1e-3) / 1e9,
                                  "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": c["store_bytes"] / (store_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}})
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = time_oracle_write(shape, T_sample, 3)
        cpu = {"value": r["value"], "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle", "sample": r["sample"]}
    if rank == 0:
        line = {"metric": WRITE_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
                "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": shape.dtype_name, "data": "synthetic",
                "config": write_config(shape), "clocks": clk,
                "e2e": {"value": world * c["flops"] / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
                "gpu_launches": launches, "roofline": roof, "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


CP_METRIC = ("MoDA context-parallel fwd/bwd TFLOP/s (every rank's chunk pairs run in turn on one GPU) "
             "and fraction of roofline, 1\u00d7GB300")
# workload -> (problem, ranks simulated, chunk layout)
CP_WORKLOADS = {"bf16_cp2_train": ("bf16_train", 2, "zigzag"), "bf16_cp4_train": ("bf16_train", 4, "zigzag")}


def run_cp(args, name):
    """Context-parallel pieces on one GPU: one step runs, rank after rank, every chunk pair
    of the ring schedule through moda_fwd_partial / moda_merge_partial / moda_bwd_partial /
    moda_convert_f32 (the exchange is a change of references, no kernel waits on another
    rank).  value = the whole problem's FLOPs / step time, comparable with the unchunked
    step.  Also timed alone: one fully visible chunk pair's partial forward (tensor-bound)
    and one merge (HBM-bound)."""
    base_name, ranks, layout = CP_WORKLOADS[name]
    from joint_sequence_depth_gb300.inputs import WORKLOADS

    base = WORKLOADS[base_name]
    world, rank, local = dist_setup(args)
    cfg = {"workload": f"{name}: {base_name} (B={base.B} H={base.H} Hkv={base.Hkv} T={base.T} d={base.d} "
                       f"S={base.S} {base.dtype_name}) split over {ranks} ranks ({layout} chunks), "
                       f"every rank's pairs on this GPU, forward+backward",
           "global_batch": base.B, "seq_len": base.T, "depth_slots": base.S, "cp_ranks": ranks,
           "l2": "inputs larger than L2 (no flush)"}
    if args.impl == "reference":
        if rank != 0:
            return 0
        steps, warm = max(1, args.steps), max(0, args.warmup)
        time_oracle_steps(base, 1024, warm) if warm else None
        r = time_oracle_steps(base, 1024, steps)
        line = {"impl": "reference", "metric": CP_METRIC, "value": r["value"], "unit": "TFLOP/s",
                "n_gpus": args.gpus, "steps": steps, "warmup": warm, "ms_per_step": r["seconds_per_step"] * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": cfg,
                "cpu_baseline": {"value": r["value"], "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle",
                                 "sample": r["sample"]},
                "e2e": {"value": r["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0
    import torch
    import torch.distributed as dist

    from joint_sequence_depth_gb300 import binding
    from joint_sequence_depth_gb300 import build as mbuild
    from joint_sequence_depth_gb300 import context_parallel as cp
    from joint_sequence_depth_gb300.inputs import make_inputs

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mbuild.build()
    binding.load_library()
    x = make_inputs(base, seed=rank_seed(base_name, rank), device=dev, with_dout=True)
    names = ("q", "k", "v", "kd", "vd", "dout")
    owned = cp.chunks_of(base.T, ranks, layout)
    loc = {n: [[x[n].narrow(2, c.start, c.length).contiguous() for c in owned[r]] for r in range(ranks)]
           for n in names}
    kern = cp.LibraryKernels()
    stream = torch.cuda.current_stream()

    def step(inp):
        o, lse = cp.simulate_ring_forward(inp["q"], inp["k"], inp["v"], inp["kd"], inp["vd"], base.T, ranks,
                                          layout, kernels=kern)
        grads = cp.simulate_ring_backward(inp["q"], inp["k"], inp["v"], inp["kd"], inp["vd"], o, lse, inp["dout"],
                                          base.T, ranks, layout, kernels=kern)
        return o, lse, grads

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(max(3, args.warmup)):
        step(loc)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = binding.moda_launch_count()
    e0.record(stream)
    for _ in range(K):
        step(loc)
    e1.record(stream)
    torch.cuda.synchronize()
    launches = binding.moda_launch_count() - launches0
    clk = clocks.stop()
    if binding.moda_device_status() != 0:
        raise RuntimeError("device status set after the timed steps")
    ms_step = e0.elapsed_time(e1) / K
    # one fully visible chunk pair (query chunk ranks..., key chunk 0) and one merge, alone
    c_q, c_k = owned[ranks - 1][0], owned[0][0]
    qq = loc["q"][ranks - 1][0]
    kk, vv = loc["k"][0][0], loc["v"][0][0]
    delta = c_q.start - c_k.start
    o_p, l_p = binding.moda_fwd_partial(qq, kk, vv, None, None, delta)
    o_acc = torch.empty(qq.shape, dtype=torch.float32, device=dev)
    l_acc = torch.empty(qq.shape[:3], dtype=torch.float32, device=dev)
    binding.moda_merge_partial(o_acc, l_acc, o_p, l_p, first=True)
    reps = 20
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    tp, tm = [], []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        binding.moda_fwd_partial(qq, kk, vv, None, None, delta, o=o_p, lse=l_p)
        b.record(stream)
        flush.zero_()
        c, d_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c.record(stream)
        binding.moda_merge_partial(o_acc, l_acc, o_p, l_p)
        d_.record(stream)
        torch.cuda.synchronize()
        tp.append(a.elapsed_time(b))
        tm.append(c.elapsed_time(d_))
    del flush
    ms_pair, ms_merge = statistics.median(tp), statistics.median(tm)
    peaks, peak_kind = load_peaks()
    pair_flops = 4.0 * base.B * base.H * base.d * c_q.length * c_k.length
    e = 2
    rows = base.B * base.H * c_q.length
    merge_bytes = rows * base.d * (4 + 4 + e) + rows * 4 * 3
    roof = {"bound": "tensor", "achieved": pair_flops / (ms_pair * 1e-3) / 1e12, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof.update({"traffic": None, "kernel": "moda_fwd_tc_kernel (one fully visible chunk pair, no depth slots)",
                 "peak_source": f"{peak_kind} (bf16 burst, cuBLAS)", "ms": ms_pair,
                 "algorithmic": {"flops": pair_flops, "bytes": None}})
    merge = {"bound": "hbm", "achieved": merge_bytes / (ms_merge * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
             "unit": "GB/s", "ms": ms_merge, "bytes": merge_bytes}
    merge["frac"] = merge["achieved"] / merge["peak"]
    # end to end: the inputs from pinned host memory into the chunks, every output back
    host = {n: [[t.cpu().pin_memory() for t in per] for per in loc[n]] for n in names}
    E = max(3, args.e2e_steps)

    def e2e_step():
        for n in names:
            for r in range(ranks):
                for t_dev, t_host in zip(loc[n][r], host[n][r]):
                    t_dev.copy_(t_host, non_blocking=True)
        o, lse, grads = step(loc)
        outs = [t for per in o for t in per] + [t for per in lse for t in per]
        for g in grads:
            outs += [t for per in g for t in per if t is not None]
        return [t.to("cpu", non_blocking=True) for t in outs]

    e2e_step()
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(E):
        back = e2e_step()
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = f0.elapsed_time(f1) / E
    h2d = sum(t.numel() * t.element_size() for n in names for per in host[n] for t in per)
    d2h = sum(t.numel() * t.element_size() for t in back)
    ms_step, e2e_ms = max_over_ranks([ms_step, e2e_ms], dev)
    fl = flops(base)
    total = fl["fwd"] + fl["bwd"]
    if rank == 0:
        line = {"metric": CP_METRIC, "value": aggregate_tflops(total, ms_step, world), "unit": "TFLOP/s",
                "n_gpus": world, "steps": K, "warmup": max(3, args.warmup), "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": base.dtype_name,
                "data": "synthetic", "config": cfg, "clocks": clk,
                "e2e": {"value": aggregate_tflops(total, e2e_ms, world), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
                "gpu_launches": launches, "roofline": roof, "merge": merge, "cpu_baseline": None}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def kernel_roofline(count, ms, peaks):
    """Roofline of one kernel launch: its algorithmic FLOPs against the burst bf16 peak or
    its algorithmic bytes against the copy bandwidth, whichever takes longer."""
    fl, by = count["flops"], count["bytes"]
    if fl / (peaks["bf16_tflops"] * 1e12) >= by / (peaks["hbm_gbs"] * 1e9):
        r = {"bound": "tensor", "achieved": fl / (ms * 1e-3) / 1e12, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        r = {"bound": "hbm", "achieved": by / (ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r["ms"] = ms
    r["algorithmic"] = {"flops": fl, "bytes": by}
    return r


FORWARD_CONFIGS = ("fp32_small", "bf16_mha", "bf16_gqa", "bf16_long", "bf16_train")


def time_forward_configs(dev, peaks, reps=20):
    """moda_fwd alone on every configuration, with its depth slots and with S = 0: median of
    `reps` launches timed by CUDA events, the L2 flushed (256 MiB written) before each.
    Roofline of a configuration: max(causal FLOPs / bf16 burst peak, bytes / copy bandwidth)
    with bytes = q, k, v, kd, vd read and o, lse written once."""
    import torch

    from joint_sequence_depth_gb300 import binding
    from joint_sequence_depth_gb300.inputs import SEEDS, WORKLOADS, make_inputs, scaled

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    out = {}
    for name in FORWARD_CONFIGS:
        rec = {}
        for tag, sh in (("", WORKLOADS[name]), ("s0_", scaled(WORKLOADS[name], S=0, slot_capacity=0))):
            x = make_inputs(sh, seed=SEEDS[name], device=dev, with_dout=False)
            kd, vd = (x["kd"], x["vd"]) if sh.S > 0 else (None, None)
            o = torch.empty_like(x["q"])
            lse = torch.empty(sh.B, sh.H, sh.T, dtype=torch.float32, device=dev)

            def fwd():
                binding.moda_fwd(x["q"], x["k"], x["v"], kd, vd, o, lse)

            for _ in range(3):
                fwd()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for e0, e1 in ev:
                flush.zero_()
                e0.record(stream)
                fwd()
                e1.record(stream)
            torch.cuda.synchronize()
            if binding.moda_device_status() != 0:
                raise RuntimeError(f"device status after the forward of {name}")
            ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
            f = flops(sh)
            by = bytes_moved(sh)["fwd"]
            roof_ms = max(f["fwd_seq"] / (peaks["bf16_tflops"] * 1e12), by / (peaks["hbm_gbs"] * 1e9)) * 1e3
            rec[tag + "ms"] = ms
            rec[tag + "roofline_ms"] = roof_ms
            rec[tag + "frac"] = roof_ms / ms
            if not tag:
                rec.update({"tflops": f["fwd"] / (ms * 1e-3) / 1e12, "causal_tflops": f["fwd_seq"] / (ms * 1e-3) / 1e12,
                            "gbs": by / (ms * 1e-3) / 1e9,
                            "bound": "tensor" if f["fwd_seq"] / peaks["bf16_tflops"] / 1e3 >= by / peaks["hbm_gbs"]
                            else "hbm"})
            del x, o, lse
            torch.cuda.empty_cache()
        rec["shape"] = f"B={WORKLOADS[name].B} H={WORKLOADS[name].H} Hkv={WORKLOADS[name].Hkv} T={WORKLOADS[name].T} " \
                       f"d={WORKLOADS[name].d} S={WORKLOADS[name].S} {WORKLOADS[name].dtype_name}"
        out[name] = rec
    out["note"] = ("fp32_small runs on the CUDA cores (float32) and is bound by launch latency; its roofline "
                   "uses the same formula as the others")
    return out


def main():
    args = parse()
    from joint_sequence_depth_gb300.inputs import DECODE_WORKLOADS, WORKLOADS, WRITE_WORKLOADS

    if args.workload in DECODE_WORKLOADS:
        return run_decode(args, DECODE_WORKLOADS[args.workload])
    if args.workload in WRITE_WORKLOADS:
        return run_write(args, WRITE_WORKLOADS[args.workload])
    if args.workload in CP_WORKLOADS:
        return run_cp(args, args.workload)
    base = WORKLOADS[args.workload]
    shape = base
    if args.impl == "reference":
        return run_reference(args, shape)

    import torch
    import torch.distributed as dist

    from joint_sequence_depth_gb300 import binding
    from joint_sequence_depth_gb300 import build as mbuild
    from joint_sequence_depth_gb300.inputs import make_inputs

    world, rank, local = dist_setup(args)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mbuild.build()
    binding.load_library()

    x = make_inputs(base, seed=rank_seed(args.workload, rank), device=dev, with_dout=True)
    q, k, v, kd, vd, dout = (x[n] for n in ("q", "k", "v", "kd", "vd", "dout"))
    o = torch.empty_like(q)
    lse = torch.empty(base.B, base.H, base.T, dtype=torch.float32, device=dev)
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(kd),
             torch.empty_like(vd))
    desc = binding.make_desc(base.B, base.H, base.Hkv, base.T, base.S, base.d, base.dtype,
                             slot_capacity=base.slot_capacity)
    slots = base.S if base.slot_capacity else None  # a ring: read the first S of S_mem slots
    ws = torch.empty(binding.moda_bwd_workspace_bytes(desc), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        binding.moda_fwd(q, k, v, kd, vd, o, lse, slots=slots)
        binding.moda_bwd(q, k, v, kd, vd, o, lse, dout, grads, ws, slots=slots)

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    K = args.steps
    # per step: start, after forward, then start/end of each backward stage (Delta, depth, dK/dV, dQ)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(10)] for _ in range(K)]
    for row_ev in ev:
        for e_ in row_ev:
            e_.record(stream)  # creates the event so its handle can be passed to the library
    torch.cuda.synchronize()
    launches0 = binding.moda_launch_count()
    for i in range(K):
        ev[i][0].record(stream)
        binding.moda_fwd(q, k, v, kd, vd, o, lse, slots=slots)
        ev[i][1].record(stream)
        binding.moda_bwd(q, k, v, kd, vd, o, lse, dout, grads, ws, events=ev[i][2:10], slots=slots)
    torch.cuda.synchronize()
    launches = binding.moda_launch_count() - launches0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = ev[0][0].elapsed_time(ev[K - 1][9])
    fwd_ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
    bwd_ms = statistics.mean(ev[i][1].elapsed_time(ev[i][9]) for i in range(K))
    kernel_ms = {"moda_fwd_tc_kernel": fwd_ms}
    for j, name in enumerate(("bwd_delta_kernel", "moda_bwd_depth_kernel", bwd_kernel_name("dkdv", shape.d),
                              bwd_kernel_name("dq", shape.d))):
        if (name == "bwd_delta_kernel") != (shape.S == 0):
            continue  # with depth slots Delta is formed by the depth kernel; without, there is no depth kernel
        kernel_ms[name] = statistics.mean(ev[i][2 + 2 * j].elapsed_time(ev[i][3 + 2 * j]) for i in range(K))
    status = binding.moda_device_status()
    if status != 0:
        raise RuntimeError(f"device status {binding.STATUS_NAMES.get(status, status)} after the timed steps")

    # ------------------------------------------------------------- end to end (host buffers)
    # Every step copies its inputs from pinned host memory, runs moda_fwd + moda_bwd and
    # copies every output back to pinned host memory.  Steps are pipelined over two buffer
    # sets: H2D of step i+1 and D2H of step i-1 run on their own streams while step i
    # computes (the two copy directions use separate copy engines).
    names = ("q", "k", "v", "kd", "vd", "dout")
    host_in = {n: x[n].cpu().pin_memory() for n in names}
    del x
    sets = []
    for _ in range(2):
        din = {n: torch.empty_like(host_in[n], device=dev) for n in names}
        dout_ = (torch.empty_like(din["q"]), torch.empty(base.B, base.H, base.T, dtype=torch.float32, device=dev),
                 torch.empty_like(din["q"]), torch.empty_like(din["k"]), torch.empty_like(din["v"]),
                 torch.empty_like(din["kd"]), torch.empty_like(din["vd"]))
        hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dout_]
        sets.append((din, dout_, hout))
    ws2 = torch.empty_like(ws)
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    E = max(3, args.e2e_steps)

    def run_e2e(n_steps):
        ev_h2d = [torch.cuda.Event() for _ in range(n_steps)]
        ev_comp = [torch.cuda.Event() for _ in range(n_steps)]
        ev_d2h = [torch.cuda.Event() for _ in range(n_steps)]
        for i in range(n_steps):
            din, dout_, hout = sets[i % 2]
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(ev_comp[i - 2])  # set i%2 inputs no longer read
                for n in names:
                    din[n].copy_(host_in[n], non_blocking=True)
                ev_h2d[i].record(h2d_s)
            stream.wait_event(ev_h2d[i])
            if i >= 2:
                stream.wait_event(ev_d2h[i - 2])  # set i%2 outputs already copied out
            o_, l_, *g_ = dout_
            binding.moda_fwd(din["q"], din["k"], din["v"], din["kd"], din["vd"], o_, l_, slots=slots)
            binding.moda_bwd(din["q"], din["k"], din["v"], din["kd"], din["vd"], o_, l_, din["dout"], tuple(g_),
                             ws if i % 2 == 0 else ws2, slots=slots)
            ev_comp[i].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_comp[i])
                for h, d_ in zip(hout, dout_):
                    h.copy_(d_, non_blocking=True)
                ev_d2h[i].record(d2h_s)
        return ev_d2h[-1]

    run_e2e(2)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_s.wait_event(e0)
    last = run_e2e(E)
    stream.wait_event(last)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / E
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in sets[0][2])

    total_ms, e2e_ms, fwd_ms, bwd_ms = max_over_ranks([total_ms, e2e_ms, fwd_ms, bwd_ms], dev)

    f = flops(shape)
    step_flops = f["fwd"] + f["bwd"]
    ms_per_step = total_ms / K
    value = aggregate_tflops(step_flops, ms_per_step, world)
    e2e_value = aggregate_tflops(step_flops, e2e_ms, world)

    # ------------------------------------------------------------- roofline of each kernel
    # Each kernel runs for well under a millisecond inside a timed region of tens of
    # milliseconds, so tensor-bound kernels are measured against the burst bf16 peak.
    peaks, peak_kind = load_peaks()
    counts = kernel_counts(shape)
    kernels = {name: kernel_roofline(counts[name], ms, peaks) for name, ms in kernel_ms.items()}
    # `roofline` is the forward kernel's (the operator's own kernel); the longest backward
    # kernel is reported beside it
    def described(kernel):
        r = dict(kernels[kernel])
        r["traffic"] = traffic_record(kernel, shape.name)
        r["kernel"] = kernel
        r["peak_source"] = f"{peak_kind} ({'bf16 burst, cuBLAS' if r['bound'] == 'tensor' else 'copy'})"
        r["step_share"] = kernel_ms[kernel] / ms_per_step
        return r

    roof = described("moda_fwd_tc_kernel")
    bwd_names = [n for n in kernel_ms if n != "moda_fwd_tc_kernel"]
    roof_bwd = described(max(bwd_names, key=kernel_ms.get))
    fwd_configs = time_forward_configs(dev, peaks) if world == 1 else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = time_oracle_steps(shape, shape.T, 1)
        cpu = {"value": r["value"], "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle", "sample": r["sample"]}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
                "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": shape.dtype_name, "data": "synthetic",
                "config": workload_config(shape),
                "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
                "clocks": clk,
                "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                        "ms_per_step": e2e_ms},
                "gpu_launches": launches, "roofline": roof, "roofline_bwd": roof_bwd, "kernels": kernels,
                "forward_configs": fwd_configs, "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
