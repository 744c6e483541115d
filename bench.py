"""Throughput of the GB300 QMoE layer on one synthetic workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl reference]

The float_* workloads measure the float MoE layer of the same library
(moe_forward / moe_forward_hostio) in the same way, under the metric
"MoE layer tokens/sec"; the qkv_* workloads measure the RMSNorm + 4-bit
Q/K/V projection (matmul_nbits_qkv) under "QKV projection rows/sec"; the gmm_*
workloads measure GroupedMatMul-29 on 16-bit operands (grouped_matmul) under
"GroupedMatMul rows/sec", a row being one input row with its S selections.

One step is one full qmoe_forward call (routing, grouping, FC1 + activation,
FC2, combine) over one batch of the workload's tokens, with inputs and
weights resident in HBM.  `value` is whole-job tokens/s.  `e2e` measures the
same metric through qmoe_forward_hostio: page-locked host activations and
logits copied in, the layer, and the output copied back, every step.
Under torchrun each rank runs an independent replica (weak scaling; the
layer has no cross-GPU exchange); the elapsed time is the max over ranks.

Run with no --workload, the line is the decode workload's, and the same
measurements of the prefill, many-small-experts and large-E workloads, taken
after it in the same process, follow in its "workloads" list (--only leaves
them out).  Each line's roofline covers the dominant kernel (FC1), with FC2 and
the whole layer against the same peak under roofline.others.

`--impl reference` times the CPU oracle (the double-precision C restatement
of the operator pages) on the host cores on a bounded token sample of the
same workload.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_mixture_experts_gb300.workloads import (  # noqa: E402
    FLOAT_WORKLOADS, GMM_WORKLOADS, QKV_WORKLOADS, WORKLOADS, make_float_inputs, make_gmm_inputs,
    make_inputs, make_qkv_inputs)

METRIC = "QMoE layer tokens/sec"
UNIT = "tokens/s"
DEFAULT_STEPS = {"tiny": 2000, "decode": 8000, "prefill": 100, "many_small": 1000,
                 "large_e": 100, "float_tiny": 2000, "float_decode": 1000, "float_prefill": 40,
                 "float_prefill_e4": 100, "qkv_tiny": 2000, "qkv_decode": 5000,
                 "qkv_decode_f32": 5000, "qkv_decode_wide": 2000, "gmm_tiny": 2000,
                 "gmm_prefill": 200, "gmm_prefill_bf16": 200, "gmm_prefill_f32": 40, "gmm_prefill_f64": 3}
QKV_METRIC = "QKV projection rows/sec"
FLOAT_METRIC = "MoE layer tokens/sec"
GMM_METRIC = "GroupedMatMul rows/sec"
# dense TF32 / dense BF16 tensor throughput, nominal (1.1 and 2.25 PFLOP/s)
TF32_PER_BF16 = 1.1 / 2.25
# nominal dense fp64 rate of the part (TFLOP/s)
FP64_TFLOPS_NOMINAL = 1.25
L2_BYTES = 129 * 1024 * 1024
# measured after the decode line when no workload is named (the tensor-bound configurations)
EXTRA_WORKLOADS = ("prefill", "many_small", "large_e")


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


# ----------------------------------------------------------------------------
# Ranks (one process per GPU, launched by torch.distributed.run; replicas only)
# ----------------------------------------------------------------------------

def ranks_init(device_kind):
    """(world, rank, local) from the launcher's environment.  With more than one
    rank the process group is set up: NCCL over the ranks' GPUs (each rank on
    its LOCAL_RANK device), gloo for CPU-only use."""
    import torch.distributed as dist
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local = _env_int("LOCAL_RANK", 0)
    if world > 1:
        if device_kind == "cuda":
            import torch
            torch.cuda.set_device(local)
            dist.init_process_group(backend="nccl")
        else:
            dist.init_process_group(backend="gloo")
    return world, rank, local


def ranks_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    """The largest of the ranks' values of x (the whole job's time is the slowest
    rank's)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def ranks_done(world):
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# Algorithmic work (bytes and FLOPs the method must move or compute)
# ----------------------------------------------------------------------------

def expert_bytes(wl, which):
    """Packed weight + scale bytes of one expert for FC1 or FC2."""
    H, I, f, pk = wl.hidden, wl.inter, wl.fusion, wl.pack
    if which == 1:
        rows, K, nb = f * I, H, (H // wl.block_size if wl.block_size else 1)
    else:
        rows, K, nb = H, I, (I // wl.block_size if wl.block_size else 1)
    return rows * (K // pk) + rows * nb * 4


def layer_flops(wl, slots):
    return 2.0 * slots * (wl.fusion * wl.inter * wl.hidden + wl.hidden * wl.inter)


def fc1_flops(wl, slots):
    return 2.0 * slots * wl.fusion * wl.inter * wl.hidden


# ----------------------------------------------------------------------------
# Clocks during the timed region
# ----------------------------------------------------------------------------

QUERY = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = open(os.path.join(tempfile.gettempdir(),
                                         f".qmoe_clocks_{os.getpid()}.csv"), "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.out is not None:
            self.out.close()

    def summary(self):
        if self.out is None or self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.out.name) as f:
            for r in csv.reader(f):
                r = [x.strip() for x in r]
                if len(r) < 10:
                    continue
                if self.uuid and self.uuid not in r[1]:
                    continue
                rows.append(r)
        try:
            os.remove(self.out.name)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        loaded = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------
# Measured peaks and the ncu traffic record
# ----------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "quantized_mixture_experts_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(profile_name, kernel_files):
    """Per-launch DRAM bytes recorded under profiles/, if the kernel source still
    matches the one the counters were taken from."""
    path = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_source_sha(kernel_files):
        return None
    return float(m.group(1))


def prequeue(stream, ms=2.0):
    """Keep the device busy for about `ms` before a timed region starts, so that the
    host enqueues the region's first steps while the device is still busy and the
    events around them measure device time, not the host's first launches (for
    short regions: the driver's default is a few dozen steps)."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(ms * 2.0e6))   # ~2 cycles per ns at the SM clock


def kernel_pass(q, step, steps, kernel_id, before=None):
    """Average device time of the launches of one kernel of the path, from CUDA
    events recorded around those launches on the call stream, over a second pass of
    the timed steps.  The events are kept out of the timed pass itself: recorded
    between two launches they would stop the second from starting as a
    programmatic dependent of the first, and so change the time being measured."""
    import torch
    torch.cuda.synchronize()
    q.profile_begin(kernel_id)
    prequeue(torch.cuda.current_stream())
    for i in range(steps):
        if before is not None:
            before(i)
        step()
    torch.cuda.synchronize()
    n, ms = q.profile_end()
    return n, ms


# ----------------------------------------------------------------------------
# Reference arm: the CPU oracle
# ----------------------------------------------------------------------------

def run_reference(args, wl):
    import oracle
    rank = _env_int("RANK", 0)
    if rank != 0:
        return
    inp = make_inputs(wl)
    cores = os.cpu_count() or 1
    sample = min(wl.tokens, 16)
    rng = np.random.default_rng(7)
    times = []
    for step in range(args.warmup + args.steps):
        tok = np.sort(rng.choice(wl.tokens, size=sample, replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        oracle.qmoe(inp["input"], inp["router_probs"], inp["fc1_experts_weights"],
                    inp["fc1_scales"], inp["fc2_experts_weights"], inp["fc2_scales"],
                    tokens=tok, nthreads=cores, **wl.attrs())
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = sample * len(times) / total
    used = min(cores, sample)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                             "sample": f"{sample} of {wl.tokens} tokens per step, seeded"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(wl):
    return {"workload": f"QMoE {wl.name}", "input_shape": list(wl.input_shape),
            "tokens": wl.tokens, "hidden": wl.hidden, "inter": wl.inter,
            "experts": wl.experts, "k": wl.k, "bits": wl.bits,
            "block_size": wl.block_size or "column-wise", "activation": wl.activation}


# ----------------------------------------------------------------------------
# CPU baseline (oracle) beside the GPU number
# ----------------------------------------------------------------------------

def cpu_baseline(wl, inp):
    import oracle
    cores = os.cpu_count() or 1
    sample = min(wl.tokens, 16)
    tok = np.arange(sample, dtype=np.int64) if sample == wl.tokens else \
        np.sort(np.random.default_rng(3).choice(wl.tokens, size=sample, replace=False))
    t0 = time.perf_counter()
    oracle.qmoe(inp["input"], inp["router_probs"], inp["fc1_experts_weights"], inp["fc1_scales"],
                inp["fc2_experts_weights"], inp["fc2_scales"], tokens=tok.astype(np.int64),
                nthreads=cores, **wl.attrs())
    dt = time.perf_counter() - t0
    return {"value": sample / dt, "unit": UNIT, "cores": min(cores, sample), "kind": "oracle",
            "sample": f"{sample} of {wl.tokens} tokens, {dt:.2f} s"}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def run_gpu(args, wl, extra=()):
    """The bench line of workload `wl`; with `extra`, the same measurements of
    those workloads, taken after it in this process, go in its `workloads` list."""
    import torch

    import __graft_entry__
    import quantized_mixture_experts_gb300 as q

    world, rank, local = ranks_init("cuda")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    ranks_barrier(world)
    q.load()
    line = measure_qmoe(args, wl, args.steps, world, rank, dev)
    if extra:
        subs = []
        for name in extra:
            steps = args.steps if args.steps_given else DEFAULT_STEPS[name]
            sub = measure_qmoe(args, WORKLOADS[name], steps, world, rank, dev)
            torch.cuda.empty_cache()
            if rank == 0:
                subs.append(sub)
        if rank == 0:
            line["workloads"] = subs
    if rank == 0:
        print(json.dumps(line), flush=True)
    ranks_done(world)


def measure_qmoe(args, wl, steps, world, rank, dev):
    """One workload's measurements (rank 0 gets the line, other ranks None)."""
    import torch

    import quantized_mixture_experts_gb300 as q

    inp = make_inputs(wl, salt=rank)
    t = {k: torch.from_numpy(v).to(dev) for k, v in inp.items()}
    attrs = q.make_attrs(**wl.attrs())
    path = q.choose_path(wl.input_shape, tuple(t["fc1_experts_weights"].shape), attrs)
    ws = q.alloc_workspace(q.workspace_size(wl.input_shape, tuple(t["fc1_experts_weights"].shape),
                                            attrs), dev)
    y = torch.empty_like(t["input"])
    sel = torch.empty((wl.tokens, wl.k), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        q.qmoe_forward(t["input"], t["router_probs"], t["fc1_experts_weights"], t["fc1_scales"],
                       t["fc2_experts_weights"], t["fc2_scales"], attrs=attrs, output=y,
                       workspace=ws, topk_idx=sel, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    err = q.get_device_error(ws, stream)
    touched = int(torch.unique(sel).numel())

    bound = "hbm" if path == q.PATH_DECODE else "tensor"
    dominant = q.KERNEL_FC1
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass

    ranks_barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = q.launch_count()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(uuid) as clocks:
        prequeue(stream)
        start.record(stream)
        for _ in range(steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize(dev)
    launches = q.launch_count() - launches0
    n_launch, fc1_ms = kernel_pass(q, step, min(steps, 1000), dominant)
    n_launch2, fc2_ms = kernel_pass(q, step, min(steps, 1000), q.KERNEL_FC2)
    ranks_barrier(world)
    elapsed_ms = start.elapsed_time(stop)
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    tokens_total = wl.tokens * steps * world
    value = tokens_total / (elapsed_ms / 1e3)

    # end to end through the host-IO entry point
    hx = torch.from_numpy(inp["input"]).pin_memory()
    hl = torch.from_numpy(inp["router_probs"]).pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    ws_io = q.alloc_workspace(q.workspace_size(wl.input_shape,
                                               tuple(t["fc1_experts_weights"].shape), attrs,
                                               hostio=True), dev)
    e2e_steps = max(1, min(steps, 2000))

    def step_io():
        q.qmoe_forward_hostio(hx, hl, t["fc1_experts_weights"], t["fc1_scales"],
                              t["fc2_experts_weights"], t["fc2_scales"], hy, attrs=attrs,
                              workspace=ws_io, stream=stream)
        stream.synchronize()

    for _ in range(3):
        step_io()
    ranks_barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        step_io()
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, world, dev)
    e2e_value = wl.tokens * e2e_steps * world / e2e_s
    if not np.array_equal(hy.numpy(), y.cpu().numpy()):
        raise RuntimeError("host-IO output differs from the device-resident output")

    if rank != 0:
        return None

    peaks = measured_peaks()
    avg_ms = fc1_ms / max(1, n_launch)
    if bound == "hbm":
        per_unit = expert_bytes(wl, 1)
        algo = per_unit * touched + wl.tokens * wl.hidden * 2
        achieved = algo / (avg_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
        profile_name = "decode_fc1_decode.md"
        files = ["gemv_decode.cu", "decode_core.cuh", "ptx.cuh"]
    else:
        slots = wl.tokens * wl.k
        algo = fc1_flops(wl, slots)
        achieved = algo / (avg_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops_sustained"] if steps * avg_ms > 1000 else peaks["bf16_tflops"]
        unit = "TFLOP/s"
        profile_name = f"grouped_fc1_{wl.name}.md"
        files = ["gemm_pair.cu", "ptx.cuh"]
    # the second projection and the whole layer against the same peak
    avg2_ms = fc2_ms / max(1, n_launch2)
    step_ms = elapsed_ms / steps
    if bound == "hbm":
        algo2 = expert_bytes(wl, 2) * touched
        layer_algo = (expert_bytes(wl, 1) + expert_bytes(wl, 2)) * touched + \
            inp["input"].nbytes * 2 + inp["router_probs"].nbytes
        scale = 1e9
    else:
        algo2 = layer_flops(wl, wl.tokens * wl.k) - algo
        layer_algo = layer_flops(wl, wl.tokens * wl.k)
        scale = 1e12
    fc2_ach = algo2 / (avg2_ms / 1e3) / scale if avg2_ms > 0 else None
    layer_ach = layer_algo / (step_ms / 1e3) / scale
    others = {"FC2": {"kernel_ms": avg2_ms, "launches": n_launch2, "algorithmic": algo2,
                      "achieved": fc2_ach, "frac": fc2_ach / peak if fc2_ach and peak else None},
              "layer": {"ms": step_ms, "algorithmic": layer_algo, "achieved": layer_ach,
                        "frac": layer_ach / peak if peak else None}}
    traffic = ncu_traffic(profile_name, files) if os.path.exists(
        os.path.join(ROOT, "quantized_mixture_experts_gb300", "csrc", files[0])) else None

    cfg = config_dict(wl)
    cfg.update({"path": q.PATH_NAMES.get(path, str(path)), "touched_experts": touched,
                "l2": ("weights of touched experts exceed the 129 MB L2; no flush"
                       if expert_bytes(wl, 1) * touched > L2_BYTES else "L2 flush not applied"),
                "parallelism": f"replicas{world}" if world > 1 else "single GPU",
                "logits_sigma": wl.logit_sigma, "device_error": err})
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded; random packed weights)", "config": cfg,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak if peak else None, "traffic": traffic,
                     "kernel": "FC1", "kernel_ms": avg_ms, "launches": n_launch,
                     "algorithmic": algo, "peak_source": peaks["source"],
                     "others": others},
        "e2e": {"value": e2e_value, "unit": UNIT,
                "h2d_bytes_per_step": int(inp["input"].nbytes + inp["router_probs"].nbytes),
                "d2h_bytes_per_step": int(inp["input"].nbytes), "steps": e2e_steps},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, inp)
    return line


# ----------------------------------------------------------------------------
# Float MoE layer (moe_forward)
# ----------------------------------------------------------------------------

F_OPTIONAL = ("fc1_experts_bias", "fc2_experts_bias", "fc3_experts_weights", "fc3_experts_bias")


def float_config(wl):
    return {"workload": f"MoE {wl.name}", "input_shape": list(wl.input_shape),
            "tokens": wl.tokens, "hidden": wl.hidden, "inter": wl.inter,
            "experts": wl.experts, "k": wl.k, "activation": wl.activation,
            "swiglu_fusion": wl.swiglu_fusion, "fc3": wl.fc3, "biases": wl.biases,
            "normalize_routing_weights": wl.normalize}


def float_fc1_rows(wl):
    """Weight rows FC1 (with FC3) reads per expert."""
    paired = wl.activation == "swiglu" or (wl.activation == "silu" and wl.fc3)
    return (2 if paired else 1) * wl.inter


def float_oracle(wl, inp, tok, cores):
    import oracle
    return oracle.moe(inp["input"], inp["router_probs"], inp["fc1_experts_weights"],
                      inp["fc2_experts_weights"], fc1_bias=inp.get("fc1_experts_bias"),
                      fc2_bias=inp.get("fc2_experts_bias"), fc3_w=inp.get("fc3_experts_weights"),
                      fc3_bias=inp.get("fc3_experts_bias"), tokens=tok, nthreads=cores,
                      **wl.attrs())


def run_reference_float(args, wl):
    if _env_int("RANK", 0) != 0:
        return
    inp = make_float_inputs(wl)
    cores = os.cpu_count() or 1
    sample = min(wl.tokens, 16)
    rng = np.random.default_rng(7)
    times = []
    for step in range(args.warmup + args.steps):
        tok = np.sort(rng.choice(wl.tokens, size=sample, replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        float_oracle(wl, inp, tok, cores)
        if step >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = sample * len(times) / total
    line = {"impl": "reference", "metric": FLOAT_METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": float_config(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(cores, sample),
                             "kind": "oracle",
                             "sample": f"{sample} of {wl.tokens} tokens per step, seeded"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gpu_float(args, wl):
    import torch

    import __graft_entry__
    import quantized_mixture_experts_gb300 as q

    world, rank, local = ranks_init("cuda")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    ranks_barrier(world)
    q.load()

    inp = make_float_inputs(wl, salt=rank)
    t = {k: torch.from_numpy(v).to(dev) for k, v in inp.items()}
    opt = {k: t.get(k) for k in F_OPTIONAL}
    attrs = q.make_moe_attrs(**wl.attrs())
    fc1_shape = tuple(t["fc1_experts_weights"].shape)
    path = q.moe_choose_path(wl.input_shape, fc1_shape, attrs)
    ws = q.alloc_workspace(q.moe_workspace_size(wl.input_shape, fc1_shape, attrs), dev)
    y = torch.empty_like(t["input"])
    sel = torch.empty((wl.tokens, wl.k), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        q.moe_forward(t["input"], t["router_probs"], t["fc1_experts_weights"],
                      t["fc2_experts_weights"], attrs=attrs, output=y, workspace=ws,
                      topk_idx=sel, stream=stream, **opt)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    err = q.moe_get_device_error(ws, stream)
    touched = int(torch.unique(sel).numel())
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    ranks_barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = q.launch_count()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(uuid) as clocks:
        prequeue(stream)
        start.record(stream)
        for _ in range(args.steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize(dev)
    launches = q.launch_count() - launches0
    n_launch, fc1_ms = kernel_pass(q, step, min(args.steps, 1000), q.KERNEL_FC1)
    elapsed_ms = start.elapsed_time(stop)
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    value = wl.tokens * args.steps * world / (elapsed_ms / 1e3)

    hx = torch.from_numpy(inp["input"]).pin_memory()
    hl = torch.from_numpy(inp["router_probs"]).pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    ws_io = q.alloc_workspace(q.moe_workspace_size(wl.input_shape, fc1_shape, attrs,
                                                   hostio=True), dev)
    e2e_steps = max(1, min(args.steps, 1000))

    def step_io():
        q.moe_forward_hostio(hx, hl, t["fc1_experts_weights"], t["fc2_experts_weights"], hy,
                             attrs=attrs, workspace=ws_io, stream=stream, **opt)
        stream.synchronize()

    for _ in range(3):
        step_io()
    ranks_barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        step_io()
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, world, dev)
    e2e_value = wl.tokens * e2e_steps * world / e2e_s
    if not np.array_equal(hy.numpy(), y.cpu().numpy()):
        raise RuntimeError("host-IO output differs from the device-resident output")
    if rank != 0:
        ranks_done(world)
        return

    peaks = measured_peaks()
    avg_ms = fc1_ms / max(1, n_launch)
    slots = wl.tokens * wl.k
    # decode-sized batches stream the touched experts' fp32 weights; large ones are
    # bound by the TF32 tensor cores
    weight_bytes = float_fc1_rows(wl) * wl.hidden * 4 * touched
    flops = 2.0 * slots * float_fc1_rows(wl) * wl.hidden
    bound = "hbm" if flops / weight_bytes < 200 else "tensor"
    if bound == "hbm":
        algo = weight_bytes + slots * wl.hidden * 4
        achieved = algo / (avg_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    else:
        algo = flops
        achieved = algo / (avg_ms / 1e3) / 1e12
        bf16 = peaks["bf16_tflops_sustained"] if args.steps * avg_ms > 1000 else peaks["bf16_tflops"]
        peak = bf16 * TF32_PER_BF16
        unit = "TFLOP/s"
    files = ["moe_float.cu", "ptx.cuh"]
    traffic = ncu_traffic(f"float_fc1_{wl.name}.md", files)
    cfg = float_config(wl)
    cfg.update({"path": {q.MOE_PATH_GROUPED: "grouped", q.MOE_PATH_GENERIC: "generic"}.get(
        path, str(path)), "touched_experts": touched,
        "l2": ("weights of touched experts exceed the 129 MB L2; no flush"
               if weight_bytes > L2_BYTES else "L2 flush not applied"),
        "parallelism": f"replicas{world}" if world > 1 else "single GPU",
        "logits_sigma": wl.logit_sigma, "device_error": err})
    line = {
        "metric": FLOAT_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "tf32",
        "data": "synthetic (seeded; random fp32 weights)", "config": cfg,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak if peak else None, "traffic": traffic,
                     "kernel": "FC1", "kernel_ms": avg_ms, "launches": n_launch,
                     "algorithmic": algo,
                     "peak_source": peaks["source"] + (
                         "" if bound == "hbm" else " bf16 x nominal TF32/BF16 ratio")},
        "e2e": {"value": e2e_value, "unit": UNIT,
                "h2d_bytes_per_step": int(inp["input"].nbytes + inp["router_probs"].nbytes),
                "d2h_bytes_per_step": int(inp["input"].nbytes), "steps": e2e_steps},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        sample = min(wl.tokens, 16)
        tok = np.sort(np.random.default_rng(3).choice(wl.tokens, size=sample,
                                                      replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        float_oracle(wl, inp, tok, cores)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": sample / dt, "unit": UNIT, "cores": min(cores, sample),
                                "kind": "oracle",
                                "sample": f"{sample} of {wl.tokens} tokens, {dt:.2f} s"}
    print(json.dumps(line), flush=True)
    ranks_done(world)


# ----------------------------------------------------------------------------
# RMSNorm + 4-bit Q/K/V projection (matmul_nbits_qkv)
# ----------------------------------------------------------------------------

def qkv_config(wl):
    return {"workload": f"MatMulNBitsQkv {wl.name}", "input_shape": list(wl.input_shape),
            "rows": wl.rows, "K": wl.K, "Nq": wl.Nq, "Nkv": wl.Nkv, "T1": wl.dtype,
            "skip": wl.skip, "residual": wl.residual, "bits": 4, "block_size": 32}


def qkv_weight_bytes(wl):
    """Packed codes + block scales of the three projections."""
    n = wl.Nq + 2 * wl.Nkv
    return n * wl.kblocks * 16 + n * wl.kblocks * (2 if wl.dtype == "float16" else 4)


def qkv_oracle(inp, wl, cores):
    import oracle
    f = lambda k: None if k not in inp else inp[k].astype(np.float64)
    return oracle.qkv(f("A"), f("norm_scale"), inp["q_B"], f("q_scales"), inp["k_B"],
                      f("k_scales"), inp["v_B"], f("v_scales"), skip=f("skip"),
                      residual=wl.residual)


def run_reference_qkv(args, wl):
    if _env_int("RANK", 0) != 0:
        return
    inp = make_qkv_inputs(wl)
    times = []
    for step in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        qkv_oracle(inp, wl, 1)
        if step >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = wl.rows * len(times) / total
    line = {"impl": "reference", "metric": QKV_METRIC, "value": value, "unit": "rows/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": qkv_config(wl),
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                             "sample": f"all {wl.rows} rows per step"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gpu_qkv(args, wl):
    import torch

    import __graft_entry__
    import quantized_mixture_experts_gb300 as q

    world, rank, local = ranks_init("cuda")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    ranks_barrier(world)
    q.load()
    inp = make_qkv_inputs(wl, salt=rank)
    t = {k: torch.from_numpy(v).to(dev) for k, v in inp.items()}
    dt = t["A"].dtype
    attrs = q.make_qkv_attrs(K=wl.K, Nq=wl.Nq, Nkv=wl.Nkv)
    path = q.qkv_choose_path(wl.input_shape, attrs, dt)
    ws = q.alloc_workspace(q.qkv_workspace_size(wl.input_shape, attrs, dt), dev)
    lead = tuple(wl.input_shape[:-1])
    outs = (torch.empty(lead + (wl.Nq,), dtype=dt, device=dev),
            torch.empty(lead + (wl.Nkv,), dtype=dt, device=dev),
            torch.empty(lead + (wl.Nkv,), dtype=dt, device=dev))
    res = torch.empty_like(t["A"]) if wl.residual else None
    stream = torch.cuda.current_stream(dev)
    # a buffer six times L2, rewritten between timed steps: the weights (tens of MB)
    # would otherwise stay in the 129 MB L2 from one step to the next
    flush = torch.empty(6 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        q.matmul_nbits_qkv(t["A"], t["norm_scale"], t["q_B"], t["q_scales"], t["k_B"],
                           t["k_scales"], t["v_B"], t["v_scales"], skip=t.get("skip"),
                           residual=res if res is not None else None, attrs=attrs,
                           outputs=outs, workspace=ws, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    ranks_barrier(world)
    torch.cuda.synchronize(dev)
    # A decode-sized call is shorter than its host-side enqueue (argument marshalling,
    # tensor-map encoding, two launches).  Each timed step therefore starts with an
    # L2 flush long enough (about 130 us of device time) for the host to enqueue the
    # whole call behind it, so that the events around the call see device time only.
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches0 = q.launch_count()
    with ClockSampler(uuid) as clocks:
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            step()
            stops[i].record(stream)
        torch.cuda.synchronize(dev)
    launches = q.launch_count() - launches0
    n_launch, gemv_ms = kernel_pass(q, step, min(args.steps, 1000), q.KERNEL_FC1,
                                    before=lambda i: flush.fill_(float(i)))
    elapsed_ms = sum(a.elapsed_time(b) for a, b in zip(starts, stops))
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    value = wl.rows * args.steps * world / (elapsed_ms / 1e3)

    # end to end: pinned host activations in, the three projections back, every step
    hA = torch.from_numpy(inp["A"]).pin_memory()
    hs = torch.from_numpy(inp["skip"]).pin_memory() if "skip" in inp else None
    hq = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    dA = torch.empty_like(t["A"])
    ds = torch.empty_like(t["skip"]) if hs is not None else None
    e2e_steps = max(1, min(args.steps, 2000))

    def step_io():
        dA.copy_(hA, non_blocking=True)
        if ds is not None:
            ds.copy_(hs, non_blocking=True)
        q.matmul_nbits_qkv(dA, t["norm_scale"], t["q_B"], t["q_scales"], t["k_B"], t["k_scales"],
                           t["v_B"], t["v_scales"], skip=ds,
                           residual=res if res is not None else None, attrs=attrs, outputs=outs,
                           workspace=ws, stream=stream)
        for h, o in zip(hq, outs):
            h.copy_(o, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        step_io()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        step_io()
    e2e_s = time.perf_counter() - t0
    e2e_value = wl.rows * e2e_steps * world / e2e_s
    if rank != 0:
        ranks_done(world)
        return
    peaks = measured_peaks()
    avg_ms = gemv_ms / max(1, n_launch)
    algo = qkv_weight_bytes(wl) + wl.rows * wl.K * 2
    achieved = algo / (avg_ms / 1e3) / 1e9
    cfg = qkv_config(wl)
    cfg.update({"path": {q.QKV_PATH_DECODE: "decode", q.QKV_PATH_GENERIC: "generic"}.get(path),
                "l2": "a 774 MB buffer is rewritten before every timed step (outside the events)",
                "timing": "events around each call, enqueued behind the flush (device time)",
                "parallelism": f"replicas{world}" if world > 1 else "single GPU"})
    h2d = int(inp["A"].nbytes + (inp["skip"].nbytes if "skip" in inp else 0))
    d2h = int(sum(o.numel() * o.element_size() for o in outs))
    line = {
        "metric": QKV_METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if wl.dtype == "float16" else "f32",
        "data": "synthetic (seeded; random packed weights)", "config": cfg,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": ncu_traffic(f"qkv_gemv_{wl.name}.md",
                                            ["qkv_gemv.cu", "decode_core.cuh", "ptx.cuh"]),
                     "kernel": "QKV GEMV", "kernel_ms": avg_ms, "launches": n_launch,
                     "algorithmic": algo, "peak_source": peaks["source"]},
        "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
    }
    if not args.no_cpu_baseline:
        t0 = time.perf_counter()
        qkv_oracle(inp, wl, 1)
        dt_s = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": wl.rows / dt_s, "unit": "rows/s", "cores": 1,
                                "kind": "oracle", "sample": f"all {wl.rows} rows, {dt_s:.2f} s"}
    print(json.dumps(line), flush=True)
    ranks_done(world)


# ----------------------------------------------------------------------------
# GroupedMatMul-29 on 16-bit operands (grouped_matmul, tensor-core path)
# ----------------------------------------------------------------------------

def gmm_config(wl):
    return {"workload": f"GroupedMatMul {wl.name}", "M": wl.M, "K": wl.K, "G": wl.G,
            "N": wl.N, "S": wl.S, "T": wl.dtype, "Tind": "int64", "bias": None}


def gmm_rounded(a, dtype):
    """float32 host array -> float64 holding the values of the workload's type."""
    import torch
    if dtype in ("float32", "float64"):
        return np.asarray(a, dtype=np.float64)
    tdt = torch.float16 if dtype == "float16" else torch.bfloat16
    return torch.from_numpy(np.ascontiguousarray(a)).to(tdt).double().numpy()


def gmm_oracle_sample(inp, wl, seed, rows=256, cols=512):
    """The oracle on a seeded sample of input rows and output columns: output[m, i, n]
    for those rows and columns is the GroupedMatMul definition applied to the sampled
    rows and to weights[:, :, cols].  Returns (seconds, rows-equivalent of work)."""
    import oracle
    rng = np.random.default_rng(seed)
    r = np.sort(rng.choice(wl.M, size=min(rows, wl.M), replace=False))
    c = np.sort(rng.choice(wl.N, size=min(cols, wl.N), replace=False))
    x = gmm_rounded(inp["input"][r], wl.dtype)
    w = gmm_rounded(inp["weights"][:, :, c], wl.dtype)
    t0 = time.perf_counter()
    _, st = oracle.grouped_matmul(x, w, inp["group_indices"][r])
    dt = time.perf_counter() - t0
    if st != oracle.OK:
        raise RuntimeError("oracle rejected the GroupedMatMul sample")
    return dt, len(r) * len(c) / wl.N, f"{len(r)} of {wl.M} rows x {len(c)} of {wl.N} columns"


def run_reference_gmm(args, wl):
    if _env_int("RANK", 0) != 0:
        return
    inp = make_gmm_inputs(wl)
    times, work = [], 0.0
    for step in range(args.warmup + args.steps):
        dt, rows_eq, sample = gmm_oracle_sample(inp, wl, seed=step)
        if step >= args.warmup:
            times.append(dt)
            work += rows_eq
    total = sum(times)
    value = work / total
    line = {"impl": "reference", "metric": GMM_METRIC, "value": value, "unit": "rows/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": gmm_config(wl),
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                             "sample": f"{sample} per step, seeded; rows/s scaled by the "
                                       "column fraction"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gpu_gmm(args, wl):
    import torch

    import __graft_entry__
    import quantized_mixture_experts_gb300 as q

    world, rank, local = ranks_init("cuda")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    if rank == 0 or world == 1:
        __graft_entry__.build()
    ranks_barrier(world)
    q.load()
    inp = make_gmm_inputs(wl, salt=rank)
    tdt = {"float16": torch.float16, "bfloat16": torch.bfloat16, "float32": torch.float32,
           "float64": torch.float64}[wl.dtype]
    x = torch.from_numpy(inp["input"]).to(dev).to(tdt)
    w = torch.from_numpy(inp["weights"]).to(dev).to(tdt)
    idx = torch.from_numpy(inp["group_indices"]).to(dev)
    out = torch.empty((wl.M, wl.S, wl.N), dtype=tdt, device=dev)
    ws = q.alloc_workspace(q.binding.grouped_matmul_workspace_size(wl.M, wl.K, wl.G, wl.N,
                                                                   wl.S, tdt), dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        q.grouped_matmul(x, w, idx, output=out, workspace=ws, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    err = q.get_device_error(ws, stream)
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    ranks_barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = q.launch_count()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(uuid) as clocks:
        prequeue(stream)
        start.record(stream)
        for _ in range(args.steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize(dev)
    launches = q.launch_count() - launches0
    n_launch, gemm_ms = kernel_pass(q, step, min(args.steps, 1000), q.KERNEL_GMM)
    ranks_barrier(world)
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), world, dev)
    value = wl.M * args.steps * world / (elapsed_ms / 1e3)

    # end to end: page-locked host rows and indices in, the output back, every step
    hx = x.cpu().pin_memory()
    hi = torch.from_numpy(inp["group_indices"]).pin_memory()
    ho = torch.empty(out.shape, dtype=tdt).pin_memory()
    dx, di = torch.empty_like(x), torch.empty_like(idx)
    e2e_steps = max(1, min(args.steps, 200))

    def step_io():
        dx.copy_(hx, non_blocking=True)
        di.copy_(hi, non_blocking=True)
        q.grouped_matmul(dx, w, di, output=out, workspace=ws, stream=stream)
        ho.copy_(out, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        step_io()
    ranks_barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        step_io()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    e2e_value = wl.M * e2e_steps * world / e2e_s
    if rank != 0:
        ranks_done(world)
        return
    peaks = measured_peaks()
    avg_ms = gemm_ms / max(1, n_launch)
    achieved = wl.flops / (avg_ms / 1e3) / 1e12
    # f16 and bf16 have the same nominal dense rate: the measured bf16 peak serves both.
    # f32 runs as three TF32 products per step: its peak is the measured bf16 peak x the
    # nominal TF32 / BF16 ratio (1.1 / 2.25), and a third of that bounds the f32 rate.
    peak = peaks["bf16_tflops_sustained"] if args.steps * avg_ms > 1000 else peaks["bf16_tflops"]
    bound = "tensor"
    if wl.dtype == "float32":
        peak = peak * TF32_PER_BF16
    elif wl.dtype == "float64":
        # fp64 runs on the general kernel (GB300's fp64 tensor rate is no faster): its
        # ceiling is the nominal fp64 rate, no measured figure exists for it
        peak, bound = FP64_TFLOPS_NOMINAL, "alu"
    cfg = gmm_config(wl)
    cfg.update({"l2": f"weights {w.numel() * 2 / 1e9:.2f} GB per step exceed the 129 MB L2; "
                      "no flush",
                "parallelism": f"replicas{world}" if world > 1 else "single GPU",
                "device_error": err})
    line = {
        "metric": GMM_METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"float16": "f16", "bfloat16": "bf16", "float32": "f32 (3 x tf32)",
                  "float64": "f64"}[wl.dtype],
        "data": "synthetic (seeded; uniform activations and weights)", "config": cfg,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak if peak else None,
                     "traffic": ncu_traffic(f"gmm_tc_{wl.name}.md", ["gemm_f16.cu", "ptx.cuh"]),
                     "kernel": "GroupedMatMul GEMM", "kernel_ms": avg_ms, "launches": n_launch,
                     "algorithmic": wl.flops,
                     "peak_source": ("nominal fp64" if wl.dtype == "float64" else peaks["source"])},
        "e2e": {"value": e2e_value, "unit": "rows/s",
                "h2d_bytes_per_step": int(hx.numel() * 2 + hi.numel() * 8),
                "d2h_bytes_per_step": int(ho.numel() * 2), "steps": e2e_steps},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        dt, rows_eq, sample = gmm_oracle_sample(inp, wl, seed=0)
        line["cpu_baseline"] = {"value": rows_eq / dt, "unit": "rows/s", "cores": 1,
                                "kind": "oracle",
                                "sample": f"{sample}, {dt:.2f} s; rows/s scaled by the "
                                          "column fraction"}
    print(json.dumps(line), flush=True)
    ranks_done(world)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=None,
                    choices=sorted(WORKLOADS) + sorted(FLOAT_WORKLOADS) + sorted(QKV_WORKLOADS)
                    + sorted(GMM_WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", action="store_true",
                    help="without --workload: the decode line alone, no extra workloads")
    args = ap.parse_args()
    args.steps_given = args.steps is not None
    if args.workload in GMM_WORKLOADS:
        gwl = GMM_WORKLOADS[args.workload]
        if args.steps is None:
            args.steps = 3 if args.impl == "reference" else DEFAULT_STEPS[gwl.name]
        args.warmup = max(3, args.warmup)
        if args.impl == "reference":
            run_reference_gmm(args, gwl)
        else:
            run_gpu_gmm(args, gwl)
        return
    if args.workload in QKV_WORKLOADS:
        qwl = QKV_WORKLOADS[args.workload]
        if args.steps is None:
            args.steps = 10 if args.impl == "reference" else DEFAULT_STEPS[qwl.name]
        args.warmup = max(3, args.warmup)
        if args.impl == "reference":
            run_reference_qkv(args, qwl)
        else:
            run_gpu_qkv(args, qwl)
        return
    if args.workload in FLOAT_WORKLOADS:
        fwl = FLOAT_WORKLOADS[args.workload]
        if args.steps is None:
            args.steps = 10 if args.impl == "reference" else DEFAULT_STEPS[fwl.name]
        args.warmup = max(3, args.warmup)
        if args.impl == "reference":
            run_reference_float(args, fwl)
        else:
            run_gpu_float(args, fwl)
        return
    # no workload named: the decode line, with the three tensor-bound workloads measured
    # after it in the same process and listed under "workloads"
    extra = EXTRA_WORKLOADS if args.workload is None and not args.only else ()
    wl = WORKLOADS[args.workload or "decode"]
    if args.steps is None:
        args.steps = 10 if args.impl == "reference" else DEFAULT_STEPS[wl.name]
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_gpu(args, wl, extra)


if __name__ == "__main__":
    main()
