"""Benchmark of the GPT-2 small MLP backward (fc then fc_proj) on GB300.

One step = the backward pass of both MLP linear layers of one GPT-2 small
block, B=8, T=1024, bf16 storage, fp32 accumulation, with bias:
    fc      C=768  -> OC=3072
    fc_proj C=3072 -> OC=768
each one call of mmbwd_run (dinp += dout.W, dweight += dout^T.inp, dbias).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Prints one JSON line (rank 0). The metric is TFLOP/s with
FLOPs = 4*B*T*C*OC + B*T*OC (the bias sum) per layer.

* value: device-resident inputs, CUDA events on the launching stream around
  exactly K steps (barrier + synchronize on both sides), three rotating input
  sets (~620 MB) so no step starts with its inputs in the 129 MB L2.
* e2e: the same steps through the same C-ABI call, with pinned HOST inputs:
  every step copies dout, inp, weight host->device and reads dinp, dweight,
  dbias back, copies inside the timed region.
* roofline: the step launches only the tensor-core kernel (one launch per
  layer), so its mean launch time is the timed region over its launches;
  FLOPs per launch over that time, against the measured bf16 peak. Each
  layer alone (back-to-back calls) is reported beside it.
* windows: the K steps cut into up to five windows (events between steps
  only), min / median / max TFLOP/s over them.
* queued start: after the synchronize that opens a timed region, a device
  spin (torch's `_sleep` kernel) holds the stream while the host enqueues the
  timed launches, so the first window measures the device running queued
  work and not the host's latency to its first launch; whether the spin was
  still running when the last launch was queued is reported.
* cpu_baseline / --impl reference: the C oracle (OpenMP build, all host
  cores) on a bounded row sample of the same workload; the single-threaded
  build on a smaller sample beside it.
* other_configs: every other configuration timed alone, each with its
  largest scaled error against the oracle on sampled rows and whether a
  second call from identical buffers repeats every bit.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

WORKLOAD = "mlp"
METRIC = "matmul_backward TFLOP/s at GPT-2 shapes; % of GB300 dense bf16 peak"
UNIT = "TFLOP/s"
N_SETS = 3
N_WINDOWS = 5  # the timed steps are cut into this many windows (events between steps only)
SPIN_CYCLES_PER_US = 2070  # the GB300's maximum SM clock in MHz: a spin of us * this cycles lasts >= us


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-other", action="store_true", help="skip the other configurations")
    ap.add_argument("--no-verify", action="store_true",
                    help="skip the oracle check and repeat check of the other configurations")
    ap.add_argument("--case", default=None,
                    help="time only this one configuration of the other-configs list (for example "
                         "ln_xl or attn_proj) with --steps batches, print its line and exit")
    return ap.parse_args(argv)


def config_dict():
    wl = synth.WORKLOADS[WORKLOAD]
    l0 = wl.layers[0]
    set_bytes = sum(layer_bytes(l) for l in wl.layers)
    return {
        "workload": "gpt2_small_mlp_backward",
        "B": l0.B, "T": l0.T,
        "layers": [{"name": l.name, "C": l.C, "OC": l.OC, "bias": l.bias} for l in wl.layers],
        "dtype_storage": "bf16", "accumulate": "fp32",
        "flops_per_step": wl.flops(),
        "l2": f"{N_SETS} rotating input sets of {set_bytes / 1e6:.0f} MB each (> 129 MB L2)",
        "parallelism": "replicas",
    }


def layer_bytes(l):
    """Bytes of one layer's six tensors (the footprint of an input set)."""
    es = l.elem_bytes()
    return es * (l.BT * l.OC + 2 * l.BT * l.C + 2 * l.OC * l.C + l.OC)


def layer_alg_bytes(l):
    """Algorithmic bytes of one call: dout, inp and weight read once, dinp and
    dweight read and written, dbias written."""
    es = l.elem_bytes()
    return es * (l.BT * l.OC + 3 * l.BT * l.C + 3 * l.OC * l.C + (l.OC if l.bias else 0))


# ----------------------------------------------------------------------------- distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(units: float, seconds: float, group=None):
    """Whole-job throughput over replicas: units summed over ranks, divided by
    the slowest rank's time. Works for any torch.distributed backend."""
    import torch
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized():
        return units, seconds
    t = torch.tensor([units, seconds], dtype=torch.float64)
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = t.to(dev)
    u = t[0:1].clone()
    s = t[1:2].clone()
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    dist.all_reduce(s, op=dist.ReduceOp.MAX, group=group)
    return float(u.item()), float(s.item())


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[4:8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, _, r in rows for i in range(4) if r[i].lower() == "active"})
        load = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(load),
                "power_w_max": max(r[2] for r in rows)}


def gpu_id_for_smi(torch, dev_index: int) -> str:
    try:
        u = torch.cuda.get_device_properties(dev_index).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev_index] if vis else str(dev_index)


# ----------------------------------------------------------------------------- peaks / profile

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_sha() -> str:
    """Hash of the tensor-core kernel's code (comments and white space ignored),
    as the ncu harness writes it into its summaries."""
    from ncu_harness import code_sha

    return code_sha([os.path.join(ROOT, "linear_layer_gemms_gb300", "csrc", f)
                     for f in ("tc_gemm.cu", "ptx.cuh", "internal.h")])


def profiled_traffic():
    """DRAM bytes per launch of the tensor-core kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "tc_mmbwd_kernel_mlp.md")
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p):
        if ":" in line and line.lstrip().startswith("- "):
            k, v = line.lstrip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha") != kernel_source_sha():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------- CPU oracle leg

def oracle_sample(seconds: float, inputs=None, seed=0, variant="omp"):
    """Time the C oracle (`variant` "omp": the OpenMP build on all host cores;
    "st": the single-threaded build) on a bounded row sample of the workload:
    first dinp rows and dweight rows (with the bias) of each layer, as many as
    fill about `seconds`. Returns (TFLOP/s, seconds, desc, threads, flops)."""
    import oracle

    orc = oracle.get(variant)
    wl = synth.WORKLOADS[WORKLOAD]
    if inputs is None:
        inputs = [synth.make_inputs(l, seed) for l in wl.layers]
    # calibrate on a few rows, then size the sample
    rows0 = max(1, orc.threads)
    t0 = time.perf_counter()
    _oracle_rows(orc, wl, inputs, rows0)
    cal = time.perf_counter() - t0
    budget = max(seconds - cal, 0.5)
    rows = max(rows0, int(rows0 * budget / max(cal, 1e-6)))
    rows = min(rows, max(l.BT for l in wl.layers))
    t0 = time.perf_counter()
    flops = _oracle_rows(orc, wl, inputs, rows)
    dt = time.perf_counter() - t0
    desc = (f"{rows} dinp rows and {rows} dweight rows (+dbias) of each MLP layer "
            f"({flops / 1e9:.1f} GFLOP of the {wl.flops() / 1e9:.1f} GFLOP step)")
    return flops / dt / 1e12, dt, desc, orc.threads, flops


def _oracle_rows(orc, wl, inputs, rows):
    flops = 0
    for l, x in zip(wl.layers, inputs):
        r_bt = np.arange(min(rows, l.BT))
        r_o = np.arange(min(rows, l.OC))
        orc.dinp_rows(x["dout"], x["weight"], l.dtype, r_bt, x["dinp"])
        orc.dweight_rows(x["dout"], x["inp"], l.dtype, r_o, x["dweight"], bias=l.bias)
        flops += 2 * len(r_bt) * l.C * l.OC + 2 * len(r_o) * l.BT * l.C + (len(r_o) * l.BT if l.bias else 0)
    return flops


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl = synth.WORKLOADS[WORKLOAD]
    inputs = [synth.make_inputs(l, 0) for l in wl.layers]
    import oracle

    orc = oracle.get("omp")
    total_steps = args.steps + args.warmup
    # rows per step so that the whole run stays within ~90 s
    rows0 = max(1, orc.threads)
    t0 = time.perf_counter()
    f0 = _oracle_rows(orc, wl, inputs, rows0)
    rate = f0 / max(time.perf_counter() - t0, 1e-6)
    per_step_flops = max(f0 / rows0, rate * 90.0 / max(total_steps, 1))
    rows = max(1, int(per_step_flops / (f0 / rows0)))
    for _ in range(args.warmup):
        _oracle_rows(orc, wl, inputs, rows)
    t0 = time.perf_counter()
    flops = 0
    for _ in range(args.steps):
        flops += _oracle_rows(orc, wl, inputs, rows)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = (f"each step: {rows} dinp rows and {rows} dweight rows (+dbias) of each MLP layer "
              f"({flops / args.steps / 1e9:.2f} GFLOP of the {wl.flops() / 1e9:.1f} GFLOP step)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": orc.threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

def to_device_tensor(torch, a, dev):
    t = torch.from_numpy(a)
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.to(dev)


def run_gpu(args):
    import torch

    import linear_layer_gemms_gb300 as mm

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    mm.load()

    def barrier():
        if ws > 1:
            import torch.distributed as dist

            dist.barrier()

    wl = synth.WORKLOADS[WORKLOAD]
    host = [synth.make_inputs(l, seed=0) for l in wl.layers]
    sets = []
    for s in range(N_SETS):
        sets.append([{k: to_device_tensor(torch, v, dev) for k, v in x.items()} for x in host])
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream

    def call(layer, t):
        rc = mm.mmbwd_run(t["dinp"].data_ptr(), t["dweight"].data_ptr(),
                          t["dbias"].data_ptr() if layer.bias else None, t["dout"].data_ptr(),
                          t["inp"].data_ptr(), t["weight"].data_ptr(), layer.B, layer.T, layer.C,
                          layer.OC, mm.BF16, sh)
        if rc != mm.OK:
            raise RuntimeError(f"mmbwd_run: {mm.strerror(rc)}")

    # warm-up (also grows the workspace outside the timed region)
    with torch.cuda.stream(stream):
        t0 = time.perf_counter()
        for k in range(args.warmup):
            for layer, t in zip(wl.layers, sets[k % N_SETS]):
                call(layer, t)
        host_us_step = (time.perf_counter() - t0) * 1e6 / max(1, args.warmup)
    torch.cuda.synchronize()
    status, info = mm.mmbwd_device_status(reset=True)
    if status != mm.OK:
        raise RuntimeError(f"device status after warm-up: {mm.strerror(status)} {info}")

    K = args.steps
    n_win = max(1, min(N_WINDOWS, K))
    bounds = [round(w * K / n_win) for w in range(n_win + 1)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_win + 1)]
    sampler = ClockSampler(gpu_id_for_smi(torch, dev.index)) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier()
    torch.cuda.synchronize()
    # The spin holds the stream while the host queues the K steps (twice the
    # warm-up's host time per step); events only between steps (at window
    # edges): an event between two launches would keep the second launch's
    # prologue from overlapping the first kernel.
    held = hold_stream(torch, stream, min(2e5, 50.0 + 2.0 * host_us_step * K))
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for w in range(n_win):
            for k in range(bounds[w], bounds[w + 1]):
                tset = sets[k % N_SETS]
                for li, layer in enumerate(wl.layers):
                    call(layer, tset[li])
            ev[w + 1].record(stream)
    queued = not held.query()
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop() if sampler else None
    elapsed_s = ev[0].elapsed_time(ev[-1]) / 1e3
    status, info = mm.mmbwd_device_status(reset=True)
    if status != mm.OK:
        raise RuntimeError(f"device status after timed region: {mm.strerror(status)} {info}")

    flops_step = wl.flops()
    units, max_s = aggregate(flops_step * K, elapsed_s)
    value = units / max_s / 1e12
    win_tf = sorted(flops_step * (bounds[w + 1] - bounds[w]) / (ev[w].elapsed_time(ev[w + 1]) / 1e3) / 1e12
                    for w in range(n_win) if bounds[w + 1] > bounds[w])
    windows = {"n": len(win_tf), "steps_each": [bounds[w + 1] - bounds[w] for w in range(n_win)],
               "tflops_min": win_tf[0], "tflops_median": statistics.median(win_tf), "tflops_max": win_tf[-1],
               "queued_before_start": queued, "host_us_per_step": round(host_us_step, 1)}

    # roofline of the tensor-core kernel: the timed step launches only this
    # kernel, one launch per layer, so its mean launch time is this rank's
    # timed region over its launches (gaps between launches included)
    peaks, peak_src = measured_peaks()
    n_launch = K * sum(mm.mmbwd_plan_info(l.B, l.T, l.C, l.OC, mm.BF16, 0)["launches"] for l in wl.layers)
    kernel_flops = flops_step * K
    achieved = kernel_flops / elapsed_s / 1e12
    peak = float(peaks["bf16_tflops"])
    traffic = profiled_traffic()
    # each layer alone: back-to-back calls over the rotating sets
    per_layer = {}
    for li, layer in enumerate(wl.layers):
        calls = [lambda t=sets[k][li], layer=layer: call(layer, t) for k in range(N_SETS)]
        sec = time_back_to_back(torch, stream, calls, 30, 5)
        per_layer[layer.name] = {"us": round(sec * 1e6, 2), "tflops": round(layer.flops() / sec / 1e12, 1),
                                 "timed": "back-to-back calls of this layer alone"}

    # context only: the same step through PyTorch's cuBLAS calls (dinp and
    # dweight by addmm with beta = 1, dbias by a column sum), on the same sets
    library = library_context(torch, wl, sets, stream, flops_step, value)

    # end to end through host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(torch, mm, wl, host, dev, stream, args.e2e_steps, barrier)

    other = None
    if not args.no_other and rank == 0:
        other = measure_other_configs(torch, mm, dev, stream, verify=not args.no_verify)

    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline and ws >= 1:
        v, dt, desc, cores, _ = oracle_sample(args.cpu_seconds, inputs=host)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
               "seconds": round(dt, 2), "build": "OpenMP, -O2, all host cores"}
        v1, dt1, desc1, _, _ = oracle_sample(args.cpu_seconds / 3, inputs=host, variant="st")
        cpu["single_thread"] = {"value": v1, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc1,
                                "seconds": round(dt1, 2), "build": "single-threaded, -O2"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": max_s / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded normal inputs, GPT-2 small MLP shapes)",
        "config": config_dict(),
        "frac_of_bf16_peak": value / peak,
        "windows": windows,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "tc_mmbwd_kernel", "peak_source": f"{peak_src} bf16_tflops (burst)",
                     # context: the timed region runs thousands of launches back to back
                     # under the power cap, the regime of the sustained measurement
                     "frac_of_sustained": achieved / float(peaks["bf16_tflops_sustained"]),
                     "launches": n_launch, "flops_per_launch": kernel_flops / n_launch,
                     "mean_launch_us": elapsed_s / n_launch * 1e6,
                     "timing": "CUDA events around the timed region on the launching stream; every "
                               "launch in it is this kernel's",
                     "per_layer": per_layer},
        "gpu_launches": n_launch,
        "plans": {l.name: mm.mmbwd_plan_info(l.B, l.T, l.C, l.OC, mm.BF16, 0) for l in wl.layers},
        "clocks": clocks,
        "e2e": e2e,
        "library_context": library,
        "cpu_baseline": cpu,
        "other_configs": other,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


OTHER_CONFIGS = ("tiny", "qkv", "attn_proj", "lm_head", "xl_fc_bf16", "xl_qkv_bf16", "xl_fc_f32", "xl_qkv_f32")
LN_CONFIGS = ("ln_gpt2_small", "ln_xl", "ln_xl_f32", "ln_wide")
ENC_CONFIGS = ("enc_gpt2_small", "enc_gpt2_small_f32")
# the same workload in two calls: encbwd_prepare (timed on its own) ahead of
# time, encbwd_run_planned (timed) on the backward's critical path
ENC_PLANNED_CONFIGS = (("enc_gpt2_small_planned", "enc_gpt2_small"),)
# each MLP layer alone, rounded to nearest (mmbwd_run) and stochastically
# (mmbwd_run_sr, a new seed per call)
LAYER_CONFIGS = (("mlp_fc", "mlp:0", False), ("mlp_fc_proj", "mlp:1", False),
                 ("mlp_fc_sr", "mlp:0", True), ("mlp_fc_proj_sr", "mlp:1", True))
# the same layers with dbias formed by an extra MMA against a ones tile
# (MMBWD_DBIAS=ones) instead of the bias warps
DBIAS_MMA_CONFIGS = (("mlp_fc_dbias_mma", "mlp:0"), ("mlp_fc_proj_dbias_mma", "mlp:1"),
                     ("attn_proj_dbias_mma", "attn_proj"))
FORWARD_CONFIGS = (("forward_mlp_fc", "mlp:0"), ("forward_mlp_fc_proj", "mlp:1"),
                   ("forward_lm_head", "lm_head"), ("forward_xl_fc_f32", "xl_fc_f32"))


L2_BYTES = 129 * 1024 * 1024


def library_context(torch, wl, sets, stream, flops_step, value):
    """The benchmark's step through PyTorch (cuBLAS GEMMs, a reduction kernel
    for dbias) on the same device-resident sets: context beside the library's
    number, not part of it."""
    def step(ts):
        for layer, t in zip(wl.layers, ts):
            dout = t["dout"].view(layer.BT, layer.OC)
            inp = t["inp"].view(layer.BT, layer.C)
            t["dinp"].view(layer.BT, layer.C).addmm_(dout, t["weight"].view(layer.OC, layer.C))
            t["dweight"].view(layer.OC, layer.C).addmm_(dout.t(), inp)
            if layer.bias:
                torch.sum(dout, 0, out=t["dbias"].view(layer.OC))
    try:
        sec = time_back_to_back(torch, stream, [lambda ts=ts: step(ts) for ts in sets], 30, 5)
    except RuntimeError as e:  # a PyTorch without these kernels for the type
        return {"unavailable": str(e).splitlines()[0]}
    tf = flops_step / sec / 1e12
    return {"impl": "torch addmm (cuBLAS) + torch.sum", "tflops": round(tf, 1), "ms_per_step": round(sec * 1e3, 4),
            "library_over_torch": round(value / tf, 3), "timed": "back-to-back steps over the rotating sets"}


def hold_stream(torch, stream, us):
    """Queue on `stream` a device spin of at least `us` microseconds and return
    an event recorded behind it. Launches enqueued next wait behind the spin,
    so a timed window that starts after it starts with its work queued; the
    event not yet complete once the last launch is queued shows that held."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * SPIN_CYCLES_PER_US))
        e = torch.cuda.Event()
        e.record(stream)
    return e


def time_back_to_back(torch, stream, calls, per_batch, batches=5):
    """Median over `batches` of (time of `per_batch` back-to-back calls) /
    per_batch, CUDA events on `stream`; the calls cycle through `calls` (one
    per resident input set) so that consecutive calls touch different memory.
    Each batch is queued behind a device spin (`hold_stream`), lengthened and
    the batch taken again if the spin ended before the batch was queued."""
    with torch.cuda.stream(stream):
        t0 = time.perf_counter()
        for c in calls * 2:
            c()
        host_us = (time.perf_counter() - t0) * 1e6 / (2 * len(calls))
    torch.cuda.synchronize()
    hold_us = 50.0 + 2.0 * host_us * per_batch
    times = []
    for _ in range(batches):
        while True:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            held = hold_stream(torch, stream, hold_us)
            with torch.cuda.stream(stream):
                a.record(stream)
                for k in range(per_batch):
                    calls[k % len(calls)]()
                b.record(stream)
            queued = not held.query()
            b.synchronize()
            if queued or hold_us > 1e5:
                break
            hold_us *= 2
        times.append(a.elapsed_time(b) / 1e3 / per_batch)
    return statistics.median(times)


VERIFY_ROWS = 48  # seeded random rows checked per product, beside the tile-edge rows
TOL = {"bf16": 2e-2, "f32": 1e-4}  # |gpu - ref| <= tau * (|ref| + rms(ref)), per output tensor


def _check_rows(n, seed):
    """Rows at tile edges and seeded random rows of an n-row output."""
    edges = [0, 1, 127, 128, 255, 256, n // 2, n - 129, n - 128, n - 1]
    rng = np.random.default_rng(seed)
    rows = {r for r in edges if 0 <= r < n} | {int(r) for r in rng.integers(0, n, VERIFY_ROWS)}
    return np.array(sorted(rows), dtype=np.int64)


def _scaled_error(got, ref):
    """max |got - ref| / (|ref| + rms(ref)); rms over the checked elements."""
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    den = np.abs(ref) + rms
    return float(np.max(np.abs(got - ref) / np.where(den == 0, 1.0, den)))


def _to_f64(torch, t, dtype):
    if dtype == "bf16":
        return synth.bf16_bits_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.cpu().numpy().astype(np.float64)


def _same_bits(torch, a, b):
    return bool(torch.equal(a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                            b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32)))


def verify_backward(torch, mm, layer, x, dev, sr=False):
    """Two calls of mmbwd_run (or mmbwd_run_sr with one seed) from identical
    buffers: whether every output bit repeats, and the largest scaled error of
    the first call against the oracle on sampled rows of dinp and dweight and
    on every dbias element."""
    import oracle

    dt = mm.BF16 if layer.dtype == "bf16" else mm.F32
    outs = []
    for _ in range(2):
        t = {k: to_device_tensor(torch, v, dev) for k, v in x.items()}
        args = (t["dinp"], t["dweight"], t["dbias"] if layer.bias else None, t["dout"], t["inp"], t["weight"],
                layer.B, layer.T, layer.C, layer.OC, dt)
        rc = mm.mmbwd_run_sr(*args, 12345) if sr else mm.mmbwd_run(*args)
        if rc != mm.OK:
            raise RuntimeError(mm.strerror(rc))
        torch.cuda.synchronize()
        outs.append(t)
    repeat = all(_same_bits(torch, outs[0][k], outs[1][k]) for k in ("dinp", "dweight", "dbias"))
    orc = oracle.get("omp")
    rb, ro = _check_rows(layer.BT, 1), _check_rows(layer.OC, 2)
    g = outs[0]
    errs = {"dinp": _scaled_error(_to_f64(torch, g["dinp"][torch.from_numpy(rb).to(dev)], layer.dtype),
                                  orc.dinp_rows(x["dout"], x["weight"], layer.dtype, rb, x["dinp"])),
            "dweight": _scaled_error(_to_f64(torch, g["dweight"][torch.from_numpy(ro).to(dev)], layer.dtype),
                                     orc.dweight_rows(x["dout"], x["inp"], layer.dtype, ro, x["dweight"],
                                                      bias=False)[0])}
    if layer.bias:
        empty = np.zeros((layer.BT, 0), dtype=x["inp"].dtype)
        errs["dbias"] = _scaled_error(_to_f64(torch, g["dbias"], layer.dtype),
                                      orc.dweight_rows(x["dout"], empty, layer.dtype, None, None, bias=True)[1])
    del outs
    return {"max_scaled_error": max(errs.values()), "tolerance": TOL[layer.dtype], "bitwise_repeat": repeat,
            "checked": f"{len(rb)} dinp rows, {len(ro)} dweight rows" + (", every dbias element" if layer.bias else "")
                       + " against the OpenMP oracle; a second call from identical buffers for the repeat"}


def verify_encoder(torch, p, x, dev, run, like):
    """Two runs of the encoder backward (`run(t)` on buffers shaped like
    `like`) from identical buffers: whether every bit repeats, and the largest
    scaled error of the first against the oracle (every element)."""
    import oracle

    outs = []
    for _ in range(2):
        t = {k: to_device_tensor(torch, x[k], dev) for k in ("dout", "dwte", "dwpe")}
        t["inp"] = torch.from_numpy(x["inp"]).to(dev)
        run(t)
        torch.cuda.synchronize()
        outs.append(t)
    rte, rpe = oracle.get("omp").encoder_backward(x["dout"], x["inp"], p.B, p.T, p.V, p.dtype, x["dwte"], x["dwpe"])
    g = outs[0]
    err = max(_scaled_error(_to_f64(torch, g["dwte"], p.dtype), rte),
              _scaled_error(_to_f64(torch, g["dwpe"], p.dtype), rpe))
    rep = all(_same_bits(torch, outs[0][k], outs[1][k]) for k in ("dwte", "dwpe"))
    return {"max_scaled_error": err, "tolerance": TOL[p.dtype], "bitwise_repeat": rep,
            "checked": "every dwte and dwpe element against the OpenMP oracle; a second run from identical "
                       "buffers for the repeat"}


def input_sets(nbytes_one, cap=8):
    """How many copies of a configuration's tensors to rotate through so that
    they span more than the L2 (capped; tiny problems stay L2-resident)."""
    return max(1, min(cap, -(-2 * L2_BYTES // max(nbytes_one, 1))))


def enc_input_sets(torch, x, set_bytes, dev):
    """Copies of an encoder problem (dout, token ids, dwte, dwpe) to rotate
    through, enough that the bytes one call touches span twice the L2 (at most
    24); the first is copied from the host, the others cloned on the device."""
    n = input_sets(set_bytes, cap=24)
    first = {k: to_device_tensor(torch, x[k], dev) for k in ("dout", "dwte", "dwpe")}
    first["inp"] = torch.from_numpy(x["inp"]).to(dev)
    return n, [first] + [{k: v.clone() for k, v in first.items()} for _ in range(n - 1)]


def measure_other_configs(torch, mm, dev, stream, only=None, batches=5, verify=True):
    """The remaining configurations of the workload set and the forward of the
    GPT-2 layers: back-to-back calls on device-resident inputs rotated over
    enough copies to exceed the L2 (see `input_sets`), timed with CUDA events,
    reported with their plan and the fraction of the peak that bounds them:
    the measured bf16 tensor peak for bf16; for fp32, the peak of the path the
    plan chose -- the TF32 tensor peak (the measured bf16 peak x the nominal
    tf32/bf16 ratio 1.1/2.25) for the three-product tensor-core path, whose own
    ceiling is a third of it, or the FP32 ALU peak (152 SMs x 128 lanes x 2
    FLOP at the maximum SM clock) for the FMA kernel."""
    peaks, _ = measured_peaks()
    fp32_peak = 152 * 128 * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12
    tf32_peak = float(peaks["bf16_tflops"]) * 1.1 / 2.25
    sh = stream.cuda_stream
    out = {}

    hbm = float(peaks.get("hbm_gbs", 6800.0))

    def finish(name, layer, flops, sec, n_sets, set_bytes, plan=None, alg_bytes=None):
        tf = flops / sec / 1e12
        rec = {"B": layer.B, "T": layer.T, "C": layer.C, "OC": layer.OC, "dtype": layer.dtype,
               "bias": layer.bias, "us": round(sec * 1e6, 2), "tflops": round(tf, 2)}
        if alg_bytes:  # the same time against HBM: algorithmic bytes (inputs once, outputs read and written)
            gbs = alg_bytes / sec / 1e9
            rec.update(alg_bytes=alg_bytes, gb_per_s=round(gbs, 1), frac_of_hbm=round(gbs / hbm, 4),
                       hbm_peak=f"HBM copy (measured) {hbm:.0f} GB/s")
        if layer.dtype == "bf16":
            rec.update(frac_of_peak=round(tf / float(peaks["bf16_tflops"]), 4), peak="bf16 tensor (measured)")
        elif plan is not None and plan.get("path") == 2:
            rec.update(frac_of_peak=round(tf / tf32_peak, 4),
                       frac_of_3xtf32_ceiling=round(3 * tf / tf32_peak, 4),
                       peak=f"tf32 tensor {tf32_peak:.0f} TFLOP/s (measured bf16 x 1.1/2.25); "
                            "three tf32 products per fp32 product")
        else:
            rec.update(frac_of_peak=round(tf / fp32_peak, 4),
                       peak=f"fp32 ALU {fp32_peak:.1f} TFLOP/s (152 SMs x 128 lanes x 2 x max clock)")
        rec.update(input_sets=n_sets, l2="rotating sets > L2" if n_sets * set_bytes > L2_BYTES else "L2-resident")
        out[name] = rec
        if plan is not None:
            out[name]["plan"] = plan

    backward = ([(n, n, False) for n in OTHER_CONFIGS] + list(LAYER_CONFIGS) +
                [(n, spec, False) for n, spec in DBIAS_MMA_CONFIGS])
    dbias_mma = {n for n, _ in DBIAS_MMA_CONFIGS}
    for name, spec, sr in backward:
        if only is not None and name not in only:
            continue
        if name in dbias_mma:
            os.environ["MMBWD_DBIAS"] = "ones"
        else:
            os.environ.pop("MMBWD_DBIAS", None)
        wl, _, i = spec.partition(":")
        layer = synth.WORKLOADS[wl].layers[int(i or 0)]
        x = synth.make_inputs(layer, seed=0)
        set_bytes = sum(v.nbytes for v in x.values())
        n_sets = input_sets(set_bytes)
        sets = [{k: to_device_tensor(torch, v, dev) for k, v in x.items()} for _ in range(n_sets)]
        dt = mm.BF16 if layer.dtype == "bf16" else mm.F32

        def make_call(t, layer=layer, dt=dt, sr=sr):
            seeds = iter(range(1, 1 << 62))

            def call():
                args = (t["dinp"].data_ptr(), t["dweight"].data_ptr(), t["dbias"].data_ptr() if layer.bias else None,
                        t["dout"].data_ptr(), t["inp"].data_ptr(), t["weight"].data_ptr(), layer.B, layer.T,
                        layer.C, layer.OC, dt)
                rc = mm.mmbwd_run_sr(*args, next(seeds), sh) if sr else mm.mmbwd_run(*args, sh)
                if rc != mm.OK:
                    raise RuntimeError(mm.strerror(rc))
            return call

        calls = [make_call(t) for t in sets]
        per_batch = max(len(calls), 20 if layer.flops() < 5e11 else 8)
        sec = time_back_to_back(torch, stream, calls, per_batch, batches)
        info = mm.mmbwd_plan_info(layer.B, layer.T, layer.C, layer.OC, dt, 0)
        finish(name, layer, layer.flops(), sec, n_sets, set_bytes,
               {k: info[k] for k in ("path", "grid", "items", "splits", "launches")}, alg_bytes=layer_alg_bytes(layer))
        if layer.dtype == "bf16" and not sr and name not in dbias_mma:
            # context only: the same backward through PyTorch's cuBLAS calls
            def torch_step(t, layer=layer):
                dout = t["dout"].view(layer.BT, layer.OC)
                t["dinp"].view(layer.BT, layer.C).addmm_(dout, t["weight"].view(layer.OC, layer.C))
                t["dweight"].view(layer.OC, layer.C).addmm_(dout.t(), t["inp"].view(layer.BT, layer.C))
                if layer.bias:
                    torch.sum(dout, 0, out=t["dbias"].view(layer.OC))
            tsec = time_back_to_back(torch, stream, [lambda t=t: torch_step(t) for t in sets], per_batch, batches)
            out[name]["torch_cublas_us"] = round(tsec * 1e6, 2)
        if sr:
            out[name]["rounding"] = "stochastic (mmbwd_run_sr, new seed per call)"
        del sets, calls
        torch.cuda.empty_cache()
        if verify:
            out[name].update(verify_backward(torch, mm, layer, x, dev, sr))
            torch.cuda.empty_cache()
        if name in dbias_mma:
            out[name]["dbias"] = "extra pair MMA against a ones tile (MMBWD_DBIAS=ones)"
        os.environ.pop("MMBWD_DBIAS", None)
    # the forward of the same layers (mmbwd_forward): 2*B*T*C*OC FLOPs (+ B*T*OC with the bias)
    for name, lname in FORWARD_CONFIGS:
        if only is not None and name not in only:
            continue
        wl, _, i = lname.partition(":")
        layer = synth.WORKLOADS[wl].layers[int(i or 0)]
        x = synth.make_inputs(layer, seed=0)
        set_bytes = x["inp"].nbytes + x["weight"].nbytes + x["dbias"].nbytes + layer.BT * layer.OC * x["inp"].itemsize
        n_sets = input_sets(set_bytes)
        sets = []
        for _ in range(n_sets):
            t = {k: to_device_tensor(torch, x[k], dev) for k in ("inp", "weight", "dbias")}
            t["out"] = torch.empty((layer.BT, layer.OC), dtype=t["inp"].dtype, device=dev)
            sets.append(t)
        dt = mm.BF16 if layer.dtype == "bf16" else mm.F32

        def make_fcall(t, layer=layer, dt=dt):
            def fcall():
                rc = mm.mmbwd_forward(t["out"].data_ptr(), t["inp"].data_ptr(), t["weight"].data_ptr(),
                                      t["dbias"].data_ptr() if layer.bias else None, layer.B, layer.T,
                                      layer.C, layer.OC, dt, sh)
                if rc != mm.OK:
                    raise RuntimeError(mm.strerror(rc))
            return fcall

        calls = [make_fcall(t) for t in sets]
        flops = 2 * layer.BT * layer.C * layer.OC + (layer.BT * layer.OC if layer.bias else 0)
        per_batch = max(len(calls), 20 if flops < 2.5e11 else 8)
        sec = time_back_to_back(torch, stream, calls, per_batch, batches)
        es = layer.elem_bytes()
        finish(name, layer, flops, sec, n_sets, set_bytes,
               {"path": mm.mmbwd_forward_path(layer.B, layer.T, layer.C, layer.OC, dt)},
               alg_bytes=es * (layer.BT * layer.C + layer.OC * layer.C + layer.BT * layer.OC
                               + (layer.OC if layer.bias else 0)))
        if verify:
            t = sets[0]
            first = t["out"].clone()
            make_fcall(t)()
            torch.cuda.synchronize()
            import oracle

            rows = _check_rows(layer.BT, 3)
            ref = oracle.get("omp").forward_rows(x["inp"], x["weight"], layer.dtype, rows,
                                                 bias=x["dbias"] if layer.bias else None)
            err = _scaled_error(_to_f64(torch, t["out"][torch.from_numpy(rows).to(dev)], layer.dtype), ref)
            out[name].update(max_scaled_error=err, tolerance=TOL[layer.dtype],
                             bitwise_repeat=_same_bits(torch, first, t["out"]),
                             checked=f"{len(rows)} rows of out against the OpenMP oracle; the previous "
                                     "call's output for the repeat")
        del sets, calls
        torch.cuda.empty_cache()
    # the LayerNorm backward (lnbwd_run): bound by HBM, reported in GB/s of
    # algorithmic bytes against the measured copy bandwidth
    for name in LN_CONFIGS:
        if only is not None and name not in only:
            continue
        p = synth.LN_WORKLOADS[name]
        x = synth.make_ln_inputs(p, seed=0)
        # row statistics as the forward caches them (fp32), computed on the host
        xi = synth.to_f64(x["inp"], p.dtype)
        mean = xi.mean(axis=1).astype(np.float32)
        rstd = (1.0 / np.sqrt(xi.var(axis=1) + 1e-5)).astype(np.float32)
        set_bytes = p.bytes()
        n_sets = input_sets(set_bytes)
        sets = []
        for _ in range(n_sets):
            t = {k: to_device_tensor(torch, v, dev) for k, v in x.items()}
            t["mean"], t["rstd"] = torch.from_numpy(mean).to(dev), torch.from_numpy(rstd).to(dev)
            sets.append(t)
        dt = mm.BF16 if p.dtype == "bf16" else mm.F32

        def make_lcall(t, p=p, dt=dt):
            def lcall():
                rc = mm.lnbwd_run(t["dinp"].data_ptr(), t["dweight"].data_ptr(), t["dbias"].data_ptr(),
                                  t["dout"].data_ptr(), t["inp"].data_ptr(), t["weight"].data_ptr(),
                                  t["mean"].data_ptr(), t["rstd"].data_ptr(), p.B, p.T, p.C, dt, sh)
                if rc != mm.OK:
                    raise RuntimeError(mm.strerror(rc))
            return lcall

        calls = [make_lcall(t) for t in sets]
        sec = time_back_to_back(torch, stream, calls, max(len(calls), 40), batches)
        gbs = p.bytes() / sec / 1e9
        out[name] = {"B": p.B, "T": p.T, "C": p.C, "dtype": p.dtype, "us": round(sec * 1e6, 2),
                     "gb_per_s": round(gbs, 1), "frac_of_peak": round(gbs / hbm, 4),
                     "peak": f"HBM copy (measured) {hbm:.0f} GB/s", "bytes": p.bytes(),
                     "input_sets": n_sets,
                     "l2": "rotating sets > L2" if n_sets * set_bytes > L2_BYTES else "L2-resident"}
        del sets, calls
        torch.cuda.empty_cache()
        if verify:
            import oracle

            orc = oracle.get("omp")
            outs = []
            for _ in range(2):
                t = {k: to_device_tensor(torch, v, dev) for k, v in x.items()}
                t["mean"], t["rstd"] = torch.from_numpy(mean).to(dev), torch.from_numpy(rstd).to(dev)
                make_lcall(t)()
                torch.cuda.synchronize()
                outs.append(t)
            rows = _check_rows(p.BT, 4)
            g = outs[0]
            e = [_scaled_error(_to_f64(torch, g["dinp"][torch.from_numpy(rows).to(dev)], p.dtype),
                               orc.layernorm_dinp_rows(x["dout"], x["inp"], x["weight"], mean, rstd, p.dtype, rows,
                                                       x["dinp"]))]
            rdw, rdb = orc.layernorm_params(x["dout"], x["inp"], mean, rstd, p.dtype, x["dweight"], x["dbias"])
            e += [_scaled_error(_to_f64(torch, g["dweight"], p.dtype), rdw),
                  _scaled_error(_to_f64(torch, g["dbias"], p.dtype), rdb)]
            out[name].update(max_scaled_error=max(e), tolerance=TOL[p.dtype],
                             bitwise_repeat=all(_same_bits(torch, outs[0][k], outs[1][k])
                                                for k in ("dinp", "dweight", "dbias")),
                             checked=f"{len(rows)} dinp rows, every dweight and dbias element against the "
                                     "OpenMP oracle; a second call from identical buffers for the repeat")
            del outs
            torch.cuda.empty_cache()
    # the encoder backward (encbwd_run): bound by HBM, GB/s of algorithmic bytes
    for name in ENC_CONFIGS:
        if only is not None and name not in only:
            continue
        p = synth.ENC_WORKLOADS[name]
        x = synth.make_enc_inputs(p, seed=0)
        distinct = int(np.unique(x["inp"]).size)
        set_bytes = p.bytes(distinct)
        n_sets, sets = enc_input_sets(torch, x, set_bytes, dev)
        dt = mm.BF16 if p.dtype == "bf16" else mm.F32

        def make_ecall(t, p=p, dt=dt):
            def ecall():
                rc = mm.encbwd_run(t["dwte"].data_ptr(), t["dwpe"].data_ptr(), t["dout"].data_ptr(),
                                   t["inp"].data_ptr(), p.B, p.T, p.C, p.V, dt, sh)
                if rc != mm.OK:
                    raise RuntimeError(mm.strerror(rc))
            return ecall

        calls = [make_ecall(t) for t in sets]
        sec = time_back_to_back(torch, stream, calls, max(len(calls), 40), batches)
        gbs = set_bytes / sec / 1e9
        check = verify_encoder(torch, p, x, dev, lambda t: make_ecall(t)(), sets[0]) if verify else {}
        out[name] = {"B": p.B, "T": p.T, "C": p.C, "V": p.V, "dtype": p.dtype, "us": round(sec * 1e6, 2),
                     "gb_per_s": round(gbs, 1), "frac_of_peak": round(gbs / hbm, 4),
                     "peak": f"HBM copy (measured) {hbm:.0f} GB/s", "bytes": set_bytes,
                     "tokens": f"Zipf(s=1.1) over 50257 ids, {distinct} distinct", "input_sets": n_sets,
                     "l2": "rotating sets > L2" if n_sets * set_bytes > L2_BYTES else "L2-resident", **check}
        del sets, calls
        torch.cuda.empty_cache()
    for name, wname in ENC_PLANNED_CONFIGS:
        if only is not None and name not in only:
            continue
        p = synth.ENC_WORKLOADS[wname]
        x = synth.make_enc_inputs(p, seed=0)
        distinct = int(np.unique(x["inp"]).size)
        set_bytes = p.bytes(distinct)
        n_sets, sets = enc_input_sets(torch, x, set_bytes, dev)
        dt = mm.BF16 if p.dtype == "bf16" else mm.F32
        nplan = mm.encbwd_plan_bytes(p.B, p.T, p.C, p.V, dt)
        for t in sets:
            t["plan"] = torch.empty(nplan, dtype=torch.uint8, device=dev)

        def make_prep(t, p=p, dt=dt):
            def prep():
                rc = mm.encbwd_prepare(t["plan"].data_ptr(), nplan, t["inp"].data_ptr(), p.B, p.T, p.C, p.V, dt, sh)
                if rc != mm.OK:
                    raise RuntimeError(mm.strerror(rc))
            return prep

        def make_run(t, p=p, dt=dt):
            def run():
                rc = mm.encbwd_run_planned(t["dwte"].data_ptr(), t["dwpe"].data_ptr(), t["dout"].data_ptr(),
                                           t["plan"].data_ptr(), p.B, p.T, p.C, p.V, dt, None, sh)
                if rc != mm.OK:
                    raise RuntimeError(mm.strerror(rc))
            return run

        preps = [make_prep(t) for t in sets]
        sec_prep = time_back_to_back(torch, stream, preps, max(len(preps), 40), batches)
        runs = [make_run(t) for t in sets]
        sec = time_back_to_back(torch, stream, runs, max(len(runs), 40), batches)
        gbs = set_bytes / sec / 1e9

        def planned(t, p=p, dt=dt):
            t["plan"] = torch.empty(nplan, dtype=torch.uint8, device=dev)
            make_prep(t)()
            make_run(t)()

        check = verify_encoder(torch, p, x, dev, planned, sets[0]) if verify else {}
        out[name] = {"B": p.B, "T": p.T, "C": p.C, "V": p.V, "dtype": p.dtype, "us": round(sec * 1e6, 2),
                     "gb_per_s": round(gbs, 1), "frac_of_peak": round(gbs / hbm, 4),
                     "peak": f"HBM copy (measured) {hbm:.0f} GB/s", "bytes": set_bytes,
                     "prepare_us": round(sec_prep * 1e6, 2),
                     "timed": "encbwd_run_planned; encbwd_prepare (the sort of the token ids) timed apart",
                     "tokens": f"Zipf(s=1.1) over 50257 ids, {distinct} distinct", "input_sets": n_sets,
                     "l2": "rotating sets > L2" if n_sets * set_bytes > L2_BYTES else "L2-resident", **check}
        del sets, preps, runs
        torch.cuda.empty_cache()
    status, info = mm.mmbwd_device_status(reset=True)
    if status != mm.OK:
        raise RuntimeError(f"device status after other configs: {mm.strerror(status)} {info}")
    return out


def run_e2e(torch, mm, wl, host, dev, stream, steps, barrier):
    """Same steps through mmbwd_run with pinned host inputs: every step copies
    its dout, inp and weight in and its dinp, dweight and dbias out, inside the
    timed region. Pipelined as a training loop would run it: a copy-in stream,
    the compute stream and a copy-out stream, two device buffer sets used by
    alternate steps, events ordering each buffer's copy-in, compute and
    copy-out (step k's copy-in waits for step k-2's compute on the same set,
    step k's compute for step k-2's copy-out)."""
    pin_in = [{k: torch.from_numpy(x[k]).pin_memory() for k in ("dout", "inp", "weight")} for x in host]
    pin_out = [{k: torch.from_numpy(x[k].copy()).pin_memory() for k in ("dinp", "dweight", "dbias")} for x in host]
    sets = [[{k: to_device_tensor(torch, v, dev) for k, v in x.items()} for x in host] for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for x in pin_in for v in x.values())
    d2h = sum(v.numel() * v.element_size() for x in pin_out for v in x.values())
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    ev = {(name, b): None for name in ("in", "comp", "out") for b in (0, 1)}

    def record(name, b, st):
        e = torch.cuda.Event()
        e.record(st)
        ev[(name, b)] = e

    def step(k):
        b = k % 2
        d = sets[b]
        with torch.cuda.stream(s_in):
            if ev[("comp", b)] is not None:
                s_in.wait_event(ev[("comp", b)])
            for pi, t in zip(pin_in, d):
                for key in ("dout", "inp", "weight"):
                    t[key].view(torch.int16).copy_(pi[key].view(torch.int16), non_blocking=True)
            record("in", b, s_in)
        stream.wait_event(ev[("in", b)])
        if ev[("out", b)] is not None:
            stream.wait_event(ev[("out", b)])
        for layer, t in zip(wl.layers, d):
            rc = mm.mmbwd_run(t["dinp"].data_ptr(), t["dweight"].data_ptr(),
                              t["dbias"].data_ptr() if layer.bias else None, t["dout"].data_ptr(),
                              t["inp"].data_ptr(), t["weight"].data_ptr(), layer.B, layer.T, layer.C,
                              layer.OC, mm.BF16, sh)
            if rc != mm.OK:
                raise RuntimeError(mm.strerror(rc))
        record("comp", b, stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev[("comp", b)])
            for po, t in zip(pin_out, d):
                for key in ("dinp", "dweight", "dbias"):
                    po[key].view(torch.int16).copy_(t[key].view(torch.int16), non_blocking=True)
            record("out", b, s_out)

    for k in range(3):
        step(k)
    torch.cuda.synchronize()
    a, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    a.record(s_in)  # before the first copy-in
    for k in range(steps):
        step(k)
    s_in.wait_event(ev[("out", (steps - 1) % 2)])  # after the last copy-out
    e_end.record(s_in)
    torch.cuda.synchronize()
    barrier()
    s = a.elapsed_time(e_end) / 1e3
    units, max_s = aggregate(wl.flops() * steps, s)
    return {"value": units / max_s / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": max_s / steps * 1e3,
            "pipelined": "copy-in, compute and copy-out streams; two device buffer sets"}


def run_case(args):
    """One configuration of the other-configs list on its own (used to profile
    a single kernel): its usual timing with `--steps` batches, one JSON line."""
    import torch

    import linear_layer_gemms_gb300 as mm

    names = (set(OTHER_CONFIGS) | set(LN_CONFIGS) | set(ENC_CONFIGS) | {n for n, _ in FORWARD_CONFIGS}
             | {n for n, _ in DBIAS_MMA_CONFIGS}
             | {n for n, _, _ in LAYER_CONFIGS} | {n for n, _ in ENC_PLANNED_CONFIGS})
    if args.case not in names:
        raise SystemExit(f"unknown case {args.case}; one of {sorted(names)}")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    mm.load()
    stream = torch.cuda.Stream(device=dev)
    out = measure_other_configs(torch, mm, dev, stream, only={args.case}, batches=max(1, args.steps),
                                verify=not args.no_verify)
    print(json.dumps({"case": args.case, **out[args.case]}))
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.case:
        return run_case(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
