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
* roofline: the tensor-core kernel's FLOPs per launch / its mean launch time
  (events around each launch), against the measured bf16 peak.
* cpu_baseline / --impl reference: the C oracle (OpenMP build, all host
  cores) on a bounded row sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
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
sys.path.insert(0, ROOT)

import synth  # noqa: E402

WORKLOAD = "mlp"
METRIC = "matmul_backward TFLOP/s at GPT-2 shapes; % of GB300 dense bf16 peak"
UNIT = "TFLOP/s"
N_SETS = 3
EVENT_EVERY = 4  # steps between the ones timed launch by launch (for the roofline)


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
    es = l.elem_bytes()
    return es * (l.BT * l.OC + 2 * l.BT * l.C + 2 * l.OC * l.C + l.OC)


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
    h = hashlib.sha1()
    for f in ("tc_gemm.cu", "ptx.cuh", "internal.h"):
        with open(os.path.join(ROOT, "linear_layer_gemms_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


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

def oracle_sample(seconds: float, inputs=None, seed=0):
    """Time the C oracle (OpenMP build, all host cores) on a bounded row sample
    of the workload: first dinp rows and dweight rows (with the bias) of each
    layer, as many as fill about `seconds`. Returns (TFLOP/s, seconds, desc, threads)."""
    import oracle

    orc = oracle.get("omp")
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
        for k in range(args.warmup):
            for layer, t in zip(wl.layers, sets[k % N_SETS]):
                call(layer, t)
    torch.cuda.synchronize()
    status, info = mm.mmbwd_device_status(reset=True)
    if status != mm.OK:
        raise RuntimeError(f"device status after warm-up: {mm.strerror(status)} {info}")

    K = args.steps
    L = len(wl.layers)
    ev = {k: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(L)] for k in range(0, K, EVENT_EVERY)}
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_id_for_smi(torch, dev.index)) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier()
    torch.cuda.synchronize()
    # Per-launch events on every EVENT_EVERY-th step only (they sit between
    # launches and would otherwise keep the next launch's prologue from
    # overlapping the previous kernel on every step).
    with torch.cuda.stream(stream):
        e_start.record(stream)
        for k in range(K):
            tset = sets[k % N_SETS]
            timed = k % EVENT_EVERY == 0
            for li, layer in enumerate(wl.layers):
                if timed:
                    ev[k][li][0].record(stream)
                call(layer, tset[li])
                if timed:
                    ev[k][li][1].record(stream)
        e_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop() if sampler else None
    elapsed_s = e_start.elapsed_time(e_end) / 1e3
    status, info = mm.mmbwd_device_status(reset=True)
    if status != mm.OK:
        raise RuntimeError(f"device status after timed region: {mm.strerror(status)} {info}")

    launch_ms = [[ev[k][li][0].elapsed_time(ev[k][li][1]) for k in range(0, K, EVENT_EVERY)] for li in range(L)]
    flops_step = wl.flops()
    units, max_s = aggregate(flops_step * K, elapsed_s)
    value = units / max_s / 1e12

    # roofline of the tensor-core kernel (the only kernel these launches run)
    peaks, peak_src = measured_peaks()
    kernel_flops = sum(l.flops() for l in wl.layers) * len(launch_ms[0])
    kernel_s = sum(sum(x) for x in launch_ms) / 1e3
    achieved = kernel_flops / kernel_s / 1e12
    peak = float(peaks["bf16_tflops"])
    traffic = profiled_traffic()

    # end to end through host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(torch, mm, wl, host, dev, stream, args.e2e_steps, barrier)

    other = None
    if not args.no_other and rank == 0:
        other = measure_other_configs(torch, mm, dev, stream)

    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline and ws >= 1:
        v, dt, desc, cores, _ = oracle_sample(args.cpu_seconds, inputs=host)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
               "seconds": round(dt, 2)}

    per_layer = {l.name: {"mean_us": 1e3 * statistics.mean(launch_ms[i]),
                          "tflops": l.flops() / (statistics.mean(launch_ms[i]) / 1e3) / 1e12}
                 for i, l in enumerate(wl.layers)}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": max_s / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded normal inputs, GPT-2 small MLP shapes)",
        "config": config_dict(),
        "frac_of_bf16_peak": value / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "tc_mmbwd_kernel", "peak_source": f"{peak_src} bf16_tflops (burst)",
                     "per_layer": per_layer},
        "gpu_launches": K * sum(mm.mmbwd_plan_info(l.B, l.T, l.C, l.OC, mm.BF16, 0)["launches"]
                                for l in wl.layers),
        "plans": {l.name: mm.mmbwd_plan_info(l.B, l.T, l.C, l.OC, mm.BF16, 0) for l in wl.layers},
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "other_configs": other,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


OTHER_CONFIGS = ("tiny", "attn_proj", "lm_head", "xl_fc_bf16", "xl_qkv_bf16", "xl_fc_f32", "xl_qkv_f32")
LN_CONFIGS = ("ln_gpt2_small", "ln_xl", "ln_xl_f32")
ENC_CONFIGS = ("enc_gpt2_small", "enc_gpt2_small_f32")
# the same workload in two calls: encbwd_prepare (timed on its own) ahead of
# time, encbwd_run_planned (timed) on the backward's critical path
ENC_PLANNED_CONFIGS = (("enc_gpt2_small_planned", "enc_gpt2_small"),)
# each MLP layer alone, rounded to nearest (mmbwd_run) and stochastically
# (mmbwd_run_sr, a new seed per call)
LAYER_CONFIGS = (("mlp_fc", "mlp:0", False), ("mlp_fc_proj", "mlp:1", False),
                 ("mlp_fc_sr", "mlp:0", True), ("mlp_fc_proj_sr", "mlp:1", True))
FORWARD_CONFIGS = (("forward_mlp_fc", "mlp:0"), ("forward_mlp_fc_proj", "mlp:1"),
                   ("forward_lm_head", "lm_head"), ("forward_xl_fc_f32", "xl_fc_f32"))


L2_BYTES = 129 * 1024 * 1024


def time_back_to_back(torch, stream, calls, per_batch, batches=5):
    """Median over `batches` of (time of `per_batch` back-to-back calls) /
    per_batch, CUDA events on `stream`; the calls cycle through `calls` (one
    per resident input set) so that consecutive calls touch different memory."""
    with torch.cuda.stream(stream):
        for c in calls * 2:
            c()
    torch.cuda.synchronize()
    times = []
    for _ in range(batches):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for k in range(per_batch):
                calls[k % len(calls)]()
            b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b) / 1e3 / per_batch)
    return statistics.median(times)


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


def measure_other_configs(torch, mm, dev, stream, only=None, batches=5):
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

    def finish(name, layer, flops, sec, n_sets, set_bytes, plan=None):
        tf = flops / sec / 1e12
        rec = {"B": layer.B, "T": layer.T, "C": layer.C, "OC": layer.OC, "dtype": layer.dtype,
               "bias": layer.bias, "us": round(sec * 1e6, 2), "tflops": round(tf, 2)}
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

    backward = [(n, n, False) for n in OTHER_CONFIGS] + list(LAYER_CONFIGS)
    for name, spec, sr in backward:
        if only is not None and name not in only:
            continue
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
               {k: info[k] for k in ("path", "grid", "items", "splits", "launches")})
        if sr:
            out[name]["rounding"] = "stochastic (mmbwd_run_sr, new seed per call)"
        del sets, calls
        torch.cuda.empty_cache()
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
        finish(name, layer, flops, sec, n_sets, set_bytes,
               {"path": mm.mmbwd_forward_path(layer.B, layer.T, layer.C, layer.OC, dt)})
        del sets, calls
        torch.cuda.empty_cache()
    # the LayerNorm backward (lnbwd_run): bound by HBM, reported in GB/s of
    # algorithmic bytes against the measured copy bandwidth
    hbm = float(peaks.get("hbm_gbs", 6800.0))
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
        out[name] = {"B": p.B, "T": p.T, "C": p.C, "V": p.V, "dtype": p.dtype, "us": round(sec * 1e6, 2),
                     "gb_per_s": round(gbs, 1), "frac_of_peak": round(gbs / hbm, 4),
                     "peak": f"HBM copy (measured) {hbm:.0f} GB/s", "bytes": set_bytes,
                     "tokens": f"Zipf(s=1.1) over 50257 ids, {distinct} distinct", "input_sets": n_sets,
                     "l2": "rotating sets > L2" if n_sets * set_bytes > L2_BYTES else "L2-resident"}
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
        out[name] = {"B": p.B, "T": p.T, "C": p.C, "V": p.V, "dtype": p.dtype, "us": round(sec * 1e6, 2),
                     "gb_per_s": round(gbs, 1), "frac_of_peak": round(gbs / hbm, 4),
                     "peak": f"HBM copy (measured) {hbm:.0f} GB/s", "bytes": set_bytes,
                     "prepare_us": round(sec_prep * 1e6, 2),
                     "timed": "encbwd_run_planned; encbwd_prepare (the sort of the token ids) timed apart",
                     "tokens": f"Zipf(s=1.1) over 50257 ids, {distinct} distinct", "input_sets": n_sets,
                     "l2": "rotating sets > L2" if n_sets * set_bytes > L2_BYTES else "L2-resident"}
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
             | {n for n, _, _ in LAYER_CONFIGS} | {n for n, _ in ENC_PLANNED_CONFIGS})
    if args.case not in names:
        raise SystemExit(f"unknown case {args.case}; one of {sorted(names)}")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    mm.load()
    stream = torch.cuda.Stream(device=dev)
    out = measure_other_configs(torch, mm, dev, stream, only={args.case}, batches=max(1, args.steps))
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
