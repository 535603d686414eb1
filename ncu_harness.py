"""ncu harness: per-kernel counters of the benchmarked configurations.

    python ncu_harness.py [CASE ...] [--raw-dir DIR] [--out-dir DIR] [--list]
    python ncu_harness.py [CASE ...] --from-raw     # summaries from saved CSVs

For each case (default: all of CASES) on one GPU:

1. runs the case's command once without ncu; it must exit 0, else the case
   is skipped (a program that faults is never profiled);
2. the launch list: every launch of the same command with
   `gpu__time_duration.sum` alone (one pass), summed per kernel: launches,
   total time, share (cold-cache and serialised, so the shares count, not
   the absolute times);
3. the counters of the case's kernels on a few launches after the warm-up
   ones: time, SM clock, tensor-pipe activity (of elapsed and of active
   cycles), DRAM bytes read and written, DRAM and L2 throughput, L2 hit
   rate, registers per thread -- a handful of passes, on the same small
   command;

and writes `profiles/<kernel>_<case>.md`: the commands, the hash of the
kernel's source files, `dram_bytes_per_launch` (the mean DRAM traffic of the
captured launches of the top kernel, which bench.py reports as the roofline
traffic while the hash matches), and the tables. Raw CSV goes to --raw-dir,
with the capture times; `--from-raw` writes the summaries from those files
alone (on a machine without the GPU, from the same sources).
Every ncu command runs with --clock-control none.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(ROOT, "linear_layer_gemms_gb300", "csrc")
PY = sys.executable

METRICS = [
    "gpu__time_duration.sum",
    "sm__cycles_elapsed.avg.per_second",
    "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed",
    "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active",
    "dram__bytes_read.sum",
    "dram__bytes_write.sum",
    "dram__throughput.avg.pct_of_peak_sustained_elapsed",
    "lts__throughput.avg.pct_of_peak_sustained_elapsed",
    "lts__t_sector_hit_rate.pct",
    "launch__registers_per_thread",
    "launch__grid_size",
]

TC_SOURCES = ("tc_gemm.cu", "ptx.cuh", "internal.h")


def _bench(*args):
    return [PY, os.path.join(ROOT, "bench.py"), *args]


def _case_bench(name, steps=1):
    return _bench("--case", name, "--steps", str(steps), "--no-verify")


# name: command, kernel regex for the counters, launches to skip and to
# capture, per-launch labels, algorithmic FLOPs and bytes of each captured
# launch (None where the launch is not the unit), the file's kernel name, the
# source files hashed, and a title.
def _mlp_units():
    # fc (C=768, OC=3072), fc_proj (C=3072, OC=768); B*T = 8192; bf16 with bias
    return [_bw_units(8192, C, OC, True, 2) for C, OC in ((768, 3072), (3072, 768))]


def _bw_units(bt, C, OC, bias, es):
    """FLOPs 4*BT*C*OC (+ BT*OC for the bias sum) and algorithmic bytes: dout,
    inp, weight read once, dinp and dweight read and written, dbias written."""
    flops = 4 * bt * C * OC + (bt * OC if bias else 0)
    byt = es * (bt * OC + 3 * bt * C + 3 * OC * C + (OC if bias else 0))
    return flops, byt


CASES = {
    "mlp": {
        "title": "GPT-2 small MLP backward (fc then fc_proj), bf16, B=8 T=1024, in the benchmark's step",
        "cmd": _bench("--steps", "3", "--warmup", "3", "--no-e2e", "--no-cpu-baseline", "--no-other"),
        "kernel": "tc_mmbwd_kernel", "skip": 6, "count": 2, "labels": ["fc", "fc_proj"],
        "units": _mlp_units(), "file": "tc_mmbwd_kernel_mlp", "sources": TC_SOURCES,
    },
    "attn_proj": {
        "title": "GPT-2 small attention-projection backward, bf16, B=8 T=1024 C=OC=768 (split dweight reduction)",
        "cmd": _case_bench("attn_proj"),
        "kernel": "tc_mmbwd_kernel|tc_splitk_fixup", "skip": 24, "count": 2,
        "labels": ["GEMM", "split fixup"],
        "units": [_bw_units(8192, 768, 768, True, 2), None],
        "file": "tc_mmbwd_kernel_attn_proj", "sources": TC_SOURCES,
    },
    "lm_head": {
        "title": "GPT-2 small LM-head backward, bf16, B=8 T=1024 C=768 OC=50304, no bias",
        "cmd": _case_bench("lm_head"),
        "kernel": "tc_mmbwd_kernel", "skip": 2, "count": 1, "labels": ["LM head"],
        "units": [_bw_units(8192, 768, 50304, False, 2)], "file": "tc_mmbwd_kernel_lm_head", "sources": TC_SOURCES,
    },
    "forward_mlp": {
        "title": "Forward of the GPT-2 small MLP layers (fc, then fc_proj), bf16, B=8 T=1024",
        "cmd": _case_bench("forward_mlp_fc"),
        "kernel": "tc_mmbwd_kernel", "skip": 8, "count": 2, "labels": ["forward fc", "forward fc"],
        "units": [(2 * 8192 * 768 * 3072 + 8192 * 3072, 2 * (8192 * 768 + 3072 * 768 + 8192 * 3072 + 3072))] * 2,
        "file": "tc_mmbwd_kernel_forward_mlp_fc", "sources": TC_SOURCES,
    },
    "xl_fc_f32": {
        "title": "GPT-2 XL fc backward in fp32 (three tf32 products), B=4 T=1024 C=1600 OC=6400",
        "cmd": _case_bench("xl_fc_f32"),
        "kernel": "tc_mmbwd_kernel", "skip": 4, "count": 2,
        "labels": ["both products", "next call"], "units": [_bw_units(4096, 1600, 6400, False, 4)] * 2,
        "file": "tc_mmbwd_kernel_x3_xl_fc_f32",
        "sources": TC_SOURCES + ("split_tf32.cu",),
    },
    "ln_xl": {
        "title": "LayerNorm backward, GPT-2 XL width, bf16, B=8 T=1024 C=1600",
        "cmd": _case_bench("ln_xl"),
        "kernel": "ln_bwd_rows|ln_bwd_params", "skip": 4, "count": 2, "labels": None, "units": None,
        "file": "layernorm_bwd_rows_kernel_ln_xl", "sources": ("layernorm_bwd.cu",),
    },
    "enc": {
        "title": "Encoder backward, GPT-2 small, bf16, B=8 T=1024 C=768, Zipf token ids",
        "cmd": _case_bench("enc_gpt2_small"),
        "kernel": "enc_window|enc_sort", "skip": 24, "count": 2, "labels": None, "units": None,
        "file": "enc_window_kernel_enc_gpt2_small", "sources": ("encoder_bwd.cu",),
    },
}


def strip_comments(text: str) -> str:
    """C/C++/CUDA source without its comments and with every run of white space
    as one space: what the compiler reads, so that a summary stays matched to
    its kernel across edits of comments or layout. String and character
    literals are copied as they are."""
    out = []
    i, n = 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def code_sha(paths) -> str:
    """First 12 hex digits of the SHA-1 of the files' code (strip_comments), in order."""
    h = hashlib.sha1()
    for path in paths:
        with open(path) as fh:
            h.update(strip_comments(fh.read()).encode())
        h.update(b"\0")
    return h.hexdigest()[:12]


def source_sha(files) -> str:
    return code_sha([os.path.join(CSRC, f) for f in files])


def _num(v: str) -> float | None:
    try:
        return float(v.replace(",", ""))
    except ValueError:
        return None


def parse_csv(text: str):
    """Launches in order: (id, kernel name, {metric: value}) from ncu --csv output."""
    start = text.find('"ID"')
    if start < 0:
        return []
    rows = csv.DictReader(io.StringIO(text[start:]))
    launches, order = {}, []
    for r in rows:
        i = r.get("ID")
        if i is None:
            continue
        if i not in launches:
            launches[i] = (r.get("Kernel Name", ""), {})
            order.append(i)
        launches[i][1][r.get("Metric Name", "")] = _num(r.get("Metric Value", ""))
    return [(i, launches[i][0], launches[i][1]) for i in order]


def short_name(k: str) -> str:
    for p in ("void ", "mmbwd::", "(anonymous namespace)::", "<unnamed>::"):
        k = k.replace(p, "")
    return k.split("(")[0].strip()


def run(cmd, log_path, timeout=None):
    """Run to completion (ncu commands get no timeout: a capture killed midway
    can leave the GPU hung, so every capture is sized to end by itself)."""
    t0 = time.time()
    with open(log_path, "w") as f:
        r = subprocess.run(cmd, stdout=f, stderr=subprocess.STDOUT, cwd=ROOT, timeout=timeout)
    return r.returncode, time.time() - t0


def ncu_cmd(extra, log_file, cmd):
    return ["ncu", "--clock-control", "none", "--print-units", "base", "--csv", "--log-file", log_file,
            *extra, *cmd]


def profile(name: str, raw_dir: str, out_dir: str, max_launches: int) -> str | None:
    spec = CASES[name]
    cmd = spec["cmd"]
    plain_log = os.path.join(raw_dir, f"{name}_plain.log")
    rc, _ = run(cmd, plain_log, 600)
    if rc != 0:
        print(f"[{name}] plain run exited {rc}; not profiled (see {plain_log})", flush=True)
        return None
    # 1. launch list (one pass)
    lfile = os.path.join(raw_dir, f"{name}_launches.csv")
    lcmd = ncu_cmd(["--metrics", "gpu__time_duration.sum", "-c", str(max_launches)], lfile, cmd)
    rc, dt_l = run(lcmd, os.path.join(raw_dir, f"{name}_launches.log"))
    if rc != 0:
        print(f"[{name}] launch list: ncu exited {rc}", flush=True)
        return None
    # 2. counters of the case's kernels
    mfile = os.path.join(raw_dir, f"{name}_metrics.csv")
    mcmd = ncu_cmd(["--metrics", ",".join(METRICS), "-k", f"regex:{spec['kernel']}", "-s", str(spec["skip"]),
                    "-c", str(spec["count"])], mfile, cmd)
    rc, dt_m = run(mcmd, os.path.join(raw_dir, f"{name}_metrics.log"))
    if rc != 0:
        print(f"[{name}] counters: ncu exited {rc}", flush=True)
        return None
    with open(os.path.join(raw_dir, f"{name}_times.json"), "w") as f:
        json.dump({"launch_list_s": dt_l, "counters_s": dt_m}, f)
    return summarize(name, raw_dir, out_dir, lcmd, mcmd)


def summarize(name: str, raw_dir: str, out_dir: str, lcmd=None, mcmd=None, max_launches: int = 400) -> str | None:
    """Summary of case `name` from the CSV files in raw_dir (written by profile)."""
    spec = CASES[name]
    cmd = spec["cmd"]
    lfile = os.path.join(raw_dir, f"{name}_launches.csv")
    mfile = os.path.join(raw_dir, f"{name}_metrics.csv")
    if not (os.path.exists(lfile) and os.path.exists(mfile)):
        print(f"[{name}] no raw files in {raw_dir}", flush=True)
        return None
    if lcmd is None:
        lcmd = ncu_cmd(["--metrics", "gpu__time_duration.sum", "-c", str(max_launches)], lfile, cmd)
    if mcmd is None:
        mcmd = ncu_cmd(["--metrics", ",".join(METRICS), "-k", f"regex:{spec['kernel']}", "-s", str(spec["skip"]),
                        "-c", str(spec["count"])], mfile, cmd)
    times = {}
    tpath = os.path.join(raw_dir, f"{name}_times.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            times = json.load(f)
    launches = parse_csv(open(lfile).read())
    per_kernel = {}
    for _, k, m in launches:
        s = per_kernel.setdefault(short_name(k), [0, 0.0])
        s[0] += 1
        s[1] += (m.get("gpu__time_duration.sum") or 0.0)
    total = sum(v[1] for v in per_kernel.values()) or 1.0
    caps = parse_csv(open(mfile).read())
    sha = source_sha(spec["sources"])
    return write_summary(name, spec, sha, lcmd, mcmd, per_kernel, total, caps, times.get("launch_list_s"),
                         times.get("counters_s"), out_dir)


def _took(dt) -> str:
    return "(capture time not recorded)" if dt is None else f"({dt:.0f} s)"


def _fmt(v, scale=1.0, nd=1, unit=""):
    return "n/a" if v is None else f"{v * scale:.{nd}f}{unit}"


def write_summary(name, spec, sha, lcmd, mcmd, per_kernel, total, caps, dt_l, dt_m, out_dir) -> str:
    rel = lambda c: " ".join(os.path.relpath(x, ROOT) if os.path.isabs(x) and x.startswith(ROOT) else  # noqa: E731
                             ("python" if x == PY else x) for x in c)
    top = [c for c in caps if spec["kernel"].split("|")[0] in c[1]]
    dram = [(m.get("dram__bytes_read.sum") or 0) + (m.get("dram__bytes_write.sum") or 0) for _, _, m in top]
    lines = [f"# {spec['file']} -- {spec['title']}", "",
             "Written by `ncu_harness.py` (the case's command ran once without ncu and exited 0 first).", "",
             f"- case: `{name}`",
             f"- kernel_source_sha: `{sha}`",
             f"- hashed sources (code only: comments and white space are not hashed): {', '.join(spec['sources'])}"]
    if dram:
        lines.append(f"- dram_bytes_per_launch: `{sum(dram) / len(dram):.0f}`")
    lines += ["", "## Launch list (`gpu__time_duration.sum` alone: one pass, cold-cache and serialised)", "",
              f"    {rel(lcmd)}", "", _took(dt_l), "",
              "| kernel | launches | total | share | mean |", "|---|---|---|---|---|"]
    for k, (n, t) in sorted(per_kernel.items(), key=lambda kv: -kv[1][1]):
        lines.append(f"| `{k}` | {n} | {t / 1e3:.1f} us | {100 * t / total:.1f} % | {t / n / 1e3:.2f} us |")
    lines += ["", "## Counters of the captured launches", "", f"    {rel(mcmd)}", "", _took(dt_m), ""]
    head = ["metric"]
    for i, (_, k, _) in enumerate(caps):
        lab = spec["labels"][i] if spec.get("labels") and i < len(spec["labels"]) else short_name(k)
        head.append(lab)
    lines.append("| " + " | ".join(head) + " |")
    lines.append("|" + "---|" * len(head))
    rows = [("gpu__time_duration.sum", 1e-3, 2, " us"), ("sm__cycles_elapsed.avg.per_second", 1e-9, 3, " GHz"),
            ("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed", 1, 1, " %"),
            ("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active", 1, 1, " %"),
            ("dram__bytes_read.sum", 1e-6, 2, " MB"), ("dram__bytes_write.sum", 1e-6, 2, " MB"),
            ("dram__throughput.avg.pct_of_peak_sustained_elapsed", 1, 1, " %"),
            ("lts__throughput.avg.pct_of_peak_sustained_elapsed", 1, 1, " %"),
            ("lts__t_sector_hit_rate.pct", 1, 1, " %"), ("launch__registers_per_thread", 1, 0, ""),
            ("launch__grid_size", 1, 0, "")]
    for metric, sc, nd, unit in rows:
        lines.append(f"| {metric} | " + " | ".join(_fmt(m.get(metric), sc, nd, unit) for _, _, m in caps) + " |")
    units = spec.get("units")
    if units:
        ach, alg, ratio = ["achieved (algorithmic FLOPs / time)"], ["algorithmic bytes"], ["DRAM bytes / algorithmic"]
        for i, (_, _, m) in enumerate(caps):
            u = units[i] if i < len(units) else None
            t = m.get("gpu__time_duration.sum")
            if u is None or not t:
                ach.append("")
                alg.append("")
                ratio.append("")
                continue
            d = (m.get("dram__bytes_read.sum") or 0) + (m.get("dram__bytes_write.sum") or 0)
            ach.append(f"{u[0] / (t * 1e-9) / 1e12:.0f} TFLOP/s")
            alg.append(f"{u[1] / 1e6:.1f} MB")
            ratio.append(f"{d / u[1]:.2f}")
        for r in (ach, alg, ratio):
            lines.append("| " + " | ".join(r) + " |")
    lines.append("")
    path = os.path.join(out_dir, spec["file"] + ".md")
    with open(path, "w") as f:
        f.write("\n".join(lines))
    print(f"[{name}] wrote {os.path.relpath(path, ROOT)}", flush=True)
    return path


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("cases", nargs="*")
    ap.add_argument("--raw-dir", default=os.path.join(ROOT, "ncu_raw"))
    ap.add_argument("--out-dir", default=os.path.join(ROOT, "profiles"))
    ap.add_argument("--max-launches", type=int, default=400)
    ap.add_argument("--list", action="store_true")
    ap.add_argument("--from-raw", action="store_true",
                    help="write the summaries from the CSV files already in --raw-dir (no GPU, no ncu)")
    a = ap.parse_args(argv)
    if a.list:
        for k, v in CASES.items():
            print(f"{k}: {v['title']}")
        return 0
    os.makedirs(a.raw_dir, exist_ok=True)
    os.makedirs(a.out_dir, exist_ok=True)
    names = a.cases or list(CASES)
    bad = [n for n in names if n not in CASES]
    if bad:
        raise SystemExit(f"unknown case(s) {bad}; one of {list(CASES)}")
    failed = 0
    for n in names:
        if a.from_raw:
            r = summarize(n, a.raw_dir, a.out_dir, max_launches=a.max_launches)
        else:
            r = profile(n, a.raw_dir, a.out_dir, a.max_launches)
        if r is None:
            failed += 1
    return 1 if failed else 0


if __name__ == "__main__":
    sys.exit(main())
