#!/usr/bin/env python3
"""Benchmark of the block-scaled linear layer on GB300.

One step = the whole hot path over one batch: for every linear layer of the workload, quantize
its activations A (M x K) and weights B (N x K) along K (one batched launch), then the
block-scaled GEMM with the fused bias + bf16 epilogue.
Default workload: the largest single-GPU configuration, the ViT-L/16 MLP at M = 51200 tokens
(32 frames of 640 x 640): fc1 (K = 1024, N = 4096) and fc2 (K = 4096, N = 1024, its A a bf16
GELU output) in MXFP4 and in NVFP4 (per-tensor scale from the tensor's amax), four layers per
step. Inputs are seeded synthetic data resident in HBM; the L2 cache is flushed (a 256 MB write)
between timed steps and every step is timed with CUDA events on the stream the kernels run on.
One step (the L2 flush, an event, every layer's quantize and GEMM back to back, an event) is
captured once into a CUDA graph with the events as graph nodes and replayed every timed step,
so host launch overhead cannot open gaps inside the timed interval and the library kernels
overlap each other's prologue and tail through programmatic dependent launch, as they do in a
layer sequence; the kernels are exactly those the direct library calls launch. The per-kernel
times behind `roofline`, `gemms` and `quantize` come from a second graph of the same step with
events around each layer's quantize and GEMM (an event between two kernels serialises them),
replayed after the timed loop.

Printed JSON line: value = TFLOP/s of the whole step (2 M N K per GEMM); `gemms` = one entry per
layer (GEMM time, TFLOP/s, fraction of the format's peak: the measured bf16 tensor peak times the
nominal FP8 (x2) or FP4 (x6) ratio, and of the 4.5 / 9 PF dense peaks the target is stated
against, and of the attainable roofline); `quantize` = the quantizer kernels' algorithmic GB/s
against the measured HBM copy bandwidth; `roofline` = the kernel class (GEMM or quantizer) with
the larger share of the step; `e2e` = the same metric through the C ABI with pinned host buffers
and the host<->device copies inside the timed region; `cpu_baseline` = the CPU oracle timed on a
bounded sample of the same workload, with its quantize-only GB/s on one thread and on all cores;
`other_configs` = the other configurations of the study (the tiny fp32 check, ViT-B/16 fc1,
the ViT-L/16 MXFP8 and NVFP4 sweeps) timed per layer in the same run, for reference only.

`e2e` goes through the Python API call by call (no graphs): per step the pinned host inputs
are copied in, quantized, multiplied and the bf16 result is copied back; consecutive steps
overlap on three streams (copy in / compute / copy out) with double-buffered device memory.

--impl reference times the CPU oracle (the reference implementation of this path) alone.
With --gpus N (N > 1, launched by torchrun) every rank runs an independent replica of the
workload on its own GPU: the path shards by rows with no exchange (weak scaling).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import (MXFP8, NVFP4, MXFP4, WORKLOADS, make_activations, make_bias,  # noqa: E402
                       make_layernorm_affine, make_output_grad, make_weights)

METRIC = "block-scaled GEMM TFLOPS (% dense FP8/FP4 peak); quantize GB/s (% HBM)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_RATIO = {MXFP8: 4.5 / 2.25, NVFP4: 13.5 / 2.25, MXFP4: 13.5 / 2.25}
# the dense peaks the target of the study is stated against (TFLOP/s)
STATED_PEAK = {MXFP8: 4500.0, NVFP4: 9000.0, MXFP4: 9000.0}
HEADLINE = "vitl_mlp_large"
OTHER_CONFIGS = ("tiny_mxfp8", "vitb_fc1_mxfp8", "vitl_mxfp8", "vitl_nvfp4")
L2_FLUSH_BYTES = 256 << 20
FMT_NAME = {MXFP8: "mxfp8", NVFP4: "nvfp4", MXFP4: "mxfp4"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def quant_bytes(fmt: str, rows: int, cols: int, src_bytes: int, computed_global: bool) -> int:
    """Algorithmic HBM bytes of one quantizer call: read the source once (twice for NVFP4
    with a computed per-tensor scale: the amax pass), write codes and scales."""
    n = rows * cols
    codes = n if fmt == MXFP8 else n // 2
    scales = n // (16 if fmt == NVFP4 else 32)
    reads = n * src_bytes * (2 if (fmt == NVFP4 and computed_global) else 1)
    return reads + codes + scales


def dual_bytes(fmt: str, rows: int, cols: int, src_bytes: int, computed_global: bool = False) -> int:
    """Algorithmic bytes of one dual-layout quantization: the source read once (twice for an
    NVFP4 scale computed from the tensor's amax), codes and scales of both layouts written."""
    n = rows * cols
    reads = 2 if (fmt == NVFP4 and computed_global) else 1
    return reads * n * src_bytes + 2 * (n if fmt == MXFP8 else n // 2) + 2 * (n // (16 if fmt == NVFP4 else 32))


def gemm_bytes(fmt: str, M: int, N: int, K: int, bias: bool) -> int:
    """Algorithmic HBM bytes of one GEMM: codes and scales of A and B once, bf16 out, bias."""
    cb = 1 if fmt == MXFP8 else 0.5
    sb = 1 / (16 if fmt == NVFP4 else 32)
    return int((M + N) * K * (cb + sb) + 2 * M * N + (2 * N if bias else 0))


# ----------------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 100 ms while the timed loop runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str, out_path: str):
        self.out_path = out_path
        self.proc = None
        try:
            self.f = open(out_path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", gpu_index], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.out_path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------------- oracle timing
def _sample_rows(g, rows: int) -> int:
    """Rows of A the oracle sample takes: for a transposed convolution whole image rows of the
    first frame (a sub-image: kernel = stride = 2 has no halo)."""
    if g.convt is not None:
        return max(g.convt[2], min(rows, g.convt[1] * g.convt[2]) // g.convt[2] * g.convt[2])
    return rows


def _oracle_linear_rows(g, rows: int) -> float:
    import oracle

    rows = _sample_rows(g, rows)
    a = make_activations(g, rows=rows) if g.a_dist != "normal_outlier50" else make_activations(g)
    b = make_weights(g)
    bias = make_bias(g)
    t0 = time.perf_counter()
    qa = oracle.quantize(g.fmt, a)
    qb = oracle.quantize(g.fmt, b)
    alpha = qa.g * qb.g if qa.fmt == oracle.NVFP4 else 1.0
    if g.convt is not None:
        oracle.convt2x2(qa.decode(), qb.decode(), bias, 1, rows // g.convt[2], g.convt[2], alpha, gelu=True)
    else:
        oracle.gemm(qa.decode(), qb.decode(), bias, alpha, want_abs=False)
    return time.perf_counter() - t0


def _oracle_train_rows(g, rows: int, sr: bool) -> float:
    """One training step of the layer on the first `rows` tokens: dual quantization of X, W and
    dY, then forward, dgrad and wgrad (the latter summing over the `rows` tokens only)."""
    import oracle

    x, w, dy, bias = make_activations(g, rows=rows), make_weights(g), make_output_grad(g, rows=rows), make_bias(g)
    t0 = time.perf_counter()
    xr, xc = oracle.quantize_dual(g.fmt, x)
    wr, wc = oracle.quantize_dual(g.fmt, w)
    dr, dc = oracle.quantize_dual(g.fmt, dy, stochastic=sr, seed=1)
    nv = g.fmt == NVFP4  # alpha = g_A g_B
    oracle.gemm(xr.decode(), wr.decode(), bias, xr.g * wr.g if nv else 1.0, want_abs=False)
    oracle.gemm(dr.decode(), wc.decode(), None, dr.g * wc.g if nv else 1.0, want_abs=False)
    oracle.gemm(dc.decode(), xc.decode(), None, dc.g * xc.g if nv else 1.0, want_abs=False)
    return time.perf_counter() - t0


def cpu_oracle_train_sample(wl, target_s: float = 10.0):
    """The training step's oracle on R leading tokens (R a multiple of 32), R calibrated from two
    runs to take about `target_s` seconds. Returns (TFLOP/s, seconds, cores, description)."""
    import oracle

    g = wl.gemms[0]
    t32, t160 = _oracle_train_rows(g, 32, wl.grad_sr), _oracle_train_rows(g, 160, wl.grad_sr)
    per_row = max((t160 - t32) / 128.0, 1e-9)
    fixed = max(t32 - 32 * per_row, 0.0)
    rows = int(min(g.M, max(32, (target_s - fixed) / per_row))) // 32 * 32
    secs = _oracle_train_rows(g, rows, wl.grad_sr)
    desc = ("oracle training step on %d of %d tokens: dual quantization of X (R rows), W and dY (R rows), "
            "decode, fp64 forward, dgrad and wgrad GEMMs" % (rows, g.M))
    return 3 * 2 * rows * g.N * g.K / secs / 1e12, secs, oracle.num_threads(), desc


def oracle_sample(wl, target_s: float):
    return cpu_oracle_train_sample(wl, target_s) if wl.chain == "train" else cpu_oracle_sample(wl.gemms, target_s)


def cpu_oracle_sample(gemms, target_s: float = 10.0):
    """Time the CPU oracle (as it stands, all host cores) on a bounded sample of the workload:
    for each GEMM, quantize R rows of A and all of B, decode, fp64 GEMM of those R rows, with R
    chosen from two calibration runs so that the sample takes about `target_s` seconds (at
    most the whole of A). Returns (TFLOP/s, seconds, cores, description)."""
    import oracle

    flops, secs, parts = 0, 0.0, []
    for g in gemms:
        rows = g.M
        if g.a_dist != "normal_outlier50":
            # t(R) = fixed (all of B) + R * per_row
            r1, r2 = _sample_rows(g, 32), _sample_rows(g, 160)
            if r2 == r1:
                r2 = _sample_rows(g, 2 * r1)
            t1, t2 = _oracle_linear_rows(g, r1), _oracle_linear_rows(g, r2)
            per_row = max((t2 - t1) / max(r2 - r1, 1), 1e-9)
            fixed = max(t1 - r1 * per_row, 0.0)
            rows = int(min(g.M, max(32, (target_s / len(gemms) - fixed) / per_row)))
        rows = _sample_rows(g, rows)
        secs += _oracle_linear_rows(g, rows)
        flops += 2 * rows * g.N * g.K
        parts.append("%s: %d of %d rows" % (g.name, rows, g.M))
    desc = ("oracle quantize (R rows of A, all of B) + decode + fp64 GEMM of R rows (transposed convolutions: "
            "the sub-image of those rows, by definition); " + ", ".join(parts))
    return flops / secs / 1e12, secs, oracle.num_threads(), desc


def cpu_quantize_sample(wl, target_s: float = 3.0):
    """The oracle's quantizer alone (as it stands) on the largest activation matrix of each format
    of the workload: R leading rows, R calibrated to about `target_s` seconds, timed once with one
    thread and once with all host cores. GB/s on the algorithmic bytes the GPU quantizer is
    measured on (source read once, twice for an NVFP4 scale computed from the tensor's amax;
    codes and scales written). Returns a dict for cpu_baseline."""
    import oracle

    by_fmt = {}
    for g in wl.gemms:
        if g.fmt not in by_fmt or g.M * g.K > by_fmt[g.fmt].M * by_fmt[g.fmt].K:
            by_fmt[g.fmt] = g
    cores = oracle.num_threads()
    out = {"unit": "GB/s", "cores": cores}
    try:
        for nthreads, key in ((1, "one_thread"), (cores, "all_cores")):
            oracle.set_num_threads(nthreads)
            nbytes, secs, parts = 0, 0.0, []
            for fmt, g in sorted(by_fmt.items()):
                eb = 4 if g.src_f32 else 2
                full = g.a_dist == "normal_outlier50"  # the tiny case is drawn whole
                r0 = g.M if full else min(g.M, 64)
                x = make_activations(g) if full else make_activations(g, rows=r0)
                t0 = time.perf_counter()
                oracle.quantize(fmt, x)
                t = max(time.perf_counter() - t0, 1e-6)
                rows = r0 if full else int(min(g.M, max(r0, r0 * target_s / len(by_fmt) / t)))
                if rows != r0:
                    x = make_activations(g, rows=rows)
                    t0 = time.perf_counter()
                    oracle.quantize(fmt, x)
                    t = time.perf_counter() - t0
                nbytes += quant_bytes(fmt, rows, g.K, eb, True)
                secs += t
                parts.append("%s %d of %d rows x %d" % (fmt, rows, g.M, g.K))
            out[key] = nbytes / secs / 1e9
            out[key + "_sample"] = ", ".join(parts)
    finally:
        oracle.set_num_threads(cores)
    return out


def config_of(wl):
    return {"workload": wl.name, "description": wl.description,
            "gemms": [{"name": g.name, "format": g.fmt, "M": g.M, "N": g.N, "K": g.K} for g in wl.gemms],
            "chain": wl.chain,
            "grad_rounding": ("stochastic (Philox4x32-10)" if wl.grad_sr else "nearest even") if wl.chain == "train" else None,
            "grad_scale": ("delayed: previous step's amax x %g / 2688" % wl.grad_headroom) if wl.grad_headroom else None,
            "l2": "flushed between timed steps (256 MB write)",
            "launch": "one step (L2 flush, then every layer's quantize and GEMM back to back) captured once "
                      "into a CUDA graph with CUDA events as graph nodes at the step's ends, replayed every timed "
                      "step (value, ms_per_step); per-kernel times (roofline, quantize) from a second graph of "
                      "the same step with events around each kernel, replayed after the timed loop"}


# ----------------------------------------------------------------------------------- reference arm
def run_reference(args, rank: int, world: int):
    """The CPU oracle, as it stands, on the host cores (rank 0 only)."""
    if rank != 0:
        return 0
    wl = WORKLOADS[args.workload]
    import oracle

    oracle.build()
    oracle_sample(wl, target_s=0.5)  # warm-up: page in the inputs and the library
    vals, secs_total = [], 0.0
    steps = max(1, min(args.steps, 3))
    cores, desc = None, ""
    for _ in range(steps):
        v, secs, cores, desc = oracle_sample(wl, target_s=args.cpu_seconds)
        vals.append(v)
        secs_total += secs
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": secs_total / steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": config_of(wl),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------------- replicas
def replica_throughput(ms_local: float, flops_per_rank: int, world: int, device=None):
    """Whole-job throughput of N independent replicas: every rank processed the same work,
    the job took the slowest rank's time. Returns (max ms over ranks, TFLOP/s of all ranks)."""
    ms = ms_local
    if world > 1:
        import torch
        import torch.distributed as dist

        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * flops_per_rank / (ms * 1e-3) / 1e12


# ----------------------------------------------------------------------------------- GPU arm
def _code_only(text: str) -> str:
    """C / C++ / CUDA source without its comments and with runs of whitespace collapsed (string
    literals kept as they are): what the compiler sees, so that editing a comment does not count
    as a kernel change."""
    import re

    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':  # string literal
            j = i + 1
            while j < n and text[j] != '"':
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
    return re.sub(r"\s+", " ", "".join(out)).strip()


def kernel_source_hash() -> str:
    """Hash of the code (comments and whitespace aside) of every kernel source of the library
    (csrc/*.cu, *.cuh, *.h) and of the public header: the key of the recorded DRAM traffic, so
    that any kernel change invalidates the record."""
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "block_scaled_precision_bsq_gb300", "csrc")
    paths = sorted(os.path.join(pkg, n) for n in os.listdir(pkg) if n.endswith((".cu", ".cuh", ".h")))
    for path in paths + [os.path.join(ROOT, "include", "bsq.h")]:
        with open(path, encoding="utf-8") as f:
            h.update(os.path.basename(path).encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")


def kernel_class(name: str):
    """The bench's kernel class of a launch in an ncu launch list: "gemm" for the GEMM kernels,
    "quantize" for the library's other kernels, None for anything else (the L2 flush, copies)."""
    if "bsq::" not in name:
        return None
    return "gemm" if ("gemm" in name or "splitk" in name) else "quantize"


def recorded_traffic(kernel_hash: str, workload: str, cls: str, path: str = TRAFFIC_PATH):
    """DRAM bytes (read + write) per step of kernel class `cls`, from the ncu record
    `profiles/traffic.json` (written by --record-traffic), if that capture was taken on the
    current kernel sources; else None."""
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_source_hash") != kernel_hash:
        return None
    return e.get("classes", {}).get(cls, {}).get("dram_bytes_per_step")


def traffic_capture(args):
    """--traffic-capture SIDECAR: the workload's step `--warmup` times through the direct library
    calls, each after an L2 flush, nothing else on the device; for an ncu launch list with DRAM
    counters (`ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum
    --csv`). Writes SIDECAR: the workload, the number of steps run and the kernel source hash,
    which --record-traffic needs to turn the launch list into bytes per step."""
    import torch

    import __graft_entry__ as ge

    ge.build()
    import block_scaled_precision_bsq_gb300 as bsq

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = WORKLOADS[args.workload]
    layers = args.layers.split(",") if args.layers else None
    units = build_units(wl, bsq, dev, layers)
    assert units, "no layer of %s is named %s" % (wl.name, args.layers)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        flush.zero_()
        for U in units:
            U["quant"](U["D"], s)
            U["gemm"](U["D"], s)
        torch.cuda.synchronize()
    assert bsq.device_status() == 0
    with open(args.traffic_capture, "w") as f:
        json.dump({"workload": wl.name + ("[%s]" % args.layers if args.layers else ""), "steps": args.warmup,
                   "kernel_source_hash": kernel_source_hash(),
                   "launches_per_step": sum(U["launches"] for U in units)}, f)
    return 0


def record_traffic(csv_path: str, sidecar_path: str, command: str, out_path: str = TRAFFIC_PATH):
    """--record-traffic CSV SIDECAR: per kernel class, the DRAM bytes per step of a
    --traffic-capture run's ncu launch list, into profiles/traffic.json under the workload."""
    import csv
    import re

    with open(sidecar_path) as f:
        side = json.load(f)
    with open(csv_path, newline="") as f:
        rows = [r for r in csv.reader(f)]
    head = next(i for i, r in enumerate(rows) if "Kernel Name" in r and "Metric Name" in r)
    h = rows[head]
    col = {k: h.index(k) for k in ("ID", "Kernel Name", "Metric Name", "Metric Unit", "Metric Value")}
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "ns": 1e-3, "nsecond": 1e-3, "us": 1.0,
             "usecond": 1.0, "ms": 1e3, "msecond": 1e3}
    launches = {}
    for r in rows[head + 1:]:
        if len(r) < len(h):
            continue
        e = launches.setdefault(r[col["ID"]], {"name": r[col["Kernel Name"]]})
        e[r[col["Metric Name"]]] = float(r[col["Metric Value"]].replace(",", "")) * scale[r[col["Metric Unit"]]]
    steps = side["steps"]
    ours = [e for e in launches.values() if kernel_class(e["name"]) is not None]
    if len(ours) != steps * side["launches_per_step"]:
        raise SystemExit("launch list holds %d library launches, expected %d steps x %d" % (
            len(ours), steps, side["launches_per_step"]))
    classes, kernels = {}, {}
    for e in ours:
        b = e["dram__bytes_read.sum"] + e["dram__bytes_write.sum"]
        for d, key in ((classes, kernel_class(e["name"])), (kernels, re.sub(r"\(.*", "", e["name"]).replace(
                "void ", "").replace("bsq::<unnamed>::", ""))):
            a = d.setdefault(key, {"launches": 0, "dram_read": 0.0, "dram_write": 0.0, "us": 0.0})
            a["launches"] += 1
            a["dram_read"] += e["dram__bytes_read.sum"]
            a["dram_write"] += e["dram__bytes_write.sum"]
            a["us"] += e["gpu__time_duration.sum"]
    def per_step(a):
        return {"launches_per_step": a["launches"] / steps,
                "dram_bytes_per_step": int(round((a["dram_read"] + a["dram_write"]) / steps)),
                "dram_read_per_step": int(round(a["dram_read"] / steps)),
                "dram_write_per_step": int(round(a["dram_write"] / steps)),
                "ncu_us_per_step": a["us"] / steps}
    d = {}
    if os.path.exists(out_path):
        with open(out_path) as f:
            d = json.load(f)
    d[side["workload"]] = {
        "kernel_source_hash": side["kernel_source_hash"], "steps_captured": steps, "command": command,
        "note": "ncu launch list (one pass, --clock-control none): cold-cache, serialised launches; the "
                "first launch of each step follows a 256 MB L2 flush whose dirty lines it writes back",
        "classes": {k: per_step(v) for k, v in sorted(classes.items())},
        "kernels": {k: per_step(v) for k, v in sorted(kernels.items())}}
    with open(out_path, "w") as f:
        json.dump(d, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps(d[side["workload"]]["classes"]))
    return 0


def _host(x):
    """A numpy input (uint16 = bf16 bits, or fp32) as a pinned host tensor."""
    import torch

    t = torch.from_numpy(x.view(np.int16) if x.dtype == np.uint16 else x)
    return (t.view(torch.bfloat16) if x.dtype == np.uint16 else t).pin_memory()


def build_units(wl, bsq, dev, layers=None):
    """The step of workload `wl` as units: one per linear layer (or one per chained MLP /
    training step). A unit holds its pinned host inputs, an `alloc` making one device buffer set
    (e2e double-buffers them), its quantize and GEMM phases, and its flops / algorithmic bytes.
    `layers`: the names of the layers to keep (unchained workloads; for profiling one layer)."""
    import torch

    units = []
    if wl.chain is None:
        for g in wl.gemms:
            if layers and g.name not in layers:
                continue
            bias = make_bias(g)
            hosts = {"a": _host(make_activations(g)), "b": _host(make_weights(g)),
                     "bias": _host(bias) if bias is not None else None}

            def alloc(g=g, hosts=hosts):
                return {"a": torch.empty_like(hosts["a"], device=dev), "b": torch.empty_like(hosts["b"], device=dev),
                        "bias": torch.empty_like(hosts["bias"], device=dev) if hosts["bias"] is not None else None,
                        "qa": bsq.empty_qtensor(g.fmt, g.M, g.K, dev), "qb": bsq.empty_qtensor(g.fmt, g.N, g.K, dev),
                        "out": torch.empty((g.M, g.N) if g.convt is None else
                                           (g.convt[0], 2 * g.convt[1], 2 * g.convt[2], g.N // 4),
                                           dtype=torch.bfloat16, device=dev)}

            def quant(D, s, g=g):
                # activations and weights of the layer in one launch (bsq_quantize_batch)
                bsq.quantize_many(g.fmt, [D["a"], D["b"]], outs=[D["qa"], D["qb"]], stream=s)

            def gemm(D, s, g=g):
                if g.convt is not None:  # head transposed convolution, GELU fused (the ScaleBlock)
                    b_, h_, w_ = g.convt
                    bsq.convt2x2(D["qa"], D["qb"], b_, h_, w_, bias=D["bias"], gelu=True, out=D["out"], stream=s)
                else:
                    bsq.gemm(D["qa"], D["qb"], D["bias"], out=D["out"], stream=s)

            units.append({"name": g.name, "gemms": [g], "hosts": hosts, "alloc": alloc, "quant": quant, "gemm": gemm,
                          # the batched quantize, the GEMM; NVFP4: one amax pass for both matrices
                          "fmt": g.fmt, "flops": g.flops, "launches": 2 + (1 if g.fmt == NVFP4 else 0),
                          "qkernels": ["stream_kernel"] + (["amax_kernel"] if g.fmt == NVFP4 else []),
                          "qbytes": quant_bytes(g.fmt, g.M, g.K, 4 if g.src_f32 else 2, True) +
                                    quant_bytes(g.fmt, g.N, g.K, 4 if g.src_f32 else 2, True),
                          "gbytes": gemm_bytes(g.fmt, g.M, g.N, g.K, bias is not None)})
    elif wl.chain == "train":
        g = wl.gemms[0]
        fmt, M, K, N = g.fmt, g.M, g.K, g.N
        delayed = fmt == NVFP4 and wl.grad_headroom is not None
        # dW = dY^T X: N x K over the M tokens, K cut into the library's number of ranges
        dw_splits = bsq.bsq_gemm_splitk_splits(fmt, N, K, M)
        assert dw_splits >= 1
        hosts = {"x": _host(make_activations(g)), "w": _host(make_weights(g)), "bias": _host(make_bias(g)),
                 "dy": _host(make_output_grad(g))}

        def alloc():
            D = {k: torch.empty_like(v, device=dev) for k, v in hosts.items()}
            D.update({"qx": (bsq.empty_qtensor(fmt, M, K, dev), bsq.empty_qtensor(fmt, K, M, dev)),
                      "qw": (bsq.empty_qtensor(fmt, N, K, dev), bsq.empty_qtensor(fmt, K, N, dev)),
                      "qdy": (bsq.empty_qtensor(fmt, M, N, dev), bsq.empty_qtensor(fmt, N, M, dev)),
                      "out": torch.empty((M, N), dtype=torch.bfloat16, device=dev),
                      "dx": torch.empty((M, K), dtype=torch.bfloat16, device=dev),
                      "dw": torch.empty((N, K), dtype=torch.bfloat16, device=dev),
                      "ws": torch.empty(dw_splits * N * K if dw_splits > 1 else 4, dtype=torch.float32, device=dev)})
            if delayed:
                # the step before the first one: dY quantized with its own amax, so that the
                # first timed step finds a recorded amax in the tail
                D["g_dy"] = torch.empty(1, dtype=torch.float32, device=dev)
                D["dy"].copy_(hosts["dy"])
                bsq.quantize_dual(fmt, D["dy"], out=D["qdy"])
            return D

        def quant(D, s):
            # both layouts of X, W and dY, each in one pass over its source
            bsq.quantize_dual(fmt, D["x"], out=D["qx"], stream=s)
            bsq.quantize_dual(fmt, D["w"], out=D["qw"], stream=s)
            g_dy = None
            if delayed:  # this step's scale from the amax the previous step recorded
                g_dy = bsq.delayed_global_scale(D["qdy"][0], wl.grad_headroom, out=D["g_dy"], stream=s)
            bsq.quantize_dual(fmt, D["dy"], stochastic=wl.grad_sr, seed=1, global_scale=g_dy, out=D["qdy"], stream=s)

        def gemm(D, s):
            bsq.gemm(D["qx"][0], D["qw"][0], D["bias"], out=D["out"], stream=s)  # Y = X W^T + b
            bsq.gemm(D["qdy"][0], D["qw"][1], None, out=D["dx"], stream=s)       # dX = dY W
            bsq.gemm_splitk(D["qdy"][1], D["qx"][1], None, splits=dw_splits, workspace=D["ws"], out=D["dw"],
                            stream=s)                                            # dW = dY^T X

        nv = fmt == NVFP4
        units.append({"name": "train_step", "gemms": [g, g, g], "hosts": hosts, "alloc": alloc, "quant": quant,
                      "gemm": gemm, "fmt": fmt, "flops": 3 * g.flops, "outs": ("out", "dx", "dw"),
                      "qkernels": ["dual_kernel"] + (["amax_kernel"] if nv else []) +
                                  (["delayed_scale_kernel"] if delayed else []),
                      # duals + GEMMs (+ the split-K sum); NVFP4: amax passes of X and W, the delayed-scale kernel
                      "launches": 6 + (1 if dw_splits > 1 else 0) + (2 if nv else 0) + (1 if delayed else 0) +
                                  (1 if nv and not delayed else 0),
                      "qbytes": dual_bytes(fmt, M, K, 2, True) + dual_bytes(fmt, N, K, 2, True) +
                                dual_bytes(fmt, M, N, 2, not delayed),
                      "gbytes": gemm_bytes(fmt, M, N, K, True) + gemm_bytes(fmt, M, K, N, False) +
                                gemm_bytes(fmt, N, K, M, False)})
    else:
        g1, g2 = wl.gemms  # fc1: M x K1 -> N1, fc2: M x N1 -> N2
        fmt = g1.fmt
        b1, b2 = make_bias(g1), make_bias(g2)
        hosts = {"x": _host(make_activations(g1)), "w1": _host(make_weights(g1)), "w2": _host(make_weights(g2)),
                 "b1": _host(b1), "b2": _host(b2)}
        fused = wl.chain in ("fused", "ln_fused")
        ln = wl.chain == "ln_fused"
        if ln:
            lg, lb = make_layernorm_affine(g1.K, g1.seed)
            hosts.update({"ln_g": _host(lg), "ln_b": _host(lb)})

        def alloc():
            D = {k: torch.empty_like(v, device=dev) for k, v in hosts.items()}
            D.update({"qx": bsq.empty_qtensor(fmt, g1.M, g1.K, dev), "qw1": bsq.empty_qtensor(fmt, g1.N, g1.K, dev),
                      "qw2": bsq.empty_qtensor(fmt, g2.N, g2.K, dev), "qh": bsq.empty_qtensor(fmt, g2.M, g2.K, dev),
                      "out": torch.empty((g2.M, g2.N), dtype=torch.bfloat16, device=dev)})
            if not fused:
                D["h"] = torch.empty((g1.M, g1.N), dtype=torch.bfloat16, device=dev)
            return D

        def quant(D, s):
            if ln:  # LayerNorm + quantize of the activations in one kernel, the weights batched
                bsq.layernorm_quantize(fmt, D["x"], D["ln_g"], D["ln_b"], 1e-6, out=D["qx"], stream=s)
                bsq.quantize_many(fmt, [D["w1"], D["w2"]], outs=[D["qw1"], D["qw2"]], stream=s)
            else:
                bsq.quantize_many(fmt, [D["x"], D["w1"], D["w2"]], outs=[D["qx"], D["qw1"], D["qw2"]], stream=s)

        def gemm(D, s):
            if fused:  # fc1's epilogue writes fc2's operand
                bsq.gemm_gelu_quantize(D["qx"], D["qw1"], D["b1"], out_fmt=fmt, out=D["qh"], stream=s)
            else:      # fc1 + GELU to bf16, then a quantize pass
                bsq.gemm_gelu(D["qx"], D["qw1"], D["b1"], out=D["h"], stream=s)
                bsq.quantize(fmt, D["h"], out=D["qh"], stream=s)
            bsq.gemm(D["qh"], D["qw2"], D["b2"], out=D["out"], stream=s)

        units.append({"name": "mlp", "gemms": [g1, g2], "hosts": hosts, "alloc": alloc, "quant": quant, "gemm": gemm,
                      "fmt": fmt, "flops": g1.flops + g2.flops, "launches": (4 if ln else 3) if fused else 4,
                      "qkernels": (["layernorm_kernel"] if ln else []) + ["stream_kernel"] +
                                  (["amax_kernel"] if fmt == NVFP4 else []),
                      "qbytes": sum(quant_bytes(fmt, r, c, 2, True) for r, c in ((g1.M, g1.K), (g1.N, g1.K), (g2.N, g2.K))),
                      "gbytes": gemm_bytes(fmt, g1.M, g1.N, g1.K, True) + gemm_bytes(fmt, g2.M, g2.N, g2.K, True) -
                                (2 * g1.M * g1.N if fused else 0) +
                                (g1.M * g1.N * (1 if fmt == MXFP8 else 0.5) if fused else 0)})
    for U in units:
        U["D"] = U["alloc"]()
        for k, v in U["hosts"].items():
            if v is not None:
                U["D"][k].copy_(v)
    return units


class StepGraphs:
    """Two CUDA graphs of one step, events recorded by graph nodes:
     - the step graph (timed loop, `value`): flush, event, every unit's quantize and GEMM back
       to back, event. Consecutive library kernels overlap their prologue with the previous
       kernel's tail (programmatic dependent launch), as in a real layer sequence;
     - the split graph (per-kernel times): flush, then per unit event / quantize / event / GEMM /
       event. An event between two kernels serialises them and blocks the overlap, so this graph
       is replayed after the timed loop, not in it."""

    def __init__(self, units, flush, dev):
        import torch

        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(torch.cuda.current_stream())
        self.step_evs = tuple(torch.cuda.Event(enable_timing=True, external=True) for _ in range(2))
        self.step_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.step_graph, stream=cap):
            flush.zero_()
            self.step_evs[0].record(cap)
            for U in units:
                U["quant"](U["D"], cap)
                U["gemm"](U["D"], cap)
            self.step_evs[1].record(cap)
        self.evs = [tuple(torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)) for _ in units]
        self.split_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.split_graph, stream=cap):
            flush.zero_()
            for U, e in zip(units, self.evs):
                e[0].record(cap)
                U["quant"](U["D"], cap)
                e[1].record(cap)
                U["gemm"](U["D"], cap)
                e[2].record(cap)
        torch.cuda.synchronize()

    def step(self):
        """One replay of the step graph; returns its ms."""
        self.step_graph.replay()
        self.step_evs[1].synchronize()
        return self.step_evs[0].elapsed_time(self.step_evs[1])

    def split_step(self):
        """One replay of the split graph; returns per unit (quantize ms, GEMM ms)."""
        self.split_graph.replay()
        self.evs[-1][2].synchronize()
        return [(e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])) for e in self.evs]


def per_unit_entries(units, split, peaks, peak_src):
    """One entry per unit from the split-graph samples: the GEMM phase's time, TFLOP/s and
    fractions of peak (measured bf16 x nominal format ratio, the stated dense peak, the
    attainable roofline max(flops / peak, bytes / HBM)) and the quantize phase's GB/s."""
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    bf16 = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    out = []
    for i, U in enumerate(units):
        g_ms = float(np.mean([t[i][1] for t in split]))
        q_ms = float(np.mean([t[i][0] for t in split]))
        peak = bf16 * NOMINAL_RATIO[U["fmt"]]
        tflops = U["flops"] / (g_ms * 1e-3) / 1e12
        t_ideal = max(U["flops"] / (peak * 1e12), U["gbytes"] / (hbm * 1e9))
        out.append({"name": U["name"], "format": FMT_NAME[U["fmt"]],
                    "shape": [{"M": g.M, "N": g.N, "K": g.K} for g in U["gemms"]],
                    "gemm_ms": g_ms, "tflops": tflops, "peak": peak, "frac": tflops / peak,
                    "frac_stated": tflops / STATED_PEAK[U["fmt"]], "attainable_frac": t_ideal / (g_ms * 1e-3),
                    "quantize_ms": q_ms, "quantize_gbs": U["qbytes"] / (q_ms * 1e-3) / 1e9,
                    "quantize_frac": U["qbytes"] / (q_ms * 1e-3) / 1e9 / hbm})
    return out


def time_other_config(name, bsq, dev, flush, peaks, peak_src, reps):
    """A configuration other than the headline: its step's split graph, per-unit entries."""
    import torch

    wl = WORKLOADS[name]
    units = build_units(wl, bsq, dev)
    for _ in range(3):
        for U in units:
            U["quant"](U["D"], torch.cuda.current_stream())
            U["gemm"](U["D"], torch.cuda.current_stream())
    torch.cuda.synchronize()
    graphs = StepGraphs(units, flush, dev)
    for _ in range(3):
        graphs.split_step()
    split = [graphs.split_step() for _ in range(reps)]
    steps = [graphs.step() for _ in range(reps)]
    assert bsq.device_status() == 0
    flops = sum(U["flops"] for U in units)
    ms = float(np.mean(steps))
    entry = {"workload": name, "description": wl.description, "ms_per_step": ms,
             "tflops": flops / (ms * 1e-3) / 1e12, "gemms": per_unit_entries(units, split, peaks, peak_src)}
    del graphs, units
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def run_gpu(args, rank: int, world: int):
    import torch

    import __graft_entry__ as ge

    ge.build()
    import block_scaled_precision_bsq_gb300 as bsq

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    wl = WORKLOADS[args.workload]
    peaks, peak_src = load_peaks()
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    peak_bf16 = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])

    # inputs resident in HBM
    units = build_units(wl, bsq, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    # warm-up through the direct calls (first calls set kernel attributes, build tables)
    for _ in range(args.warmup):
        for U in units:
            U["quant"](U["D"], stream)
            U["gemm"](U["D"], stream)
    torch.cuda.synchronize()
    assert bsq.device_status() == 0

    graphs = StepGraphs(units, flush, dev)
    # our kernels per step (the batched quantize counts once; NVFP4 adds one amax pass per
    # batch; a chained MLP's unfused variant adds its quantize pass)
    launches_per_step = sum(U["launches"] for U in units)

    for _ in range(args.warmup):
        graphs.step()
        graphs.split_step()
    torch.cuda.synchronize()
    assert bsq.device_status() == 0

    # ------------------------------------------------------------ timed region
    if "CUDA_VISIBLE_DEVICES" in os.environ:
        gpu_index = os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]
    else:
        gpu_index = str(local)
    # the nvidia-smi clock log of the timed region: BSQ_CLOCKS_DIR if set, else the build folder
    out_dir = os.environ.get("BSQ_CLOCKS_DIR") or os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    sampler = ClockSampler(gpu_index, os.path.join(out_dir, "clocks_rank%d.csv" % rank))
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    times = [graphs.step() for _ in range(args.steps)]
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    st = bsq.device_status()
    assert st == 0, "device status %d" % st

    flops = sum(U["flops"] for U in units)
    ms_per_step, value = replica_throughput(float(np.mean(times)), flops, world, dev)

    # per-kernel times: the split graph, after the timed loop
    split = [graphs.split_step() for _ in range(max(20, min(args.steps, 300)))]
    q_ms = [sum(t[0] for t in ts) for ts in split]
    g_ms = [sum(t[1] for t in ts) for ts in split]
    assert bsq.device_status() == 0
    entries = per_unit_entries(units, split, peaks, peak_src)

    # GEMM aggregate: sum of flops over the flops-weighted peak time of each layer's format
    gemm_ms = float(np.mean(g_ms))
    gemm_tflops = flops / (gemm_ms * 1e-3) / 1e12
    t_peak = sum(U["flops"] / (peak_bf16 * NOMINAL_RATIO[U["fmt"]] * 1e12) for U in units)
    peak_tc = flops / t_peak / 1e12
    g_bytes = int(sum(U["gbytes"] for U in units))
    t_ideal = sum(max(U["flops"] / (peak_bf16 * NOMINAL_RATIO[U["fmt"]] * 1e12), U["gbytes"] / (hbm * 1e9))
                  for U in units)
    fmts = sorted({FMT_NAME[U["fmt"]] for U in units})
    khash = kernel_source_hash()
    gemm_roof = {"bound": "tensor", "achieved": gemm_tflops, "peak": peak_tc, "unit": "TFLOP/s",
                 "frac": gemm_tflops / peak_tc, "traffic": recorded_traffic(khash, wl.name, "gemm"),
                 "peak_source": "%s bf16 %.1f TFLOP/s x nominal ratio (%s)" % (
                     peak_src, peak_bf16, ", ".join("%s x%.0f" % (f, NOMINAL_RATIO[f]) for f in fmts)),
                 "attainable_frac": t_ideal / (gemm_ms * 1e-3), "kernel": "gemm_kernel",
                 "ms_per_step": gemm_ms, "algorithmic_bytes": g_bytes,
                 "per_launch": "all GEMM launches of a step together: 2MNK summed over the layers / "
                               "their summed event times"}
    q_bytes = sum(U["qbytes"] for U in units)
    q_ms_mean = float(np.mean(q_ms))
    q_gbs = q_bytes / (q_ms_mean * 1e-3) / 1e9
    quant = {"bound": "hbm", "achieved": q_gbs, "unit": "GB/s", "peak": hbm, "frac": q_gbs / hbm,
             "ms_per_step": q_ms_mean, "bytes_per_step": q_bytes, "peak_source": "%s HBM copy" % peak_src,
             "traffic": recorded_traffic(khash, wl.name, "quantize"), "kernel": "quantize (%s)" % ", ".join(
                 sorted({k for U in units for k in U["qkernels"]})),
             "per_launch": "all quantizer launches of a step together (NVFP4 with a computed per-tensor "
                           "scale: its amax pass included): algorithmic bytes / summed event times"}
    # the dominant kernel class: the larger share of the split step
    gemm_share = gemm_ms / (gemm_ms + q_ms_mean)
    roofline = dict(gemm_roof if gemm_share >= 0.5 else quant)
    roofline["share"] = gemm_share if gemm_share >= 0.5 else 1.0 - gemm_share

    # ------------------------------------------------------------ end to end through host buffers
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    h2d = sum(v.numel() * v.element_size() for U in units for v in U["hosts"].values() if v is not None)
    d2h = sum(U["D"][k].numel() * 2 for U in units for k in U.get("outs", ("out",)))

    # two device buffer sets per unit; streams: copy in, compute, copy out
    s_in, s_cmp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    bufs = []
    for j in range(2):
        sets = []
        for U in units:
            D = U["alloc"]()
            for k in U.get("outs", ("out",)):
                D["h" + k] = torch.empty(D[k].shape, dtype=torch.bfloat16).pin_memory()
            sets.append(D)
        bufs.append({"D": sets, "in_done": torch.cuda.Event(), "cmp_done": torch.cuda.Event(),
                     "out_done": torch.cuda.Event()})

    def e2e_step(i):
        B = bufs[i % 2]
        with torch.cuda.stream(s_in):
            s_in.wait_event(B["cmp_done"])  # inputs of the step two back consumed
            for U, D in zip(units, B["D"]):
                for k, v in U["hosts"].items():
                    if v is not None:
                        D[k].copy_(v, non_blocking=True)
            B["in_done"].record(s_in)
        s_cmp.wait_event(B["in_done"])
        s_cmp.wait_event(B["out_done"])  # result of the step two back copied out
        for U, D in zip(units, B["D"]):
            U["quant"](D, s_cmp)
            U["gemm"](D, s_cmp)
        B["cmp_done"].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(B["cmp_done"])
            for U, D in zip(units, B["D"]):
                for k in U.get("outs", ("out",)):
                    D["h" + k].copy_(D[k], non_blocking=True)
            B["out_done"].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    s_in.wait_stream(s_out)
    e1.record(s_in)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_value = world * flops / (e2e_ms * 1e-3) / 1e12
    assert bsq.device_status() == 0
    del bufs, graphs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "+".join(fmts), "data": "synthetic", "config": config_of(wl),
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roofline,
        "gemms": entries,
        "gemm": gemm_roof,
        "quantize": quant,
        "split_ms_per_step": float(np.mean([q + g for q, g in zip(q_ms, g_ms)])),
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "how": "Python API call by call; pinned host copies in and out every step, overlapped across "
                       "consecutive steps on 3 streams with double-buffered device memory"},
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
        "kernel_source_hash": khash,
    }
    del units
    torch.cuda.empty_cache()
    if world == 1 and not args.no_other_configs and args.workload == HEADLINE:
        line["other_configs"] = [time_other_config(n, bsq, dev, flush, peaks, peak_src, reps=30)
                                 for n in OTHER_CONFIGS]
        line["other_configs_note"] = ("the study's other configurations, timed per layer in the same run "
                                      "(split graph, L2 flushed); parity cases, not the headline")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, secs, cores, desc = oracle_sample(wl, target_s=args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
                                "seconds": secs, "quantize": cpu_quantize_sample(wl)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=HEADLINE)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="size of the CPU oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true", help="skip timing the non-headline configurations")
    ap.add_argument("--traffic-capture", metavar="SIDECAR",
                    help="run --warmup steps for an ncu launch list with DRAM counters, write SIDECAR, print nothing")
    ap.add_argument("--record-traffic", nargs=2, metavar=("CSV", "SIDECAR"),
                    help="turn a --traffic-capture run's ncu CSV into profiles/traffic.json (no GPU)")
    ap.add_argument("--traffic-command", default="", help="the capture's command line, stored with the record")
    ap.add_argument("--layers", help="with --traffic-capture: only these layers (comma-separated names)")
    args = ap.parse_args()
    if args.record_traffic:
        return record_traffic(args.record_traffic[0], args.record_traffic[1], args.traffic_command)
    if args.traffic_capture:
        return traffic_capture(args)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
        try:
            return run_gpu(args, rank, world)
        finally:
            dist.destroy_process_group()
    return run_gpu(args, rank, world)


if __name__ == "__main__":
    sys.exit(main())
