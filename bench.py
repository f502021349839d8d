#!/usr/bin/env python
"""Benchmark of the GB300 Gated DeltaNet core.

Metric: GDN core tokens/s for forward + backward at H=32 V heads (16 Q/K heads),
dk = dv = 128, T = 32768, bf16 I/O, stateful (h0, dO and dHT given) -- the
single-GPU GDN-core matrix of the "Linear Attention CP 融合算子 PR #1114
测试报告" (section 4).  One step = one training-step forward (gdn_fwd_ctx) + its
backward (gdn_bwd_ctx) over the whole sequence.  Inputs are synthetic (seeded N(0,1)
etc.), resident in HBM and larger than L2 (q, k, v alone are ~0.8 GB).  The "e2e"
figure copies every step's inputs from pinned host memory (double-buffered, so that
the next step's copies overlap this step's compute) and reads h_T and dH0 back.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Prints one JSON line (rank 0).  With N > 1 (torchrun) every rank runs an
independent replica of the workload (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN core tokens/s fwd+bwd, H=32 d=128 T=32K bf16"
UNIT = "tokens/s"
C = 64

# Fallback peaks (one earlier GB300 measurement) when MEASURED_PEAKS.json is absent.
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
SM_COUNT = 152
FP32_LANES_PER_SM = 128


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="stateful32k",
                    choices=["stateful32k", "long64k", "fwd8k"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-kernel-profile", action="store_true")
    ap.add_argument("--no-lengths", action="store_true",
                    help="skip the 8K/16K/32K/64K sequence-length matrix")
    ap.add_argument("--T", type=int, default=0,
                    help="override the sequence length (smaller cases for profiling)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained",
                                                      pk["bf16_tflops"])),
                "sm_max_mhz": float(pk.get("sm_max_mhz", 2070.0)), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0, "source": "fallback"}


# ----------------------------------------------------------- algorithmic work

def step_algorithmic(w):
    """Algorithmic flops and HBM bytes of one fwd+bwd (and fwd alone) of workload w.

    Flops per token per V head (C = 64): F_fwd = 2C(3dk + 2dv) + 6 dk dv + C^2/3
    (KK^T, QK^T, T.K, T.V, P.V', the three state products, the triangular
    solve); forward + backward = 3 F_fwd.  Bytes: every input read once and every
    output written once in its I/O dtype (bf16 tensors, fp32 gates/states).
    """
    dk, dv, H, Hqk, B, T = w.dk, w.dv, w.H, w.Hqk, w.B, w.T
    e = 2  # bf16
    f_fwd = 2 * C * (3 * dk + 2 * dv) + 6 * dk * dv + C * C / 3
    tok = B * T
    flops_fwd = f_fwd * tok * H
    state = B * H * dk * dv * 4
    fwd_bytes = tok * (2 * Hqk * dk * e + H * dv * e + 2 * H * e) + tok * H * dv * e
    fwd_bytes += state * (2 if w.h0_std else 1)              # h0 read, hT written
    bwd_bytes = tok * (2 * Hqk * dk * e + H * dv * e + 2 * H * e) + tok * H * dv * e  # + dO
    bwd_bytes += tok * (2 * Hqk * dk * e + H * dv * e + 2 * H * 4)                  # grads
    bwd_bytes += state * ((1 if w.h0_std else 0) + (1 if w.with_dHT else 0) + 1)    # h0,dHT,dH0
    return {"flops_fwd": flops_fwd, "flops_step": 3 * flops_fwd, "bytes_fwd": fwd_bytes,
            "bytes_step": fwd_bytes + bwd_bytes}


def kernel_alg(name, w):
    """(flops, bytes) of the method's algorithmic work owned by one launch of `name`.

    The per-token figures of step_algorithmic, split over the launches that own them:
    each input or output tensor of a pass is counted once, at the launch that reads or
    writes it; each contraction of the method once, at the launch that performs it.
    Forward: the prologue reads q, k, v, a, b and forms K K^T, Q K^T, T K, T V and the
    solve; the output chain owns the three state products and P V', writes o and h_T and
    reads h0.  Backward: the reverse chain owns the state-gradient recurrence (K~ dS,
    W^T dV': 4 dk dv per token and head) and the state tensors h0, dH_T, dH0; the
    gradient kernel owns every other gradient contraction, reads the forward inputs
    again and dO, and writes dv, dg, dbeta; the Q/K head sum writes dq, dk.  Summaries,
    prefixes and recomputation (the recomputing backward's prologue) are overhead of the
    design: no algorithmic work.
    """
    op, kname = name.split(".", 1)
    dk, dv, H, Hqk, B = w.dk, w.dv, w.H, w.Hqk, w.B
    tok = B * w.T
    e = 2
    state = B * H * dk * dv * 4
    f_local = 2 * C * (3 * dk + dv) + C * C / 3   # K K^T, Q K^T, T K, T V, the solve
    f_chain = 6 * dk * dv + 2 * C * dv            # W S, Q S, K~^T V', P V'
    f_fwd = f_local + f_chain
    f_rev = 4 * dk * dv
    in_fwd = tok * (2 * Hqk * dk * e + H * dv * e + 2 * H * e)
    if kname == "prep_tc":
        return (f_local * tok * H, in_fwd) if op == "fwd" else (0.0, 0.0)
    if kname == "apply_chain_tc":
        return f_chain * tok * H, tok * H * dv * e + state * (2 if w.h0_std else 1)
    if kname in ("states_pair_tc", "dstates_chain_tc"):
        return f_rev * tok * H, state * ((1 if w.h0_std else 0) + (1 if w.with_dHT else 0) + 1)
    if kname == "grad_tc":
        return (2 * f_fwd - f_rev) * tok * H, in_fwd + tok * (H * dv * e + H * dv * e + 2 * H * 4)
    if kname == "qk_grad_tc":
        return 0.0, tok * 2 * Hqk * dk * e
    return 0.0, 0.0


def kernel_work(name, w, P):
    """(flops, bytes) the design itself moves and computes in one launch of `name`
    (its intermediates included): the "model" figures beside the algorithmic ones.

    name is "<fwd|bwd>.<kernel>" as listed by gdn_kernel_info.  Flops count each
    contraction the kernel performs once per (chunk, V head) at its natural size
    (C = 64, dk = dv = 128); bytes count every tensor the kernel reads or writes
    in HBM once (bf16 tiles, fp32 states and gates).
    """
    op, kname = name.split(".", 1)
    dk, dv, H, Hqk, B = w.dk, w.dv, w.H, w.Hqk, w.B
    NC = math.ceil(w.T / C)
    ch = B * H * NC                       # (chunk, V head) pairs
    tok = B * w.T
    frac = (P - 1) / P if P > 1 else 0.0
    tile = C * 128 * 2                    # one [64][128] bf16 tile
    tile_p = C * C * 2                    # one [64][64] bf16 tile
    state = dk * dv * 4
    mm = lambda m, n, k: 2.0 * m * n * k  # noqa: E731
    if kname == "prep_tc":
        f = 2 * mm(C, C, dk) + C ** 3 / 3 + mm(C, dk, C) + mm(C, dv, C)
        rd = tok * (2 * Hqk * dk * 2 + H * dv * 2 + 2 * H * 2)
        # W, U, P and T images, gates, norm factors (the T images are written for the
        # backward: by gdn_fwd_ctx into its context, by gdn_bwd's own prologue)
        wr = ch * (2 * tile + 2 * tile_p + C * 4) + B * Hqk * NC * 2 * C * 4
        return f * ch, rd + wr
    if kname == "summary_chain_tc":  # gdn_fwd_ctx: [M | S] parts of every segment
        f = 2 * (mm(C, dv, dk) + mm(dk, dv, C)) * ch
        byt = ch * (3 * tile + C * 8) + 2 * P * B * H * state
        return f, byt
    if kname == "grad_summary_tc":   # gdn_bwd_ctx: gradient summaries of segments 1..P-1
        return kernel_work("bwd.grad_summary_chain_tc", w, P)
    if kname == "ctx_init":
        return 0.0, 2 * B * H * state
    if kname == "summary_pair_tc":   # [M | S] of every segment + gradient summaries
        f1 = 2 * (mm(C, dv, dk) + mm(dk, dv, C)) * ch
        b1 = ch * (3 * tile + C * 8) + 2 * P * B * H * state
        f2, b2 = kernel_work("bwd.grad_summary_chain_tc", w, P)
        return f1 + f2, b1 + b2
    if kname == "states_pair_tc":    # chunk-start states + chunk-end state gradients
        f1, b1 = kernel_work("bwd.states_chain_tc", w, P)
        f2, b2 = kernel_work("bwd.dstate_chain_tc", w, P)
        return f1 + f2, b1 + b2
    if kname == "apply_chain_tc":  # gdn_fwd_ctx: also every chunk-start state image
        f = (2 * mm(C, dv, dk) + mm(dk, dv, C) + mm(C, dv, C)) * ch
        byt = ch * (5 * tile + tile_p + C * 12 + dk * dv * 2) + \
            B * H * state * (1 + (1 if P > 1 or w.h0_std else 0))
        return f, byt
    if kname == "states_chain_tc":
        f = (mm(C, dv, dk) + mm(dk, dv, C)) * ch
        return f, ch * (3 * tile + C * 8 + dk * dv * 2)
    if kname in ("grad_summary_chain_tc", "dstate_chain_tc"):
        f = (mm(C, dv, C) + mm(C, dv, dk) + 2 * mm(dk, dv, C)) * ch
        byt = ch * (4 * tile + tile_p + C * 12)
        if kname == "dstate_chain_tc":
            return f, byt + ch * dk * dv * 2
        return f * frac, byt * frac
    if kname == "grad_tc":
        f = (5 * mm(C, 128, 128) + 11 * mm(C, 128, C)) * ch
        byt = ch * (8 * tile + 2 * dk * dv * 2 + 2 * tile_p + 3 * tile + 2 * C * 4)
        return f, byt
    if kname == "qk_grad_tc":
        return 0.0, tok * (H * 2 * dk * 2 + Hqk * 2 * dk * 2 * 2)
    if kname in ("prefix", "prefix_bwd"):
        return mm(dk, dv, dk) * B * H * max(P - 1, 0), B * H * max(P - 1, 0) * 3 * state
    if kname == "prefix_pair":
        return 2 * mm(dk, dv, dk) * B * H * max(P - 1, 0), 2 * B * H * max(P - 1, 0) * 3 * state
    return 0.0, 0.0


# ncu-measured DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of
# a kernel at the bench workload, valid only for the source file it was taken from
# (its SHA-256); the capture is summarised under profiles/.
E2E_COPY_STREAMS = 4  # side streams for the host-to-device copies of the end-to-end step


MEASURED_TRAFFIC = {
    "bwd.grad_tc": {"T": 32768, "bytes_per_launch": 3022233856 + 837304320,
                    "src": "chunked_state_scan_gated_gb300/csrc/gdn_tc_grad.cu",
                    "sha256": "b91b783c856d86caebb1645ef9b1beef4e804b3fbdd19921f705ec142da90e2d"},
}


def _src_sha(rel):
    import hashlib
    try:
        with open(os.path.join(ROOT, rel), "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None


def measured_traffic(kernel, T):
    rec = MEASURED_TRAFFIC.get(kernel)
    if not rec or rec["T"] != T or _src_sha(rec["src"]) != rec["sha256"]:
        return None
    return rec["bytes_per_launch"]


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        out = os.environ.get("GDN_BENCH_CLOCKS_DIR", tempfile.gettempdir())
        self.path = os.path.join(out, f"gdn_bench_clocks_gpu{gpu_index}_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- per-call statistics

def stats_ms(xs):
    """median, min and p90 (nearest rank) of per-call times in ms."""
    ys = sorted(xs)
    p90 = ys[min(len(ys) - 1, max(0, math.ceil(0.9 * len(ys)) - 1))]
    return {"median": statistics.median(ys), "min": ys[0], "p90": p90, "n": len(ys)}


LENGTHS = (8192, 16384, 32768, 65536)


def measure_lengths(gdn, gi, torch, stream, peaks, args, per_step):
    """The sequence-length matrix: B = 1, Hqk = 16, H = 32, dk = dv = 128, bf16, stateful.

    Per length: gdn_fwd, the context pair (gdn_fwd_ctx + gdn_bwd_ctx) and the recompute
    pair (gdn_fwd + gdn_bwd), every call timed alone with CUDA events on the launching
    stream (median, min, p90 over --steps calls after 3 warm-up calls), tokens/s of the
    median, the fraction of the algorithmic roofline (sustained bf16 peak, measured HBM
    bandwidth) that the median reaches, and the incremental peak device memory of one
    call that allocates its own outputs, context and workspace.
    """
    import dataclasses
    out = {}
    steps = max(args.steps, 5)
    for T in LENGTHS:
        w = dataclasses.replace(gi.STATEFUL_32K, T=T, name=f"fwdbwd_bf16_T{T}_h16x32_d128_stateful")
        inp = gi.make_inputs(w)
        d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
        fwd_in = (d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"])
        p = gdn.make_problem(d["q"], d["v"])
        alg = step_algorithmic(w)
        t_fwd = max(alg["flops_fwd"] / (peaks["bf16_tflops_sustained"] * 1e12),
                    alg["bytes_fwd"] / (peaks["hbm_gbs"] * 1e9))
        t_step = max(alg["flops_step"] / (peaks["bf16_tflops_sustained"] * 1e12),
                     alg["bytes_step"] / (peaks["hbm_gbs"] * 1e9))

        def call_fwd():
            return gdn.gdn_fwd(*fwd_in, d["h0"], None, problem=p, stream=stream)

        def call_ctx():
            ctx = gdn.ctx_buffer(p)
            o, hT, _ = gdn.gdn_fwd_ctx(*fwd_in, d["h0"], None, ctx=ctx, problem=p, stream=stream)
            return gdn.gdn_bwd_ctx(*fwd_in, ctx, d["dO"], d["dHT"], None, problem=p,
                                   stream=stream), o, hT

        def call_recompute():
            o, hT = gdn.gdn_fwd(*fwd_in, d["h0"], None, problem=p, stream=stream)
            return gdn.gdn_bwd(*fwd_in, d["dO"], d["dHT"], d["h0"], None, problem=p,
                               stream=stream), o, hT

        def peak_bytes(fn):
            torch.cuda.synchronize()
            base = torch.cuda.memory_allocated()
            torch.cuda.reset_peak_memory_stats()
            r = fn()
            torch.cuda.synchronize()
            peak = torch.cuda.max_memory_allocated() - base
            del r
            return peak

        row = {"tokens": T}
        for name, fn, t_roof in (("fwd", call_fwd, t_fwd), ("fwd_bwd_ctx", call_ctx, t_step),
                                 ("fwd_bwd_recompute", call_recompute, t_step)):
            for _ in range(3):
                fn()
            st = stats_ms(per_step(fn, steps))
            row[name] = {"ms": st, "tokens_per_s": T / (st["median"] / 1e3),
                         "roofline_frac": 1e3 * t_roof / st["median"],
                         "t_roof_ms": 1e3 * t_roof,
                         "peak_mem_bytes": peak_bytes(fn)}
        out[str(T)] = row
        del d, inp, p
        torch.cuda.empty_cache()
    return {"rows": out, "timing": "each call alone, CUDA events on the launching stream; "
                                   "outputs, context and workspace allocated per call",
            "peak_mem": "torch max_memory_allocated over one call minus the bytes held "
                        "before it (inputs excluded)"}


# ---------------------------------------------------------------- CPU baseline

def oracle_sample(w, T_sample, nthreads):
    """Time the fp64 oracle's fwd + bwd on the first T_sample tokens of every head."""
    import oracle
    from chunked_state_scan_gated_gb300 import inputs as gi
    inp = gi.make_inputs(w, T=T_sample)
    n = gi.to_numpy64(inp)
    oracle.build()
    t0 = time.perf_counter()
    oracle.fwd(n["q"], n["k"], n["v"], n["a"], n["b"], n["A_log"], n["dt_bias"], h0=n["h0"],
               nthreads=nthreads)
    oracle.bwd(n["q"], n["k"], n["v"], n["a"], n["b"], n["A_log"], n["dt_bias"], n["dO"],
               n["dHT"], h0=n["h0"], nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform string)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu model")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(w, T_sample=8192, runs=3):
    """The fp64 oracle on the host cores: median of `runs` fwd + bwd over the first T_sample
    tokens of every head (all cores, one OpenMP thread per (batch, V head) at most), plus one
    single-thread run over one Q/K head group (H/Hqk V heads) of T_sample tokens."""
    import dataclasses
    threads = min(cpu_threads(), w.B * w.H)
    secs = [oracle_sample(w, T_sample, threads) for _ in range(runs)]
    med = statistics.median(secs)
    one = dataclasses.replace(w, Hqk=1, H=w.H // w.Hqk)
    s1 = oracle_sample(one, T_sample, 1)
    return {"value": T_sample * w.B / med, "unit": UNIT, "cores": threads, "kind": "oracle",
            "host_cores": cpu_threads(), "cpu_model": cpu_model(),
            "runs_s": [round(x, 3) for x in secs],
            "sample": f"first {T_sample} tokens of all {w.H} V heads, fp64 C oracle fwd+bwd "
                      f"(OpenMP, {threads} threads), median of {runs} runs",
            "single_thread": {"tokens_per_s": T_sample * w.B / s1, "seconds": round(s1, 3),
                              "sample": f"{T_sample} tokens of one Q/K head group "
                                        f"({w.H // w.Hqk} V heads), 1 thread"}}


def workload_of(name, T=0):
    import dataclasses

    from chunked_state_scan_gated_gb300 import inputs as gi
    w = {"stateful32k": gi.STATEFUL_32K, "long64k": gi.LONG_64K, "fwd8k": gi.FWD_8K}[name]
    if T:
        w = dataclasses.replace(w, T=T, name=w.name.replace(f"T{w.T}", f"T{T}"))
    return w


def config_of(w, args, world):
    return {"workload": w.name, "global_batch": w.B * world, "seq_len": w.T,
            "heads_qk": w.Hqk, "heads_v": w.H, "dk": w.dk, "dv": w.dv, "chunk": C,
            "initial_state": bool(w.h0_std), "parallelism": f"replicas{world}",
            "l2": "inputs larger than L2 (q,k,v,dO ~1.1 GB read per step); no flush"}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = workload_of(args.workload, args.T)
    threads = min(cpu_threads(), w.B * w.H)
    T_sample = 1024
    for _ in range(args.warmup):
        oracle_sample(w, T_sample, threads)
    times = [oracle_sample(w, T_sample, threads) for _ in range(args.steps)]
    total = sum(times)
    value = args.steps * T_sample * w.B / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args, 1),
        "cpu_baseline": {"kind": "oracle", "value": value, "unit": UNIT, "cores": threads,
                         "host_cores": cpu_threads(), "cpu_model": cpu_model(),
                         "sample": f"first {T_sample} tokens of all {w.H} V heads per step, "
                                   f"fp64 C oracle fwd+bwd (OpenMP)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- rank helpers

def ranks_barrier(world):
    """Barrier over the process group (no-op for one rank)."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def ranks_max(x, world, device):
    """Max of a per-rank float over all ranks (the slowest replica's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ms_max, tokens_per_rank, world):
    """Whole-job tokens/s: every replica processed its own tokens within the slowest time."""
    return world * tokens_per_rank / (ms_max / 1e3)


# ---------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    import torch.distributed as dist

    import chunked_state_scan_gated_gb300 as gdn
    from chunked_state_scan_gated_gb300 import inputs as gi

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        ranks_barrier(world)

    def max_over_ranks(x):
        return ranks_max(x, world, "cuda")

    w = workload_of(args.workload, args.T)
    inp = gi.make_inputs(w, seed=w.seed + 1000 * rank)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    p = gdn.make_problem(d["q"], d["v"])
    wsf = gdn.workspace(p, gdn.GDN_OP_FWD)
    wsb = gdn.workspace(p, gdn.GDN_OP_BWD)
    wsfc = gdn.workspace(p, gdn.GDN_OP_FWD_CTX)
    wsbc = gdn.workspace(p, gdn.GDN_OP_BWD_CTX)
    B, T, H, dv = d["v"].shape
    dk = d["q"].shape[3]
    o = torch.empty_like(d["v"])
    hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device="cuda")
    dq, dkk, dvv = torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"])
    dg = torch.empty((B, T, H), dtype=torch.float32, device="cuda")
    dbeta = torch.empty_like(dg)
    dH0 = torch.empty_like(hT)
    stream = torch.cuda.current_stream()

    ctx = gdn.ctx_buffer(p)

    def fwd():
        gdn.gdn_fwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["h0"],
                    None, o=o, hT=hT, ws=wsf, problem=p, stream=stream)

    def fwd_ctx():  # the training-step forward: also keeps the segment states for the backward
        gdn.gdn_fwd_ctx(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                        d["h0"], None, ctx=ctx, o=o, hT=hT, ws=wsfc, problem=p, stream=stream)

    def bwd_ctx():
        gdn.gdn_bwd_ctx(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], ctx,
                        d["dO"], d["dHT"], None, dq=dq, dk=dkk, dv=dvv, dg=dg, dbeta=dbeta,
                        dH0=dH0, ws=wsbc, problem=p, stream=stream)

    def bwd_recompute():  # gdn_bwd: recomputes the segment summaries and their prefix
        gdn.gdn_bwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["dO"],
                    d["dHT"], d["h0"], None, dq=dq, dk=dkk, dv=dvv, dg=dg, dbeta=dbeta, dH0=dH0,
                    ws=wsb, problem=p, stream=stream)

    def step():
        fwd_ctx()
        bwd_ctx()

    def step_recompute():
        fwd()
        bwd_recompute()

    def timed(fn, steps):
        barrier()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return ev0.elapsed_time(ev1) / steps

    def per_step(fn, steps):
        """ms of each of `steps` calls (CUDA events on the launching stream)."""
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for e0, e1 in evs:
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return [e0.elapsed_time(e1) for e0, e1 in evs]

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert gdn.gdn_check_device_status(wsbc) == gdn.GDN_OK

    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    gpu_id = vis.split(",")[local].strip() if vis else str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    ms_step = timed(step, args.steps)
    clocks = sampler.stop()
    ms_step = max_over_ranks(ms_step)
    step_stats = stats_ms(per_step(step, args.steps))
    ms_fwd = max_over_ranks(timed(fwd, args.steps))
    fwd_stats = stats_ms(per_step(fwd, args.steps))
    ms_recompute = max_over_ranks(timed(step_recompute, args.steps))
    tokens = B * T
    value = job_throughput(ms_step, tokens, world)

    nf = len(gdn.gdn_kernel_info(p, gdn.GDN_OP_FWD_CTX))
    nb = len(gdn.gdn_kernel_info(p, gdn.GDN_OP_BWD_CTX))
    peaks = load_peaks()
    alg = step_algorithmic(w)
    t_roof_step = max(alg["flops_step"] / (peaks["bf16_tflops_sustained"] * 1e12),
                      alg["bytes_step"] / (peaks["hbm_gbs"] * 1e9))
    t_roof_fwd = max(alg["flops_fwd"] / (peaks["bf16_tflops_sustained"] * 1e12),
                     alg["bytes_fwd"] / (peaks["hbm_gbs"] * 1e9))

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(w, args, world),
        "fwd": {"ms": ms_fwd, "tokens_per_s": job_throughput(ms_fwd, tokens, world),
                "per_call": fwd_stats},
        "step": "gdn_fwd_ctx + gdn_bwd_ctx (the backward reads the forward's segment states)",
        "step_per_call": step_stats,
        "fwd_bwd_recompute": {"ms": ms_recompute,
                              "tokens_per_s": job_throughput(ms_recompute, tokens, world),
                              "calls": "gdn_fwd + gdn_bwd (no context)"},
        "gpu_launches": args.steps * (nf + nb),
        "step_roofline": {
            "flops": alg["flops_step"], "bytes": alg["bytes_step"],
            "t_roof_ms": 1e3 * t_roof_step, "frac": 1e3 * t_roof_step / ms_step,
            "fwd_t_roof_ms": 1e3 * t_roof_fwd, "fwd_frac": 1e3 * t_roof_fwd / ms_fwd,
            "peaks": f"{peaks['source']}: {peaks['hbm_gbs']} GB/s, "
                     f"{peaks['bf16_tflops_sustained']} TF/s bf16 sustained"},
        "clocks": clocks,
    }

    # Per-kernel CUDA-event timing: K profiled steps made of single-kernel calls.
    if not args.no_kernel_profile:
        names_f = gdn.gdn_kernel_info(p, gdn.GDN_OP_FWD_CTX)
        names_b = gdn.gdn_kernel_info(p, gdn.GDN_OP_BWD_CTX)
        tot = {}
        reps = max(1, args.steps)
        step()
        torch.cuda.synchronize()
        for op, names in ((gdn.GDN_OP_FWD_CTX, names_f), (gdn.GDN_OP_BWD_CTX, names_b)):
            for i, nm in enumerate(names):
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(reps)]
                for e0, e1 in evs:
                    e0.record(stream)
                    if op == gdn.GDN_OP_FWD_CTX:
                        gdn.gdn_fwd_ctx_kernel(i, d["q"], d["k"], d["v"], d["a"], d["b"],
                                               d["A_log"], d["dt_bias"], d["h0"], None, o, hT,
                                               ctx, wsfc, problem=p, stream=stream)
                    else:
                        gdn.gdn_bwd_ctx_kernel(i, d["q"], d["k"], d["v"], d["a"], d["b"],
                                               d["A_log"], d["dt_bias"], ctx, None, d["dO"],
                                               d["dHT"], dq, dkk, dvv, dg, dbeta, dH0, wsbc,
                                               problem=p, stream=stream)
                    e1.record(stream)
                torch.cuda.synchronize()
                ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
                key = ("fwd." if op == gdn.GDN_OP_FWD_CTX else "bwd.") + nm
                tot[key] = ms
        P = gdn.gdn_resolved_segments(p, gdn.GDN_OP_FWD)
        dom = max(tot, key=tot.get)
        ms_dom = tot[dom]
        flops, byt = kernel_alg(dom, w)
        mflops, mbyt = kernel_work(dom, w, P)
        # the kernel is timed alone: burst peaks
        t_f = flops / (peaks["bf16_tflops"] * 1e12)
        t_b = byt / (peaks["hbm_gbs"] * 1e9)
        if t_f >= t_b:
            bound, peak, punit = "tensor", peaks["bf16_tflops"], "TFLOP/s"
            achieved = flops / (ms_dom / 1e3) / 1e12
        else:
            bound, peak, punit = "hbm", peaks["hbm_gbs"], "GB/s"
            achieved = byt / (ms_dom / 1e3) / 1e9
        traffic = measured_traffic(dom, w.T)
        line["roofline"] = {
            "kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": punit,
            "frac": achieved / peak, "traffic": traffic,
            "traffic_over_algorithmic": (traffic / byt) if (traffic and byt) else None,
            "ms_per_launch": ms_dom, "algorithmic_flops_per_launch": flops,
            "algorithmic_bytes_per_launch": byt,
            "algorithmic": "the method's own contractions and input/output tensors owned by "
                           "this launch (per-token work of step_roofline, split by launch)",
            "model_flops_per_launch": mflops, "model_bytes_per_launch": mbyt,
            "model": "what the design computes and moves, its intermediates included",
            "timing": f"CUDA events around each launch, mean of {reps} launches",
            "peak_source": f"{peaks['source']} (burst: kernel timed alone)",
        }
        kr = {}
        for k, v in tot.items():
            fl, by = kernel_alg(k, w)
            mfl, mby = kernel_work(k, w, P)
            kr[k] = {"ms": round(v, 4),
                     "alg_frac": round(max(fl / (peaks["bf16_tflops"] * 1e12),
                                           by / (peaks["hbm_gbs"] * 1e9)) / (v / 1e3), 4),
                     "model_tflops": round(mfl / (v / 1e3) / 1e12, 1),
                     "model_gbs": round(mby / (v / 1e3) / 1e9, 1)}
        line["kernel_roofline"] = kr
        line["kernel_ms"] = {k: round(v, 4) for k, v in tot.items()}
        if traffic is not None:
            line["step_roofline"]["traffic_over_algorithmic_note"] = (
                "ncu DRAM bytes of the dominant kernel only; see profiles/ for the launch list")

    # Every sequence length of the measurement matrix (B = 1, H = 32, d = 128, stateful):
    # forward, training step (context pair) and gdn_fwd + gdn_bwd, each call timed alone
    # with CUDA events (median, min, p90), the roofline fraction of the median, and the
    # incremental peak device memory of one call that allocates its own outputs and
    # workspace.
    if not args.no_lengths and world == 1:
        line["lengths"] = measure_lengths(gdn, gi, torch, stream, peaks, args, per_step)

    # The Conv1D + SiLU prologue over the projected q, k, v of this workload (C = 2 Hqk dk +
    # H dv channels, K = 4 taps, a left halo, no bias): forward and backward, each timed
    # alone with CUDA events, against the measured HBM bandwidth (both are bandwidth-bound:
    # x read and y written; x, dy read and dx written).
    if not args.no_kernel_profile:
        Cc, Kc = 2 * w.Hqk * w.dk + w.H * w.dv, 4
        ci = gi.make_conv_inputs(B, T, Cc, Kc, torch.bfloat16, seed=w.seed + 77, bias=False)
        cd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in ci.items()}
        cp = gdn.make_conv_problem(cd["x"], Kc)
        cy = torch.empty_like(cd["x"])
        cdx = torch.empty_like(cd["x"])
        cdw = torch.empty((Cc, Kc), dtype=torch.float32, device="cuda")
        cdh = torch.empty_like(cd["halo"])
        cws = torch.empty(gdn.gdn_conv_silu_bwd_workspace_size(cp), dtype=torch.uint8,
                          device="cuda")

        def conv_f():
            gdn.gdn_conv_silu_fwd(cd["x"], cd["w"], None, cd["halo"], y=cy, problem=cp,
                                  stream=stream)

        def conv_b():
            gdn.gdn_conv_silu_bwd(cd["x"], cd["w"], None, cd["halo"], cd["dy"], dx=cdx, dw=cdw,
                                  dhalo=cdh, want_dbias=False, ws=cws, problem=cp, stream=stream)

        for _ in range(3):
            conv_f()
            conv_b()
        ms_cf, ms_cb = timed(conv_f, args.steps), timed(conv_b, args.steps)
        el = B * T * Cc
        bytes_f, bytes_b = 4 * el, 6 * el + B * (Kc - 1) * Cc * 4 + Cc * Kc * 4
        line["conv1d_silu"] = {
            "shape": f"B={B} T={T} C={Cc} K={Kc} bf16, halo, no bias",
            "fwd_ms": ms_cf, "bwd_ms": ms_cb,
            "fwd_gbs": bytes_f / (ms_cf / 1e3) / 1e9, "bwd_gbs": bytes_b / (ms_cb / 1e3) / 1e9,
            "fwd_frac": bytes_f / (ms_cf / 1e3) / 1e9 / peaks["hbm_gbs"],
            "bwd_frac": bytes_b / (ms_cb / 1e3) / 1e9 / peaks["hbm_gbs"],
            "algorithmic_bytes": {"fwd": bytes_f, "bwd": bytes_b},
            "peak": f"{peaks['hbm_gbs']} GB/s ({peaks['source']})"}
        del cd, cy, cdx, cdw, cdh, cws

        # The same Conv1D fused into the training-step forward (gdn_fwd_conv: the chunk
        # prologue loads x_q, x_k, x_v, convolves each chunk in shared memory and writes the
        # activated q, k, v once), against the stand-alone Conv1D of the three tensors followed
        # by gdn_fwd_ctx; both calls timed alone with CUDA events, and their outputs compared.
        xs, wts, hls = [], [], []
        for i, heads in enumerate((w.Hqk, w.Hqk, w.H)):
            c = gi.make_conv_inputs(B, T, heads * dk, Kc, torch.bfloat16, seed=w.seed + 80 + i,
                                    bias=False)
            xs.append(c["x"].view(B, T, heads, dk).cuda())
            wts.append(c["w"].cuda())
            hls.append(c["halo"].cuda())
        ys = [torch.empty_like(x) for x in xs]
        cps = [gdn.make_conv_problem(x.view(B, T, -1), Kc) for x in xs]

        def conv_fused():
            gdn.gdn_fwd_conv(tuple(xs), tuple(wts), d["a"], d["b"], d["A_log"], d["dt_bias"],
                             d["h0"], None, halo=tuple(hls), y=tuple(ys), ctx=ctx, o=o, hT=hT,
                             ws=wsfc, problem=p, stream=stream)

        def conv_only():
            for x, wt, hl, y_, cp_ in zip(xs, wts, hls, ys, cps):
                gdn.gdn_conv_silu_fwd(x.view(B, T, -1), wt, None, hl, y=y_.view(B, T, -1),
                                      problem=cp_, stream=stream)

        def conv_separate():
            conv_only()
            gdn.gdn_fwd_ctx(ys[0], ys[1], ys[2], d["a"], d["b"], d["A_log"], d["dt_bias"],
                            d["h0"], None, ctx=ctx, o=o, hT=hT, ws=wsfc, problem=p,
                            stream=stream)

        conv_separate()
        torch.cuda.synchronize()
        o_sep, y_sep = o.clone(), [y_.clone() for y_ in ys]
        conv_fused()
        torch.cuda.synchronize()
        same = torch.equal(o, o_sep) and all(torch.equal(a_, b_) for a_, b_ in zip(ys, y_sep))
        del o_sep, y_sep
        for _ in range(3):
            conv_fused()
            conv_separate()
        ms_fused = timed(conv_fused, args.steps)
        ms_sep = timed(conv_separate, args.steps)
        ms_conv3 = timed(conv_only, args.steps)
        line["conv_fused_fwd"] = {
            "shape": f"B={B} T={T} x_q, x_k [{w.Hqk}x{dk}], x_v [{w.H}x{dv}] bf16, K={Kc}, halo",
            "fused_ms": ms_fused, "fused_tokens_per_s": B * T / (ms_fused / 1e3),
            "separate_ms": ms_sep, "separate_conv_ms": ms_conv3,
            "bit_identical": bool(same),
            "calls": "gdn_fwd_conv (ctx) vs gdn_conv_silu_fwd x3 + gdn_fwd_ctx"}
        del xs, wts, hls, ys

        # The gated RMSNorm epilogue on o (rows = B T H, D = dv), forward and backward.
        ri = gi.make_rmsnorm_inputs((B, T, H, dv), torch.bfloat16, seed=w.seed + 78)
        rd = {k: v.cuda() for k, v in ri.items()}
        rp = gdn.make_rmsnorm_problem(rd["o"])
        ry, rdo, rdz = (torch.empty_like(rd["o"]) for _ in range(3))
        rdw = torch.empty((dv,), dtype=torch.float32, device="cuda")
        rws = torch.empty(gdn.gdn_rmsnorm_gated_bwd_workspace_size(rp), dtype=torch.uint8,
                          device="cuda")

        def rms_f():
            gdn.gdn_rmsnorm_gated_fwd(rd["o"], rd["z"], rd["w"], y=ry, problem=rp, stream=stream)

        def rms_b():
            gdn.gdn_rmsnorm_gated_bwd(rd["o"], rd["z"], rd["w"], rd["dy"], d_o=rdo, dz=rdz, dw=rdw,
                                      ws=rws, problem=rp, stream=stream)

        for _ in range(3):
            rms_f()
            rms_b()
        ms_rf, ms_rb = timed(rms_f, args.steps), timed(rms_b, args.steps)
        el = B * T * H * dv
        bytes_f, bytes_b = 6 * el, 10 * el
        line["rmsnorm_gated"] = {
            "shape": f"rows={B * T * H} D={dv} bf16",
            "fwd_ms": ms_rf, "bwd_ms": ms_rb,
            "fwd_gbs": bytes_f / (ms_rf / 1e3) / 1e9, "bwd_gbs": bytes_b / (ms_rb / 1e3) / 1e9,
            "fwd_frac": bytes_f / (ms_rf / 1e3) / 1e9 / peaks["hbm_gbs"],
            "bwd_frac": bytes_b / (ms_rb / 1e3) / 1e9 / peaks["hbm_gbs"],
            "algorithmic_bytes": {"fwd": bytes_f, "bwd": bytes_b},
            "peak": f"{peaks['hbm_gbs']} GB/s ({peaks['source']})"}
        del rd, ry, rdo, rdz, rdw, rws

    # Packed variable-length row (the "next" row f4): the workload's T tokens as eight
    # sequences of mixed length (seeded cut points), each with its own h0 and dH_T;
    # gdn_fwd_varlen and gdn_fwd_varlen + gdn_bwd_varlen, each timed alone.  The padded batch
    # the call runs holds N x Lmax token slots; tokens/s count the row's T real tokens, and
    # the roofline fraction is that of the monolithic algorithmic work of T tokens.
    if not args.no_kernel_profile and world == 1:
        lens = gi.length_mix(w.T, 8, seed=w.seed + 91)
        vi = gi.make_varlen_inputs(w, lens, seed=w.seed + 91)
        vd = {k: (v.cuda() if torch.is_tensor(v) and k != "cu_seqlens" else v)
              for k, v in vi.items()}
        cu = gdn.Varlen(vi["cu_seqlens"])
        vfin = (vd["q"], vd["k"], vd["v"], vd["a"], vd["b"], vd["A_log"], vd["dt_bias"])
        vp = gdn.make_problem(vd["q"], vd["v"])
        vwf = gdn.varlen_workspace(vp, cu, gdn.GDN_OP_FWD)
        vwb = gdn.varlen_workspace(vp, cu, gdn.GDN_OP_BWD)
        vo = torch.empty_like(vd["v"])
        vhT = torch.empty((len(lens), H, dk, dv), dtype=torch.float32, device="cuda")

        def vl_fwd():
            gdn.gdn_fwd_varlen(*vfin, cu, vd["h0"], o=vo, hT=vhT, ws=vwf, problem=vp,
                               stream=stream)

        def vl_step():
            vl_fwd()
            gdn.gdn_bwd_varlen(*vfin, cu, vd["dO"], vd["dHT"], vd["h0"], ws=vwb, problem=vp,
                               stream=stream)

        for _ in range(3):
            vl_step()
        torch.cuda.synchronize()
        assert gdn.gdn_varlen_check_device_status(vwb, vp, cu, gdn.GDN_OP_BWD) == gdn.GDN_OK
        ms_vf, ms_vs = timed(vl_fwd, args.steps), timed(vl_step, args.steps)
        line["varlen"] = {
            "lengths": lens, "tokens": w.T, "padded_slots": len(lens) * max(lens),
            "fwd_ms": ms_vf, "fwd_tokens_per_s": w.T / (ms_vf / 1e3),
            "fwd_bwd_ms": ms_vs, "fwd_bwd_tokens_per_s": w.T / (ms_vs / 1e3),
            "fwd_roofline_frac": 1e3 * t_roof_fwd / ms_vf,
            "fwd_bwd_roofline_frac": 1e3 * t_roof_step / ms_vs,
            "calls": "gdn_fwd_varlen; gdn_fwd_varlen + gdn_bwd_varlen (recomputing backward)"}
        del vd, vi, vo, vhT, vwf, vwb

    # End to end: pinned host inputs copied in, fwd + bwd, result states read back, every
    # step.  As an input pipeline would, the inputs are double-buffered on the device: the
    # copies of step i + 1 (on E2E_COPY_STREAMS side streams) run while step i computes; the
    # first timed step copies its own inputs with nothing to hide them behind.
    if not args.no_e2e:
        names_in = [k for k in ("q", "k", "v", "a", "b", "A_log", "dt_bias", "h0", "dO", "dHT")
                    if inp[k] is not None]
        host = {k: inp[k].pin_memory() for k in names_in}
        h_hT = torch.empty(hT.shape, dtype=hT.dtype).pin_memory()
        h_dH0 = torch.empty(dH0.shape, dtype=dH0.dtype).pin_memory()
        bi = sum(t.numel() * t.element_size() for t in host.values())
        bo = h_hT.numel() * 4 + h_dH0.numel() * 4
        cstreams = [torch.cuda.Stream() for _ in range(E2E_COPY_STREAMS)]
        bufs = [dict(d), dict(d)]
        for k in names_in:
            bufs[1][k] = torch.empty_like(d[k])
        pipe = {"i": 0, "ready": None}

        def h2d(dst_set):
            """Copies of every input into `dst_set`, queued behind the work issued so far on
            the compute stream (the step that last read that buffer); returns done events."""
            after = torch.cuda.Event()
            after.record(stream)
            i = 0
            for cs in cstreams:
                cs.wait_event(after)
            for k in names_in:
                src, dst = host[k].view(-1), dst_set[k].view(-1)
                n = src.numel()
                parts = len(cstreams) if n * src.element_size() >= (8 << 20) else 1
                for j in range(parts):
                    a, b = n * j // parts, n * (j + 1) // parts
                    with torch.cuda.stream(cstreams[i % len(cstreams)]):
                        dst[a:b].copy_(src[a:b], non_blocking=True)
                    i += 1
            evs = []
            for cs in cstreams:
                ev = torch.cuda.Event()
                ev.record(cs)
                evs.append(ev)
            return evs

        def run_step(x):
            gdn.gdn_fwd_ctx(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"], x["dt_bias"],
                            x["h0"], None, ctx=ctx, o=o, hT=hT, ws=wsfc, problem=p, stream=stream)
            gdn.gdn_bwd_ctx(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"], x["dt_bias"], ctx,
                            x["dO"], x["dHT"], None, dq=dq, dk=dkk, dv=dvv, dg=dg, dbeta=dbeta,
                            dH0=dH0, ws=wsbc, problem=p, stream=stream)

        def e2e_step():
            cur, nxt = bufs[pipe["i"] % 2], bufs[(pipe["i"] + 1) % 2]
            ready = pipe["ready"] if pipe["ready"] is not None else h2d(cur)
            pipe["ready"] = h2d(nxt)  # behind the previous step, the last reader of `nxt`
            for ev in ready:
                stream.wait_event(ev)
            run_step(cur)
            h_hT.copy_(hT, non_blocking=True)
            h_dH0.copy_(dH0, non_blocking=True)
            pipe["i"] += 1

        e2e_step()
        torch.cuda.synchronize()
        pipe["ready"] = None  # the first timed step copies its own inputs inside the timed region
        ms_e2e = max_over_ranks(timed(e2e_step, args.steps))
        torch.cuda.synchronize()
        assert torch.equal(bufs[0]["q"], bufs[1]["q"]) and torch.equal(bufs[0]["dO"], bufs[1]["dO"])
        line["e2e"] = {"value": job_throughput(ms_e2e, tokens, world), "unit": UNIT,
                       "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": ms_e2e,
                       "copies": "every step copies all its inputs from pinned host memory, "
                                 "double-buffered: step i+1's copies overlap step i's compute, the "
                                 "first timed step's copies are exposed"}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, T_sample=min(w.T, 8192))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
