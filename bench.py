#!/usr/bin/env python
"""Benchmark of the quantized linear stack of one pi0.5-shaped control step.

One step is the whole hot path over one batch of synthetic input:
  * prefix: 18 Gemma-2B-style layers on 816 tokens; per layer the four
    distinct inputs are rotated (block Hadamard 128) and quantized per token,
    then q|k|v and gate|up run at W4A4 and o and down at W8A8;
  * expert at W4A4: 10 denoising steps x 18 Gemma-300M-style layers on 50
    action tokens, activations quantized with static per-step scales
    (calibrated beforehand from 8 seeded draws per step), all projections
    W4A4;
  * expert at W4A16: the same 10 x 18 layers with group-128 int4 weights.
The same stack with bf16 weights through cuBLAS is timed after the step as
the 16-bit comparison.  Every input is seeded and synthetic; weights are
quantized before timing (offline preparation).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl vqlin|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica (the path has no exchange step); value = steps of all ranks / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "quantized linear µs, TOPS / HBM GB/s and % roofline per shape vs bf16 cuBLAS"
UNIT = "control_steps/s"
WORKLOAD = ("pi05_control_step: 18 Gemma-2B-style prefix layers on 816 tokens (q|k|v, gate|up W4A4, "
            "o, down W8A8, block Hadamard 128, dynamic per-token activations) + 10 denoising steps x 18 "
            "Gemma-300M-style expert layers on 50 tokens at W4A4 (static per-step scales) and again at "
            "W4A16 (group 128)")
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("vqlin", "reference"), default="vqlin")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-sample-rows", type=int, default=64,
                    help="prefix tokens per projection in the CPU-oracle sample")
    ap.add_argument("--shape", default=None,
                    help="time one kernel class alone instead of the control step: KIND,M,N,K with KIND in "
                         "act_quant4, act_quant8, act_quant_static4, linear_w4a4, linear_w4a4_static, linear_w8a8, linear_w4a8, "
                         "linear_w4a16, "
                         "linear_bf16 "
                         "(N is ignored for act_quant); prints a per-shape JSON line")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be at least 3")
    if a.steps < 1:
        ap.error("--steps must be at least 1")
    return a


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def job_time_ms(ms_local: float, world: int, device) -> float:
    """The job's timed region: the slowest rank's (all-reduce MAX over the process group)."""
    if world == 1:
        return ms_local
    import torch
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, steps: int, ms_total: float) -> float:
    """Whole-job throughput: every rank's steps over the slowest rank's time (weak scaling)."""
    return world * steps / (ms_total / 1e3)


# ----------------------------------------------------------------------------- peaks

def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- CPU oracle sample

def oracle_prepare(seed: int, rows_prefix: int):
    """Inputs and offline-quantized weights of the CPU-oracle sample (untimed)."""
    import numpy as np

    from oracle import vqlin_oracle as o
    from synth import activations, weights, workloads as wl

    pre = wl.WORKLOADS["prefix_w4a4_w8a8"]
    exp = wl.WORKLOADS["expert_w4a16"]
    step = wl.WORKLOADS["pi05_control_step"]

    def groups(family):
        out = {}
        for p in wl.layer_projections(family):
            out.setdefault(p.input, []).append(p)
        return out

    # ---- preparation (untimed)
    pre_groups = []
    for inp, projs in groups("gemma2b_prefix").items():
        K = projs[0].K
        bits = 8 if all(p.name in wl.W8A8_PROJECTIONS for p in projs) else 4
        W = np.concatenate([weights(p.N, K, std=pre["w_std"], seed=seed, tags=("cpu", "pre", p.name))
                            for p in projs])
        wt = o.quantize_weights_rtn(W, bits, True, 0, pre["hadamard_block"])
        X = activations(rows_prefix, K, dist=pre["act_dist"],
                        n_outliers=wl.n_outliers(K, pre["outlier_frac"]),
                        outlier_scale=pre["outlier_scale"], seed=seed, tags=("cpu", "pre", inp))
        pre_groups.append((X, bits, wt))
    exp_groups = []
    for inp, projs in groups("gemma300m_expert").items():
        K = projs[0].K
        W = np.concatenate([weights(p.N, K, std=exp["w_std"], spike_frac=exp["spike_frac"],
                                    spike_scale=exp["spike_scale"], seed=seed, tags=("cpu", "exp", p.name))
                            for p in projs])
        w4 = o.quantize_weights_rtn(W, 4, True, 0, step["hadamard_block"])
        w16 = o.quantize_weights_rtn(W, 4, False, exp["group_size"], 0)
        X = activations(exp["M"], K, seed=seed, tags=("cpu", "exp", inp))
        s_static = o.calibrate_static_scale([activations(exp["M"], K, seed=seed, tags=("cpu", "cal", inp, d))
                                             for d in range(2)], 4, step["hadamard_block"])
        exp_groups.append((X, w4, w16, s_static))
    return dict(pre_groups=pre_groups, exp_groups=exp_groups, rows=rows_prefix)


def oracle_run(prep):
    """Time the oracle on a bounded sample of one control step.

    Sample: one prefix layer (every distinct input, `rows` of its 816
    tokens) and one expert layer at 50 tokens for both expert variants.  The
    online work is timed (activation rotation + quantization, integer GEMM,
    epilogue; W4A16 dequantization + GEMM); weight quantization is offline
    preparation and not timed.  Returns (seconds per control step,
    extrapolated by tokens and layer counts; sample description; seconds of
    the sample itself).
    """
    from oracle import vqlin_oracle as o
    from synth import workloads as wl

    pre = wl.WORKLOADS["prefix_w4a4_w8a8"]
    exp = wl.WORKLOADS["expert_w4a16"]
    step = wl.WORKLOADS["pi05_control_step"]
    pre_groups, exp_groups, rows_prefix = prep["pre_groups"], prep["exp_groups"], prep["rows"]
    t0 = time.perf_counter()
    for X, bits, wt in pre_groups:
        xq, sx = o.act_hadamard_quant(X, bits, pre["hadamard_block"])
        o.linear_epilogue(o.int_gemm(xq, wt["q"]), sx, wt["s"])
    t1 = time.perf_counter()
    for X, w4, w16, s_static in exp_groups:
        xq, sx = o.act_hadamard_quant(X, 4, step["hadamard_block"], static_scale=s_static)
        o.linear_epilogue(o.int_gemm(xq, w4["q"]), sx, w4["s"])
    t2 = time.perf_counter()
    for X, w4, w16, s_static in exp_groups:
        o.linear_w4a16(X, w16["q"], w16["s"], w16["z"], exp["group_size"])
    t3 = time.perf_counter()

    per_step = ((t1 - t0) * (pre["M"] / rows_prefix) * pre["layers"]
                + ((t2 - t1) + (t3 - t2)) * exp["layers"] * step["steps"])
    sample = (f"one prefix layer at {rows_prefix} of 816 tokens (4 distinct inputs, 7 projections) + one "
              f"expert layer at 50 tokens for W4A4-static and W4A16; extrapolated linearly by tokens "
              f"(x{pre['M'] / rows_prefix:.0f}) and layers (x18 prefix, x180 expert); weight RTN untimed")
    return per_step, sample, t3 - t0


def blas_threads() -> int:
    try:
        import threadpoolctl
        n = sum(i.get("num_threads", 0) for i in threadpoolctl.threadpool_info() if i.get("user_api") == "blas")
        if n:
            return n
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0  # the CPU oracle arm runs on rank 0 only
    import numpy as np  # noqa: F401  (loads BLAS so its thread count is visible)

    times = []
    sample_desc = ""
    prep = oracle_prepare(args.seed, args.cpu_sample_rows)
    for i in range(args.warmup + args.steps):
        per_step, sample_desc, _ = oracle_run(prep)
        if i >= args.warmup:
            times.append(per_step)
    sec = sum(times) / len(times)
    value = 1.0 / sec
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (numpy oracle)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "timing": "host wall clock of the oracle on a bounded sample, "
                   "extrapolated to one control step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample_desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU stack

class ControlStepStack:
    """Device buffers, quantized weights and launch sequences of one control step."""

    def __init__(self, dev, seed: int, input_seed: int):
        import torch

        import bit_ptq_linear_vqlin_b300 as vq
        from synth import device as sd, workloads as wl

        self.torch, self.vq, self.dev = torch, vq, dev
        pre = wl.WORKLOADS["prefix_w4a4_w8a8"]
        exp = wl.WORKLOADS["expert_w4a16"]
        step = wl.WORKLOADS["pi05_control_step"]
        self.hb = step["hadamard_block"]
        self.group = exp["group_size"]
        self.n_steps, self.exp_layers, self.pre_layers = step["steps"], exp["layers"], pre["layers"]
        self.M_pre, self.M_exp = pre["M"], exp["M"]

        def groups(family):
            out = {}
            for p in wl.layer_projections(family):
                out.setdefault(p.input, []).append(p)
            return list(out.items())

        self.pre_groups = []   # per input: dict(K, N, bits, names)
        for inp, projs in groups("gemma2b_prefix"):
            bits = 8 if all(p.name in wl.W8A8_PROJECTIONS for p in projs) else 4
            self.pre_groups.append(dict(inp=inp, K=projs[0].K, N=sum(p.N for p in projs), bits=bits,
                                        names=[p.name for p in projs], Ns=[p.N for p in projs]))
        self.exp_groups = []
        for inp, projs in groups("gemma300m_expert"):
            self.exp_groups.append(dict(inp=inp, K=projs[0].K, N=sum(p.N for p in projs),
                                        names=[p.name for p in projs], Ns=[p.N for p in projs]))

        # ---- weights (bf16 kept for the cuBLAS comparison), quantized offline
        self.pre_w = []
        for l in range(self.pre_layers):
            layer = []
            for g in self.pre_groups:
                W = torch.cat([sd.weights(n, g["K"], std=pre["w_std"], seed=seed, tags=("pre", l, nm), device=dev)
                               for nm, n in zip(g["names"], g["Ns"])])
                q, s = vq.quantize_weights_rtn(W, g["bits"], True, 0, self.hb)
                layer.append(dict(W=W, q=q, s=s))
            self.pre_w.append(layer)
        self.exp_w = []
        for l in range(self.exp_layers):
            layer = []
            for g in self.exp_groups:
                W = torch.cat([sd.weights(n, g["K"], std=exp["w_std"], spike_frac=exp["spike_frac"],
                                          spike_scale=exp["spike_scale"], seed=seed, tags=("exp", l, nm),
                                          device=dev) for nm, n in zip(g["names"], g["Ns"])])
                q4, s4 = vq.quantize_weights_rtn(W, 4, True, 0, self.hb)
                q16, s16, z16 = vq.quantize_weights_rtn(W, 4, False, self.group, 0)
                layer.append(dict(W=W, q4=q4, s4=s4, q16=q16, s16=s16, z16=z16))
            self.exp_w.append(layer)

        # ---- activations: one seeded tensor per distinct input and layer (and step)
        self.pre_x = [[sd.activations(self.M_pre, g["K"], dist=pre["act_dist"],
                                      n_outliers=wl.n_outliers(g["K"], pre["outlier_frac"]),
                                      outlier_scale=pre["outlier_scale"], seed=input_seed,
                                      tags=("pre", l, g["inp"]), device=dev)
                       for g in self.pre_groups] for l in range(self.pre_layers)]
        self.exp_x = [[[sd.activations(self.M_exp, g["K"], seed=input_seed, tags=("exp", t, l, g["inp"]), device=dev)
                        for g in self.exp_groups] for l in range(self.exp_layers)] for t in range(self.n_steps)]

        # ---- static per-step scales: max over 8 calibration draws of the dynamic scale
        self.static = torch.zeros((self.n_steps, self.exp_layers, len(self.exp_groups)), dtype=torch.float32,
                                  device=dev)
        for t in range(self.n_steps):
            for l in range(self.exp_layers):
                for gi, g in enumerate(self.exp_groups):
                    best = torch.zeros((), dtype=torch.float32, device=dev)
                    for d in range(step["calib_draws"]):
                        xc = sd.activations(self.M_exp, g["K"], seed=seed + 1000003, tags=("cal", t, l, g["inp"], d),
                                            device=dev)
                        _, sc = vq.act_hadamard_quant(xc, 4, self.hb)
                        best = torch.maximum(best, sc.max())
                    self.static[t, l, gi] = best

        # ---- reusable code / scale / output buffers (one set per group shape)
        def codes(M, K, bits):
            # activation codes in the GEMM's operand encoding: a byte (int4) or a 16-bit word (int8) each
            return torch.empty((M, K), dtype=torch.uint8 if bits == 4 else torch.int16, device=dev)
        self.pre_buf = [dict(xq=codes(self.M_pre, g["K"], g["bits"]), sx=torch.empty(self.M_pre, device=dev),
                             y=torch.empty((self.M_pre, g["N"]), dtype=torch.bfloat16, device=dev))
                        for g in self.pre_groups]
        self.exp_buf = [dict(xq=codes(self.M_exp, g["K"], 4), sx=torch.empty(self.M_exp, device=dev),
                             y4=torch.empty((self.M_exp, g["N"]), dtype=torch.bfloat16, device=dev),
                             y16=torch.empty((self.M_exp, g["N"]), dtype=torch.bfloat16, device=dev))
                        for g in self.exp_groups]
        self.launches_per_step = 0
        self.instrument = None  # callable(key, fn) while capturing an instrumented graph

    # -- launch helpers -------------------------------------------------------
    def _go(self, key, fn):
        if self.instrument is None:
            fn()
        else:
            self.instrument(key, fn)
        self.launches_per_step += 1

    def prefix(self):
        vq = self.vq
        for l in range(self.pre_layers):
            for gi, g in enumerate(self.pre_groups):
                b, w, x = self.pre_buf[gi], self.pre_w[l][gi], self.pre_x[l][gi]
                # default arguments bind this iteration's tensors (the closures may run again later)
                self._go(("act_quant", g["bits"], self.M_pre, g["K"]),
                         lambda g=g, b=b, x=x: vq.act_hadamard_quant(x, g["bits"], self.hb, q_out=b["xq"],
                                                                     scale_out=b["sx"]))
                fn = vq.linear_w4a4 if g["bits"] == 4 else vq.linear_w8a8
                self._go((f"linear_w{g['bits']}a{g['bits']}", self.M_pre, g["N"], g["K"]),
                         lambda fn=fn, b=b, w=w: fn(b["xq"], b["sx"], w["q"], w["s"], out=b["y"]))

    def expert_w4a4(self):
        vq = self.vq
        for t in range(self.n_steps):
            for l in range(self.exp_layers):
                for gi, g in enumerate(self.exp_groups):
                    b, w, x = self.exp_buf[gi], self.exp_w[l][gi], self.exp_x[t][l][gi]
                    s = self.static[t, l, gi:gi + 1]
                    # one launch: the GEMM rotates and quantizes its activations on chip (once per
                    # cluster, the codes exchanged through xq) at the step's static scale
                    self._go(("linear_w4a4_static", self.M_exp, g["N"], g["K"]),
                             lambda b=b, w=w, x=x, s=s: vq.linear_w4a4_static(x, s, w["q4"], w["s4"], self.hb,
                                                                             out=b["y4"], xq_out=b["xq"]))

    def expert_w4a16(self):
        vq = self.vq
        for t in range(self.n_steps):
            for l in range(self.exp_layers):
                for gi, g in enumerate(self.exp_groups):
                    b, w, x = self.exp_buf[gi], self.exp_w[l][gi], self.exp_x[t][l][gi]
                    self._go(("linear_w4a16", self.M_exp, g["N"], g["K"]),
                             lambda b=b, w=w, x=x: vq.linear_w4a16(x, w["q16"], w["s16"], w["z16"], self.group,
                                                                   out=b["y16"]))

    def prefix_bf16(self):
        for l in range(self.pre_layers):
            for gi, g in enumerate(self.pre_groups):
                self.vq.linear_bf16_ref(self.pre_x[l][gi], self.pre_w[l][gi]["W"], out=self.pre_buf[gi]["y"])

    def expert_bf16(self):
        for t in range(self.n_steps):
            for l in range(self.exp_layers):
                for gi, g in enumerate(self.exp_groups):
                    self.vq.linear_bf16_ref(self.exp_x[t][l][gi], self.exp_w[l][gi]["W"], out=self.exp_buf[gi]["y16"])

    # -- algorithmic work ------------------------------------------------------
    def work_of(self, key):
        """(flops, bytes) of one launch of a kernel class (formulas of the scope table)."""
        kind = key[0]
        if kind.startswith("act_quant"):
            bits, M, K = key[1], key[2], key[3]
            return 0, 2 * M * K + M * K * (1 if bits == 4 else 2) + 4 * M
        M, N, K = key[1], key[2], key[3]
        if kind == "linear_w4a4":
            return 2 * M * N * K, M * K + N * K // 2 + 4 * M + 4 * N + 2 * M * N
        if kind == "linear_w4a4_static":  # bf16 activations in, one scale
            return 2 * M * N * K, 2 * M * K + N * K // 2 + 4 + 4 * N + 2 * M * N
        if kind == "linear_w8a8":
            return 2 * M * N * K, 2 * M * K + N * K + 4 * M + 4 * N + 2 * M * N
        if kind == "linear_w4a8":
            return 2 * M * N * K, 2 * M * K + N * K // 2 + 4 * M + 4 * N + 2 * M * N
        if kind == "linear_w4a16":
            return 2 * M * N * K, 2 * M * K + N * K // 2 + 4 * N * K // self.group + 2 * M * N
        raise KeyError(key)


def capture(torch, fn):
    """Warm fn once on a side stream, then capture it into a CUDA graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        # raw samples (the JSON line carries their summary); VQLIN_CLOCKS_DIR keeps them
        out_dir = os.environ.get("VQLIN_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"vqlin_clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for ln in f:
                p = [x.strip() for x in ln.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, p[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm_sorted = sorted(sm)
        return {"sm_mhz": sm_sorted[len(sm) // 2], "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def read_traffic(kernel_key):
    """dram bytes per launch from the committed ncu summary, if it matches this kernel and source."""
    import hashlib
    try:
        lines = open(TRAFFIC_FILE).read().splitlines()
    except OSError:
        return None
    key = " ".join(str(k) for k in kernel_key)
    for ln in lines:
        if not ln.startswith("traffic "):
            continue
        fields = dict(kv.split("=", 1) for kv in ln[len("traffic "):].split(";") if "=" in kv)
        if fields.get("key") != key:
            continue
        src = os.path.join(ROOT, fields.get("source", ""))
        try:
            sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        except OSError:
            return None
        if sha != fields.get("sha"):
            return None  # the kernel changed since the counters were taken
        return float(fields["bytes"])
    return None


def run_vqlin(args):
    import torch

    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    stack = ControlStepStack(dev, seed=args.seed, input_seed=args.seed + 7919 * rank)
    torch.cuda.synchronize()

    def full_step():
        stack.prefix()
        stack.expert_w4a4()
        stack.expert_w4a16()

    # the step as three CUDA graphs (prefix, expert at W4A4, expert at W4A16)
    graphs = [capture(torch, part) for part in (stack.prefix, stack.expert_w4a4, stack.expert_w4a16)]
    stack.launches_per_step = 0
    full_step()  # count launches of one step (eager, untimed)
    torch.cuda.synchronize()
    launches_per_step = stack.launches_per_step

    def step():
        for g in graphs:
            g.replay()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # -- timed region
    import torch.cuda.nvtx as nvtx
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    nvtx.range_push("vqlin_timed")
    ev[0].record()
    for _ in range(args.steps):
        step()
    ev[1].record()
    nvtx.range_pop()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        torch.distributed.barrier()
    clock_info = clocks.stop()
    ms_total = job_time_ms(ev[0].elapsed_time(ev[1]), world, dev)
    ms_step = ms_total / args.steps
    value = job_value(world, args.steps, ms_total)

    # -- per kernel class: every launch of the class in one step (all layers,
    # so the weights rotate exactly as in the step), captured back to back in
    # one graph and timed with CUDA events on the launching stream; share =
    # launches x average duration.  (Event nodes between the step's own
    # launches would break the programmatic-dependent-launch overlap and add
    # launch latency to every bracket, so the classes are timed this way.)
    per_class_fns = {}

    def collect(key, fn):
        per_class_fns.setdefault(key, []).append(fn)
        fn()

    stack.instrument = collect
    full_step()
    stack.instrument = None
    torch.cuda.synchronize()
    per_class = {}
    for key, fns in per_class_fns.items():
        def run_class(fns=fns):
            for f in fns:
                f()
        gk = capture(torch, run_class)
        gk.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(3):
            gk.replay()
        b.record()
        torch.cuda.synchronize()
        avg = a.elapsed_time(b) / (3 * len(fns))
        per_class[key] = (avg * len(fns), len(fns), avg)
        del gk
    dom = max(per_class, key=lambda k: per_class[k][0])
    dom_avg_ms = per_class[dom][2]
    dom_launches = 3 * per_class[dom][1]

    # -- parts (separately timed after the main region, same graphs)
    part_ms = {}
    for name, g in zip(("prefix", "expert_w4a4", "expert_w4a16"), graphs):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(5):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        part_ms[name] = a.elapsed_time(b) / 5

    # -- bf16 cuBLAS comparison on the same shapes
    gb_pre = capture(torch, stack.prefix_bf16)
    gb_exp = capture(torch, stack.expert_bf16)
    bf16_ms = {}
    for name, g, reps in (("prefix", gb_pre, 5), ("expert", gb_exp, 5)):
        for _ in range(2):
            g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        bf16_ms[name] = a.elapsed_time(b) / reps
    bf16_ms["control_step (prefix + expert once)"] = bf16_ms["prefix"] + bf16_ms["expert"]
    del gb_pre, gb_exp

    # -- end to end: pinned host inputs in, the action chunk out, every step
    x_pre0 = stack.pre_x[0][0]
    x_exp0 = stack.exp_x[0][0][0]
    h_pre = torch.empty(x_pre0.shape, dtype=x_pre0.dtype, pin_memory=True).copy_(x_pre0.cpu())
    h_exp = torch.empty(x_exp0.shape, dtype=x_exp0.dtype, pin_memory=True).copy_(x_exp0.cpu())
    out4, out16 = stack.exp_buf[-1]["y4"], stack.exp_buf[-1]["y16"]
    h_out4 = torch.empty(out4.shape, dtype=out4.dtype, pin_memory=True)
    h_out16 = torch.empty(out16.shape, dtype=out16.dtype, pin_memory=True)
    e2e_steps = max(3, min(args.steps, 30))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        x_pre0.copy_(h_pre, non_blocking=True)
        x_exp0.copy_(h_exp, non_blocking=True)
        step()
        h_out4.copy_(out4, non_blocking=True)
        h_out16.copy_(out16, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    h2d = h_pre.numel() * 2 + h_exp.numel() * 2
    d2h = h_out4.numel() * 2 + h_out16.numel() * 2

    # -- roofline of the dominant kernel class
    peaks, peaks_src = load_peaks()
    flops, nbytes = stack.work_of(dom)
    if dom[0].startswith("act_quant") or dom[0] == "linear_w4a16" or dom[1] <= 64:
        bound, achieved, peak, unit = "hbm", nbytes / (dom_avg_ms / 1e3) / 1e9, peaks["hbm_gbs"], "GB/s"
        peak_note = f"hbm_gbs ({peaks_src})"
    elif dom[0] in ("linear_w4a4", "linear_w4a4_static"):
        bound, unit = "tensor", "TFLOP/s"
        achieved = flops / (dom_avg_ms / 1e3) / 1e12
        peak = 2.0 * peaks["bf16_tflops"]
        peak_note = (f"dense fp8 rate = 2 x bf16_tflops ({peaks_src}, burst: the class is timed alone); the "
                     "int4 codes run on kind::f8f6f4 (e4m3) MMAs")
    else:
        bound, unit = "tensor", "TFLOP/s"
        achieved = flops / (dom_avg_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
        peak_note = (f"dense f16 rate = bf16_tflops ({peaks_src}, burst: the class is timed alone); the int8 "
                     "codes run on kind::f16 MMAs")
    traffic = read_traffic(dom)

    # -- CPU oracle baseline (rank 0 only)
    cpu = None
    if rank == 0:
        prep = oracle_prepare(args.seed, args.cpu_sample_rows)
        runs = [oracle_run(prep) for _ in range(3)]
        per_step = sum(r[0] for r in runs) / len(runs)
        sample, sample_s = runs[0][1], sum(r[2] for r in runs)
        cpu = {"value": 1.0 / per_step, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
               "sample": sample + f" ({sample_s:.1f} s of host time)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "s4/s8 codes (int32-exact sums) + bf16 x u4 (f32 accumulate)",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": "inputs larger than L2: each step streams "
                       f"{stack_bytes(stack) / 1e9:.2f} GB of distinct weights", "graphs": "CUDA graphs per part",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": " ".join(str(k) for k in dom), "avg_launch_ms": dom_avg_ms,
                         "launches_timed": dom_launches, "peak_source": peak_note,
                         "timing": "CUDA events around a graph of every launch of the class in one step "
                                   "(all layers), replayed 3 times",
                         "algorithmic": {"flops": flops, "bytes": nbytes}},
            "cpu_baseline": cpu,
            "e2e": {"value": world / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clock_info,
            "parts_ms": part_ms,
            "bf16_cublas_ms": bf16_ms,
            "kernel_share_ms_per_step": {" ".join(str(x) for x in k): round(v[0], 4)
                                         for k, v in sorted(per_class.items(), key=lambda kv: -kv[1][0])},
            "kernel_us_per_launch": {" ".join(str(x) for x in k): round(v[2] * 1e3, 2)
                                     for k, v in sorted(per_class.items(), key=lambda kv: -kv[1][0])},
            "wall_s_timed": t_wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def stack_bytes(stack):
    total = 0
    for layer in stack.pre_w:
        for w in layer:
            total += w["q"].numel() * w["q"].element_size() + w["s"].numel() * 4
    for layer in stack.exp_w:
        for w in layer:
            total += stack.n_steps * (w["q4"].numel() + w["q16"].numel() + 2 * w["s16"].numel() * 2)
    return total


def run_shape(args):
    """Time one kernel class at one shape, inputs rotated through more than 2x L2."""
    import torch

    import bit_ptq_linear_vqlin_b300 as vq

    kind, M, N, K = args.shape.split(",")
    M, N, K = int(M), int(N), int(K)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(args.seed)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def rand_bf16(r, c):
        return torch.randn((r, c), generator=g, device=dev).to(torch.bfloat16)

    def rand_codes(r, c, bits):
        # weight codes: every byte is a valid sign-magnitude code (a negative zero reads as 0)
        return torch.randint(0, 256, (r, c // 2 if bits == 4 else c), generator=g, device=dev,
                             dtype=torch.int32).to(torch.uint8)

    def rand_act_codes(r, c, bits):
        # activation codes in the operand encoding: sign bit + magnitude <= qmax
        qmax = 7 if bits == 4 else 127
        mag = torch.randint(0, qmax + 1, (r, c), generator=g, device=dev, dtype=torch.int32)
        sgn = torch.randint(0, 2, (r, c), generator=g, device=dev, dtype=torch.int32)
        if bits == 4:
            return (mag | (sgn << 7)).to(torch.uint8)
        return (mag | (sgn << 15)).to(torch.int16)

    group = 128
    if kind.startswith("act_quant"):
        # act_quant4 / act_quant8: dynamic per-token scales; act_quant_static4: one static scale
        bits = int(kind[-1])
        per = 2 * M * K
        flops, nbytes = 0, 2 * M * K + M * K * (1 if bits == 4 else 2) + 4 * M
        mk = lambda: dict(X=rand_bf16(M, K))  # noqa: E731
        q = torch.empty((M, K), dtype=torch.uint8 if bits == 4 else torch.int16, device=dev)
        sx = torch.empty(M, device=dev)
        st = torch.full((1,), 0.5, device=dev) if kind.startswith("act_quant_static") else None
        run = lambda d: vq.act_hadamard_quant(d["X"], bits, 128, static_scale=st, q_out=q, scale_out=sx)  # noqa: E731
    elif kind in ("linear_w4a4", "linear_w8a8", "linear_w4a8"):
        bits = 4 if kind == "linear_w4a4" else 8  # activation bits
        wbits = 8 if kind == "linear_w8a8" else 4
        kb = K // 2 if wbits == 4 else K          # packed weight bytes per row
        xb = K if bits == 4 else 2 * K            # activation operand bytes per token
        per = N * kb
        flops, nbytes = 2 * M * N * K, M * xb + N * kb + 4 * M + 4 * N + 2 * M * N
        xq = rand_act_codes(M, K, bits)
        sx = torch.rand(M, generator=g, device=dev)
        mk = lambda: dict(wq=rand_codes(N, K, wbits), sw=torch.rand(N, generator=g, device=dev))  # noqa: E731
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fn = {"linear_w4a4": vq.linear_w4a4, "linear_w8a8": vq.linear_w8a8, "linear_w4a8": vq.linear_w4a8}[kind]
        run = lambda d: fn(xq, sx, d["wq"], d["sw"], out=y)  # noqa: E731
    elif kind == "linear_w4a4_static":
        per = N * K // 2
        flops, nbytes = 2 * M * N * K, 2 * M * K + N * K // 2 + 4 + 4 * N + 2 * M * N
        X = rand_bf16(M, K)
        st = torch.full((1,), 0.5, device=dev)
        mk = lambda: dict(wq=rand_codes(N, K, 4), sw=torch.rand(N, generator=g, device=dev))  # noqa: E731
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
        run = lambda d: vq.linear_w4a4_static(X, st, d["wq"], d["sw"], 128, out=y, xq_out=xq)  # noqa: E731
    elif kind == "linear_w4a16":
        per = N * K // 2
        flops, nbytes = 2 * M * N * K, 2 * M * K + N * K // 2 + 4 * N * K // group + 2 * M * N
        X = rand_bf16(M, K)

        def mk():
            q, s, z = vq.quantize_weights_rtn(rand_bf16(N, K), 4, False, group, 0)
            return dict(q=q, s=s, z=z)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        run = lambda d: vq.linear_w4a16(X, d["q"], d["s"], d["z"], group, out=y)  # noqa: E731
    elif kind == "linear_bf16":
        per = 2 * N * K
        flops, nbytes = 2 * M * N * K, 2 * M * K + 2 * N * K + 2 * M * N
        X = rand_bf16(M, K)
        mk = lambda: dict(W=rand_bf16(N, K))  # noqa: E731
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        run = lambda d: vq.linear_bf16_ref(X, d["W"], out=y)  # noqa: E731
    else:
        raise SystemExit(f"unknown kernel class {kind}")

    copies = max(2, min(64, -(-2 * l2 // max(per, 1))))
    data = [mk() for _ in range(copies)]

    def body():
        for d in data:
            run(d)
    graph = capture(torch, body)
    for _ in range(args.warmup):
        graph.replay()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(args.steps):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / (args.steps * copies)
    peaks, src = load_peaks()
    line = {"mode": "shape", "kernel": kind, "M": M, "N": N, "K": K, "us": us,
            "TOPS": flops / us / 1e6 if flops else None, "GBs": nbytes / us / 1e3,
            "hbm_frac": nbytes / us / 1e3 / peaks["hbm_gbs"],
            "tensor_frac_fp8": (flops / us / 1e6) / (2 * peaks["bf16_tflops"]) if flops else None,
            "rotating_copies": copies, "launches": args.steps * copies, "peaks": src}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.shape:
        return run_shape(args)
    return run_vqlin(args)


if __name__ == "__main__":
    sys.exit(main())
