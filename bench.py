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
    ap.add_argument("--skip-shapes", action="store_true",
                    help="leave out the per-shape lines (configs 1-4) after the control step")
    ap.add_argument("--skip-cpu", action="store_true",
                    help="leave out the CPU-oracle leg (cpu_baseline null), e.g. for profiler runs")
    ap.add_argument("--shape", default=None,
                    help="time one kernel class alone instead of the control step: KIND,M,N,K with KIND in "
                         "act_quant4, act_quant8, act_quant_static4, act_composite4, act_composite8, linear_w4a4, "
                         "linear_w4a4_static, linear_w8a8, linear_w4a8, "
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


def oracle_single_thread(seed: int, rows: int):
    """The same oracle sample on one host thread: a child process whose BLAS
    pools are limited to one thread before numpy loads (no GPU use)."""
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[var] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "p = bench.oracle_prepare(%d, %d); r = bench.oracle_run(p); "
            "print(json.dumps({'per_step': r[0], 'sample_s': r[2], 'threads': bench.blas_threads()}))"
            % (ROOT, seed, rows))
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        d = json.loads(out.stdout.strip().splitlines()[-1])
    except (OSError, ValueError, IndexError, subprocess.TimeoutExpired):
        return None
    return {"value": 1.0 / d["per_step"], "unit": UNIT, "cores": d["threads"], "sample_s": d["sample_s"]}


def oracle_tie_fraction(prep, vq, torch, dev):
    """Activation codes of the GPU kernel against the oracle's on the sample's
    inputs: the fraction that differ, and whether every difference sits within
    1e-4 of a rounding tie of the exactly rotated value (the only place the two
    may differ: the kernel rotates in float32, the oracle in float64)."""
    import numpy as np

    from oracle import vqlin_oracle as o
    from synth import workloads as wl

    hb = wl.WORKLOADS["prefix_w4a4_w8a8"]["hadamard_block"]
    total = bad_n = 0
    all_at_ties = True
    cases = [(X, bits, None) for X, bits, _ in prep["pre_groups"]]
    cases += [(X, 4, s_static) for X, _, _, s_static in prep["exp_groups"]]
    for X, bits, st in cases:
        q_ref, s_ref = o.act_hadamard_quant(X, bits, hb, st)
        Xd = torch.from_numpy(np.ascontiguousarray(X).view(np.int16)).to(dev).view(torch.bfloat16)
        std = None if st is None else torch.tensor([st], dtype=torch.float32, device=dev)
        q, _ = vq.act_hadamard_quant(Xd, bits, hb, static_scale=std)
        qn = q.cpu().numpy()
        q_gpu = o.decode_act_int4(qn) if bits == 4 else o.decode_act_int8(qn.view(np.uint16))
        diff = np.nonzero(q_gpu.astype(np.int64) - q_ref.astype(np.int64))
        if diff[0].size:
            safe = np.where(s_ref > 0, s_ref, 1).astype(np.float64)
            exact = o.rotated_f64(X, hb) / (safe[:, None] if np.ndim(safe) else safe)
            frac = np.abs(exact[diff] - np.floor(exact[diff]) - 0.5)
            all_at_ties = all_at_ties and bool(np.all(frac < 1e-4))
        total += q_ref.size
        bad_n += diff[0].size
    return {"fraction": bad_n / max(total, 1), "codes_compared": total, "mismatches": bad_n,
            "all_within_1e-4_of_a_tie": all_at_ties,
            "inputs": "the CPU sample's activations: prefix (4 inputs, dynamic scales) and expert (static scales)"}


def blas_threads() -> int:
    """Threads of the BLAS pool numpy uses: threadpoolctl's count where it is
    installed, else the pool size the environment requests, else the cores."""
    try:
        import threadpoolctl
        n = sum(i.get("num_threads", 0) for i in threadpoolctl.threadpool_info() if i.get("user_api") == "blas")
        if n:
            return n
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0  # the CPU oracle arm runs on rank 0 only
    import numpy as np  # noqa: F401  (loads BLAS so its thread count is visible)

    times, samples = [], []
    sample_desc = ""
    prep = oracle_prepare(args.seed, args.cpu_sample_rows)
    t_region = 0.0
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        per_step, sample_desc, sample_s = oracle_run(prep)
        if i >= args.warmup:
            t_region += time.perf_counter() - t0
            times.append(per_step)
            samples.append(sample_s)
    sec = sum(times) / len(times)
    value = 1.0 / sec
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_region / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (numpy oracle)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "timing": "host wall clock of the oracle: each step is one bounded "
                   "sample (ms_per_step is its real time); value extrapolates the sample to whole control "
                   "steps by tokens and layers",
                   "extrapolated_ms_per_control_step": sec * 1e3},
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
        self.instrument = None  # callable(key, fn) while capturing an instrumented graph

    # -- launch helpers -------------------------------------------------------
    def _go(self, key, fn):
        if self.instrument is None:
            fn()
        else:
            self.instrument(key, fn)

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
        """(flops, bytes) of one launch of a kernel class, bytes by the scope
        table's formulas (int4 codes half a byte, int8 codes one byte)."""
        kind = key[0]
        if kind.startswith("act_quant"):
            bits, M, K = key[1], key[2], key[3]
            return 0, alg_bytes(f"act_quant{bits}", M, 0, K)
        M, N, K = key[1], key[2], key[3]
        return 2 * M * N * K, alg_bytes(kind, M, N, K, self.group)


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
        # a class of two kernels (activation kernel + codes GEMM) lists both sources
        srcs = fields.get("source", "").split(",")
        shas = fields.get("sha", "").split(",")
        if len(srcs) != len(shas):
            return None
        for src, want in zip(srcs, shas):
            try:
                sha = hashlib.sha256(open(os.path.join(ROOT, src), "rb").read()).hexdigest()[:16]
            except OSError:
                return None
            if sha != want:
                return None  # a kernel changed since the counters were taken
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
    # count the library's kernel launches of one step (eager, untimed); a call
    # may launch more than one kernel (activation kernel + codes GEMM)
    n0 = stack.vq.kernel_launch_count()
    full_step()
    torch.cuda.synchronize()
    launches_per_step = stack.vq.kernel_launch_count() - n0
    # launches the GPU ran before the first warm-up step (the captures recorded
    # one step's worth without running it): the skip count of a launch list
    print(f"library kernel launches run before the first warm-up step: "
          f"{stack.vq.kernel_launch_count() - launches_per_step}", file=sys.stderr)

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

    # -- tensor-core peaks: the library's own rate kernels for the MMA kinds used
    peaks, peaks_src = load_peaks()
    own = measure_tensor_peaks(stack.vq)

    # -- roofline of the dominant kernel class
    flops, nbytes = stack.work_of(dom)
    kind_peak = "e4m3" if dom[0] in ("linear_w4a4", "linear_w4a4_static") else "bf16"
    rl = roofline_of(flops, nbytes, dom_avg_ms * 1e3, own[kind_peak]["tflops"], peaks["hbm_gbs"])
    if rl["bound"] == "hbm":
        bound, achieved, peak, unit = "hbm", nbytes / (dom_avg_ms / 1e3) / 1e9, peaks["hbm_gbs"], "GB/s"
        peak_note = f"hbm_gbs of MEASURED_PEAKS.json ({peaks_src}, a STREAM-style copy)"
    else:
        bound, unit = "tensor", "TFLOP/s"
        achieved = flops / (dom_avg_ms / 1e3) / 1e12
        peak = own[kind_peak]["tflops"]
        peak_note = (f"the library's own dense tcgen05 rate for the MMA kind this kernel issues "
                     f"({'kind::f8f6f4 e4m3' if kind_peak == 'e4m3' else 'kind::f16 bf16'}), measured in this run")
    traffic = read_traffic(dom)

    # -- fixed cost of a dependent launch per kernel class (rank 0)
    floor = launch_floor(torch, stack.vq, dev) if rank == 0 and not args.skip_shapes else None

    # -- per-shape lines of configs 1-4 (rank 0)
    shapes = None
    if rank == 0 and not args.skip_shapes:
        shapes = per_shape_lines(torch, stack.vq, dev, args.seed, own, peaks["hbm_gbs"])

    # -- CPU oracle baseline (rank 0 only): all cores and one thread
    cpu = None
    if rank == 0 and not args.skip_cpu:
        prep = oracle_prepare(args.seed, args.cpu_sample_rows)
        runs = [oracle_run(prep) for _ in range(3)]
        per_step = sum(r[0] for r in runs) / len(runs)
        sample, sample_s = runs[0][1], sum(r[2] for r in runs)
        single = oracle_single_thread(args.seed, args.cpu_sample_rows)
        cpu = {"value": 1.0 / per_step, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
               "sample": sample + f" ({sample_s:.1f} s of host time over 3 runs)", "single_thread": single,
               "activation_tie_fraction": oracle_tie_fraction(prep, stack.vq, torch, dev)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "s4/s8 codes (int32-exact sums) + bf16 x u4 (f32 accumulate)",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": "inputs larger than L2: "
                       f"{stack_bytes(stack)[0] / 1e9:.2f} GB of distinct quantized weights (prefix 18 layers, "
                       "expert 18 layers at W4A4 and W4A16); each step reads "
                       f"{stack_bytes(stack)[1] / 1e9:.2f} GB of them, the expert's layers once per denoising "
                       "step (their 0.15 GB per precision does not stay in the 126 MB L2)",
                       "graphs": "CUDA graphs per part", "parallelism": f"replicas x{world}"},
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                         "frac": achieved / peak, "traffic": traffic,
                         "bytes_formula": "scope table: int4 codes MK/2, int8 codes MK",
                         "kernel": " ".join(str(k) for k in dom), "avg_launch_ms": dom_avg_ms,
                         "launches_timed": dom_launches, "peak_source": peak_note,
                         "timing": "CUDA events around a graph of every launch of the class in one step "
                                   "(all layers), replayed 3 times",
                         "algorithmic": {"flops": flops, "bytes": nbytes}},
            "cpu_baseline": cpu,
            "e2e": {"value": world / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clock_info,
            "launch_floor_us": floor,
            "parts_ms": part_ms,
            "bf16_cublas_ms": bf16_ms,
            "kernel_share_ms_per_step": {" ".join(str(x) for x in k): round(v[0], 4)
                                         for k, v in sorted(per_class.items(), key=lambda kv: -kv[1][0])},
            "kernel_us_per_launch": {" ".join(str(x) for x in k): round(v[2] * 1e3, 2)
                                     for k, v in sorted(per_class.items(), key=lambda kv: -kv[1][0])},
            "wall_s_timed": t_wall,
            "peaks": {"hbm_gbs": peaks["hbm_gbs"], "cublas_bf16_tflops": peaks["bf16_tflops"],
                      "source": peaks_src, "tcgen05_e4m3_tflops": own["e4m3"]["tflops"],
                      "tcgen05_bf16_tflops": own["bf16"]["tflops"], "tcgen05_how": own["bf16"]["how"],
                      "int8_note": "kind::i8 does not assemble for sm_103a: int4 codes run exactly on "
                                   "kind::f8f6f4 (e4m3), int8 codes on kind::f16; those rates are the "
                                   "int-class peaks used"},
            "per_shape": shapes,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def stack_bytes(stack):
    """(distinct quantized weight bytes, weight bytes one control step reads):
    the 18 expert layers are shared by the 10 denoising steps, read once per
    step each."""
    pre = exp = 0
    for layer in stack.pre_w:
        for w in layer:
            pre += w["q"].numel() * w["q"].element_size() + w["s"].numel() * 4
    for layer in stack.exp_w:
        for w in layer:
            exp += (w["q4"].numel() + w["s4"].numel() * 4 + w["q16"].numel() + 2 * w["s16"].numel() * 2)
    return pre + exp, pre + stack.n_steps * exp


# ----------------------------------------------------------------------------- per-shape lines

# Algorithmic bytes of one call (the scope table's formulas): int4 codes count
# half a byte each and int8 codes one byte, whatever the storage format.
def alg_bytes(kind, M, N, K, group=128):
    if kind == "act_quant4":
        return 2 * M * K + M * K // 2 + 4 * M
    if kind == "act_quant8":
        return 2 * M * K + M * K + 4 * M
    if kind == "linear_w4a4":
        return M * K // 2 + N * K // 2 + 4 * M + 4 * N + 2 * M * N
    if kind == "linear_w8a8":
        return M * K + N * K + 4 * M + 4 * N + 2 * M * N
    if kind == "linear_w4a8":
        return M * K + N * K // 2 + 4 * M + 4 * N + 2 * M * N
    if kind == "linear_w4a4_static":  # bf16 activations in, one static scale
        return 2 * M * K + N * K // 2 + 4 + 4 * N + 2 * M * N
    if kind == "linear_w4a16":
        return 2 * M * K + N * K // 2 + 4 * N * K // group + 2 * M * N
    if kind == "linear_bf16":
        return 2 * M * K + 2 * N * K + 2 * M * N
    raise KeyError(kind)


# Bytes the library actually moves where its storage format differs: one byte
# per int4 activation code, a 16-bit word per int8 code.
def storage_bytes(kind, M, N, K, group=128):
    if kind == "act_quant4":
        return 2 * M * K + M * K + 4 * M
    if kind == "act_quant8":
        return 2 * M * K + 2 * M * K + 4 * M
    if kind == "linear_w4a4":
        return M * K + N * K // 2 + 4 * M + 4 * N + 2 * M * N
    if kind in ("linear_w8a8", "linear_w4a8"):
        return 2 * M * K + (N * K if kind == "linear_w8a8" else N * K // 2) + 4 * M + 4 * N + 2 * M * N
    return alg_bytes(kind, M, N, K, group)


def roofline_of(flops, nbytes, us, tensor_peak_tflops, hbm_gbs):
    """Achieved rate against min(tensor peak, arithmetic intensity x HBM bandwidth)."""
    if us <= 0:
        return None
    gbs = nbytes / us / 1e3
    if not flops:
        return {"bound": "hbm", "frac": gbs / hbm_gbs}
    tops = flops / us / 1e6
    ridge = flops / nbytes * hbm_gbs / 1e3  # TFLOP/s the HBM roofline allows
    bound = "hbm" if ridge < tensor_peak_tflops else "tensor"
    return {"bound": bound, "frac": tops / min(ridge, tensor_peak_tflops)}


class ShapeTimer:
    """Times launch sequences of one shape: every launch reads its own weight
    copy (the copies together exceed 2x L2), captured in one CUDA graph and
    timed with CUDA events on the launching stream."""

    def __init__(self, torch, dev):
        self.torch, self.dev = torch, dev
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def copies_for(self, weight_bytes):
        return max(2, min(48, -(-2 * self.l2 // max(weight_bytes, 1))))

    def time(self, fns, reps=8):
        torch = self.torch

        def body():
            for f in fns:
                f()
        g = capture(torch, body)
        g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        del g
        return a.elapsed_time(b) * 1e3 / (reps * len(fns))


def per_shape_lines(torch, vq, dev, seed, tensor_peaks, hbm_gbs):
    """Per-shape lines of configs 1-4 (and the static-scale expert of config 5):
    µs, TOPS, GB/s and roofline fraction of each quantized projection (its
    activation quantization and GEMM also alone), next to cuBLAS bf16 on the
    same shape in the same process."""
    from synth import device as sd, workloads as wl

    T = ShapeTimer(torch, dev)
    lines = []
    c1, c2, c3, c4 = (wl.WORKLOADS[k] for k in ("single_w4a4_16x256", "expert_w4a16", "prefix_w4a4_w8a8",
                                                   "llama2_7b"))

    def wgen(N, K, std, tags, spike=(0.0, 1.0)):
        return sd.weights(N, K, std=std, spike_frac=spike[0], spike_scale=spike[1], seed=seed, tags=tags, device=dev)

    def entry(cfg, variant, M, N, K, parts, hb, note=None):
        """parts: list of (kind, us) making up the projection."""
        us = sum(u for _, u in parts)
        flops = 2 * M * N * K
        nbytes = sum(alg_bytes(k, M, N, K) for k, _ in parts)
        sbytes = sum(storage_bytes(k, M, N, K) for k, _ in parts)
        tp = tensor_peaks["e4m3" if variant in ("w4a4", "w4a4_static") else "bf16"]
        e = {"cfg": cfg, "variant": variant, "M": M, "N": N, "K": K, "hadamard_block": hb, "us": round(us, 3),
             "TOPS": round(flops / us / 1e6, 2), "GBs": round(nbytes / us / 1e3, 1),
             "alg_bytes": nbytes, "storage_bytes": sbytes,
             "roofline": roofline_of(flops, nbytes, us, tp["tflops"], hbm_gbs)}
        if len(parts) > 1:
            e["parts"] = {}
            for k, u in parts:
                fl = 0 if k.startswith("act_quant") else flops
                e["parts"][k] = {"us": round(u, 3),
                                 "GBs": round(alg_bytes(k, M, N, K) / u / 1e3, 1),
                                 "roofline": roofline_of(fl, alg_bytes(k, M, N, K), u, tp["tflops"], hbm_gbs)}
        if note:
            e["note"] = note
        return e

    def bf16_us(M, N, K, X, std, tags):
        Ws = [wgen(N, K, std, tags + ("bf16", i)) for i in range(T.copies_for(2 * N * K))]
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        us = T.time([lambda W=W: vq.linear_bf16_ref(X, W, out=y) for W in Ws])
        del Ws
        return us

    def quant_us(X, bits, hb, M, K):
        q = torch.empty((M, K), dtype=torch.uint8 if bits == 4 else torch.int16, device=dev)
        sx = torch.empty(M, device=dev)
        us = T.time([lambda: vq.act_hadamard_quant(X, bits, hb, q_out=q, scale_out=sx)] * 16)
        return us, q, sx

    def int_variant(variant, X, M, N, K, hb, std, tags, cublas):
        abits, wbits = {"w4a4": (4, 4), "w8a8": (8, 8), "w4a8": (8, 4)}[variant]
        qus, xq, sx = quant_us(X, abits, hb, M, K)
        n = T.copies_for(N * K // (2 if wbits == 4 else 1))
        ws = []
        for i in range(n):
            q, s_ = vq.quantize_weights_rtn(wgen(N, K, std, tags + (i,)), wbits, True, 0, hb)
            ws.append((q, s_))
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fn = {"w4a4": vq.linear_w4a4, "w8a8": vq.linear_w8a8, "w4a8": vq.linear_w4a8}[variant]
        gus = T.time([lambda q=q, s_=s_: fn(xq, sx, q, s_, out=y) for q, s_ in ws])
        # the projection as a user runs it: quantize, then the GEMM, per weight copy
        pus = T.time([lambda q=q, s_=s_: (vq.act_hadamard_quant(X, abits, hb, q_out=xq, scale_out=sx),
                                          fn(xq, sx, q, s_, out=y)) for q, s_ in ws])
        del ws
        kq = f"act_quant{abits}"
        e = entry(cfg_now[0], variant, M, N, K, [(kq, qus), (f"linear_{variant}", gus)], hb)
        e["projection_us"] = round(pus, 3)
        e["cublas_bf16_us"] = round(cublas, 3)
        e["speedup_vs_bf16"] = round(cublas / pus, 3)
        return e

    def w4a16_variant(X, M, N, K, std, tags, cublas, spike=(0.0, 1.0), group=128):
        n = T.copies_for(N * K // 2)
        ws = [vq.quantize_weights_rtn(wgen(N, K, std, tags + ("w16", i), spike), 4, False, group, 0) for i in range(n)]
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        us = T.time([lambda w=w: vq.linear_w4a16(X, w[0], w[1], w[2], group, out=y) for w in ws])
        del ws
        e = entry(cfg_now[0], "w4a16", M, N, K, [("linear_w4a16", us)], 0)
        e["projection_us"] = round(us, 3)
        e["cublas_bf16_us"] = round(cublas, 3)
        e["speedup_vs_bf16"] = round(cublas / us, 3)
        return e

    def static_variant(X, M, N, K, hb, std, tags, cublas, spike):
        n = T.copies_for(N * K // 2)
        ws = [vq.quantize_weights_rtn(wgen(N, K, std, tags + ("w4s", i), spike), 4, True, 0, hb) for i in range(n)]
        _, sc = vq.act_hadamard_quant(X, 4, hb)
        st = sc.max().reshape(1).contiguous()
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
        us = T.time([lambda w=w: vq.linear_w4a4_static(X, st, w[0], w[1], hb, out=y, xq_out=xq) for w in ws])
        del ws
        e = entry("5", "w4a4_static", M, N, K, [("linear_w4a4_static", us)], hb,
                  note="one launch: rotation, static-scale quantization and GEMM")
        e["projection_us"] = round(us, 3)
        e["cublas_bf16_us"] = round(cublas, 3)
        e["speedup_vs_bf16"] = round(cublas / us, 3)
        return e

    cfg_now = ["1"]
    # ---- config 1: one W4A4 linear, 16 x 256 -> 256, block Hadamard 64
    M, N, K = c1["M"], c1["N"], c1["K"]
    X = sd.activations(M, K, n_outliers=c1["n_outliers"], outlier_scale=c1["outlier_scale"], seed=seed,
                       tags=("shape1",), device=dev)
    cb = bf16_us(M, N, K, X, c1["w_std"], ("shape1",))
    e = int_variant("w4a4", X, M, N, K, c1["hadamard_block"], c1["w_std"], ("shape1",), cb)
    e["roofline"]["bound"] = "latency"
    e["note"] = "2.1 MOP and ~55 KB: launch latency bounds it, the fraction is not a target"
    lines.append(e)

    # ---- config 2 (W4A16) and the static-scale W4A4 expert of config 5, 50 tokens
    cfg_now[0] = "2"
    spike = (c2["spike_frac"], c2["spike_scale"])
    for name, N, K in (("q|k|v", 3072, 1024), ("o", 1024, 1024), ("gate|up", 8192, 1024), ("down", 1024, 4096)):
        M = c2["M"]
        X = sd.activations(M, K, seed=seed, tags=("shape2", name), device=dev)
        cb = bf16_us(M, N, K, X, c2["w_std"], ("shape2", name))
        e = w4a16_variant(X, M, N, K, c2["w_std"], ("shape2", name), cb, spike, c2["group_size"])
        e["projection"] = name
        lines.append(e)
        e = static_variant(X, M, N, K, 128, c2["w_std"], ("shape2", name), cb, spike)
        e["projection"] = name
        lines.append(e)

    # ---- config 3: prefix backbone, 816 tokens
    cfg_now[0] = "3"
    for name, N, K, variant in (("q|k|v", 2560, 2048, "w4a4"), ("o", 2048, 2048, "w8a8"),
                                ("gate|up", 32768, 2048, "w4a4"), ("down", 2048, 16384, "w8a8")):
        M = c3["M"]
        X = sd.activations(M, K, dist=c3["act_dist"], n_outliers=wl.n_outliers(K, c3["outlier_frac"]),
                           outlier_scale=c3["outlier_scale"], seed=seed, tags=("shape3", name), device=dev)
        cb = bf16_us(M, N, K, X, c3["w_std"], ("shape3", name))
        e = int_variant(variant, X, M, N, K, c3["hadamard_block"], c3["w_std"], ("shape3", name), cb)
        e["projection"] = name
        lines.append(e)

    # ---- config 4: Llama-2-7B-shaped projections at M in {1, 64, 512}
    cfg_now[0] = "4"
    for M in c4["Ms"]:
        for name, N, K in (("q/k/v/o", 4096, 4096), ("gate/up", 11008, 4096), ("down", 4096, 11008)):
            X = sd.activations(M, K, n_outliers=wl.n_outliers(K, c4["outlier_frac"]),
                               outlier_scale=c4["outlier_scale"], seed=seed, tags=("shape4", M, name), device=dev)
            cb = bf16_us(M, N, K, X, c4["w_std"], ("shape4", M, name))
            for variant in ("w8a8", "w4a4", "w4a8"):
                e = int_variant(variant, X, M, N, K, c4["hadamard_block"], c4["w_std"], ("shape4", M, name), cb)
                e["projection"] = name
                lines.append(e)
            e = w4a16_variant(X, M, N, K, c4["w_std"], ("shape4", M, name), cb, group=c4["group_size"])
            e["projection"] = name
            lines.append(e)
            torch.cuda.empty_cache()
    return lines


def launch_floor(torch, vq, dev, n=180):
    """Per-launch time of n dependent launches of the smallest case of each
    kernel class (one CUDA graph, programmatic dependent launch as in the
    step): the fixed cost a few-token projection pays before its own work."""
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    T = ShapeTimer(torch, dev)

    def bf16(r, c):
        return torch.randn((r, c), generator=g, device=dev).to(torch.bfloat16)

    M, N, K = 16, 128, 128
    X, Xs, W = bf16(M, K), bf16(1, K), bf16(N, K)
    wq, sw = vq.quantize_weights_rtn(W, 4, True, 0, 128)
    q16, s16, z16 = vq.quantize_weights_rtn(W, 4, False, 128, 0)
    st = torch.full((1,), 0.5, device=dev)
    xq1 = torch.empty((1, K), dtype=torch.uint8, device=dev)
    sx1 = torch.empty(1, device=dev)
    xq, sx = vq.act_hadamard_quant(X, 4, 128)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    xqs = torch.empty((M, K), dtype=torch.uint8, device=dev)
    cases = {
        "act_quant 1x128": lambda: vq.act_hadamard_quant(Xs, 4, 128, q_out=xq1, scale_out=sx1),
        "linear_w4a4 16x128x128 (codes)": lambda: vq.linear_w4a4(xq, sx, wq, sw, out=y),
        "linear_w4a4_static 16x128x128 (one launch)":
            lambda: vq.linear_w4a4_static(X, st, wq, sw, 128, out=y, xq_out=xqs),
        "linear_w4a16 16x128x128": lambda: vq.linear_w4a16(X, q16, s16, z16, 128, out=y),
        "cuBLAS bf16 16x128x128": lambda: vq.linear_bf16_ref(X, W, out=y),
    }
    return {k: round(min(T.time([f] * n, reps=4) for _ in range(3)), 3) for k, f in cases.items()}


def measure_tensor_peaks(vq):
    """The library's own dense tcgen05 rate for the two MMA kinds the GEMMs
    issue: 148 CTAs, N = 256, four issuing warps with an accumulator each."""
    out = {}
    for kind in ("e4m3", "bf16"):
        best = 0.0
        for _ in range(3):
            tf, _ = vq.measure_mma_rate(kind, 256, a_in_tmem=False, accumulators=1, issuers=1, iters=8192)
            tf4, _ = vq.measure_mma_rate(kind, 64, a_in_tmem=False, accumulators=4, issuers=4, iters=8192)
            best = max(best, tf, tf4)
        out[kind] = {"tflops": best, "how": "vqlin_measure_mma_rate: one CTA per SM, operands on chip, "
                     "best of one issuer at N=256 and four issuers at N=64, 3 tries"}
    return out


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
    if kind.startswith("act_composite"):
        # composite SVD.Hadamard rotation (block 128) of activations: P and R_j
        # prepared offline from a K x K weight, then rotated and quantized
        bits = int(kind[-1])
        per = 2 * M * K
        flops, nbytes = 2 * M * K * 128, 2 * M * K + M * K * (1 if bits == 4 else 2) + 4 * M
        perm, R = vq.composite_rotation_prepare(rand_bf16(K, K), 128)
        mk = lambda: dict(X=rand_bf16(M, K))  # noqa: E731
        q = torch.empty((M, K), dtype=torch.uint8 if bits == 4 else torch.int16, device=dev)
        sx = torch.empty(M, device=dev)
        run = lambda d: vq.act_composite_quant(d["X"], bits, 128, perm, R, q_out=q, scale_out=sx)  # noqa: E731
    elif kind.startswith("act_quant"):
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

    # algorithmic bytes of the scope table (int4 codes MK/2, int8 codes MK)
    nbytes = alg_bytes(("act_quant" + kind[-1]) if kind.startswith("act_") else kind, M, N, K, group)
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
