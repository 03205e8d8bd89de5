#!/usr/bin/env python
"""Benchmark of the block-stack hot path on GB300: forward + backward tokens/s.

One step = zero the gradient buffers, xt_block_fwd, xt_block_bwd on one batch of synthetic
tokens (every op of the stack: embedding, norms, QKV / projection / MLP GEMMs, the fused causal
attention, RoPE when configured, dropout-residual adds, tied logits, cross-entropy and all
backward kernels).  Default workload: the 12-layer GPT-style stack (B 8, S 1024, d 768,
12 heads × 64, LayerNorm, exact-GELU MLP 3072, learned positions, tied 50304-vocab output,
bf16 storage with fp32 accumulation, fp32 parameter gradients).

Prints one JSON line.  --impl reference times the CPU oracle (float64 NumPy) on a bounded
sample of the same workload instead.  Under torchrun each rank runs its own replica on its
own GPU and its own batch (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block fwd+bwd tokens/s on 1 GB300; per-kernel HBM GB/s and GEMM TFLOP/s vs peak"

WORKLOAD_TEXT = {
    "gpt12": "12-layer pre-norm GPT stack: B8 S1024 d768 H12x64, LayerNorm, exact-GELU MLP 3072, learned "
             "positions, tied 50304-vocab logits + mean CE, causal fused attention (tcgen05, probabilities never "
             "stored), bf16 storage, fp32 accumulate / statistics / parameter grads",
    "block256": "1 pre-norm block: B4 S256 d256 H4x64, RMSNorm, RoPE, SwiGLU 688, tied 4096-vocab logits + mean CE, "
                "causal composed attention, residual dropout p=0.1, fp32 storage, tf32 tensor-core GEMMs",
    "tiny": "1 pre-norm block: B1 S16 d32 H2x16, RMSNorm, RoPE, SwiGLU 64, tied 64-vocab logits, fp32",
}


# The reference arm runs the float64 oracle (composed attention: probabilities formed and kept)
# on a causal prefix of one sequence; its label says so.
REFERENCE_TEXT = {
    "gpt12": "float64 NumPy oracle of the 12-layer pre-norm GPT stack (d768 H12x64, LayerNorm, exact-GELU MLP 3072, "
             "learned positions, tied 50304-vocab logits + mean CE), composed causal attention "
             "(softmax(QK^T/sqrt(hd)) kept, then @V), on the first {n} positions of one sequence per step",
    "block256": "float64 NumPy oracle of 1 pre-norm block (d256 H4x64, RMSNorm, RoPE, SwiGLU 688, tied 4096-vocab "
                "logits + mean CE, residual dropout p=0.1), composed causal attention, on the first {n} positions "
                "of one sequence per step",
    "tiny": "float64 NumPy oracle of 1 pre-norm block (d32 H2x16, RMSNorm, RoPE, SwiGLU 64, tied 64-vocab logits), "
            "composed causal attention, on the first {n} positions of one sequence per step",
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=120)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOAD_TEXT), default="gpt12")
    ap.add_argument("--recompute", action="store_true",
                    help="activation recompute: keep each layer's input only, redo its forward in the backward")
    ap.add_argument("--kernel", choices=["attention", "gemm", "layernorm", "gelu", "cross_entropy", "adamw", "fp8gemm",
                                         "ce_fanout"],
                    default=None,
                    help="time one kernel family at the workload's sizes instead of the step (for profiling)")
    ap.add_argument("--sweep", action="store_true",
                    help="per-kernel HBM GB/s of the memory-bound ops (rows 8192 x cols 768..8192, fp32 and bf16) "
                         "and of the 8192 x 128256 cross-entropy / fan-out case; one JSON line per case")
    ap.add_argument("--shape", default="8192,3072,768,0,1",
                    help="--kernel gemm: M,N,K,trans_a,trans_b (bf16 operands and output)")
    ap.add_argument("--rows", type=int, default=0,
                    help="--kernel ce_fanout: logits rows (default: the 8192 of the large-vocabulary case)")
    ap.add_argument("--pairing", type=int, choices=[0, 1, 2], default=0,
                    help="--kernel gemm: 0 model's choice, 1 single-CTA kernel only, 2 paired-CTA kernel")
    ap.add_argument("--schedule", type=int, choices=[0, 1, 2, 3, 4], default=0,
                    help="--kernel gemm: schedule override (0 model, 1 tiles, 2 K split, 3 stream-K, 4 lockstep)")
    ap.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
    # profiling runs of the step only: leave out the composed-attention pass and the oracle baseline
    ap.add_argument("--step-only", action="store_true", help=argparse.SUPPRESS)
    # two of the 8 sequences: ≈ 11 s of float64 oracle work on 16 Arm cores
    ap.add_argument("--sample-seqs", type=int, default=2, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ------------------------------------------------------------------------------ CPU oracle


def oracle_sample(workload: str, seqs: int, reps: int = 1, prefix: int = 0):
    """Times the oracle's forward + backward on `seqs` sequences of the workload (float64
    NumPy, all host cores), or, with `prefix` > 0, on the first `prefix` positions of one
    sequence (the same stack on a shorter causal sequence).  Returns (tokens/s, seconds per
    rep, tokens)."""
    import synth
    from oracle import block as OB
    cfg = dict(synth.BLOCK_CONFIGS[workload])
    params = synth.block_params(cfg)
    ids, tgt = synth.block_tokens(cfg)
    if prefix and prefix < cfg["S"]:
        sub = dict(cfg, B=1, S=prefix)
        if "P" in params:
            params = dict(params, P=params["P"][:prefix])
        n = prefix
    else:
        seqs = min(seqs, cfg["B"])
        sub = dict(cfg, B=seqs)
        n = seqs * cfg["S"]
    times = []
    for r in range(reps):
        t0 = time.perf_counter()
        OB.forward_backward(sub, params, ids[:n], tgt[:n], synth.BASE_SEED_DROPOUT + r, training=True)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    return n / t, t, n


def cpu_baseline(workload: str, seqs: int):
    """Runs the oracle sample in a fresh process (no CUDA state shared) and parses its line."""
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", "--workload", workload,
           "--sample-seqs", str(seqs)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=1800)
    if r.returncode != 0:
        return {"value": None, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                "sample": f"failed: {r.stderr.strip()[-200:]}"}
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def max_over_ranks(x: float, device=None) -> float:
    """The maximum of `x` over the ranks of the default process group (x itself with none)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "of measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "of fallback"


# ------------------------------------------------------------------------------ reference arm


REF_BUDGET_S = 150.0


def run_reference_sweep(args):
    """The oracle on the memory-bound op sweep and the large-vocabulary cross-entropy fan-out:
    each op's forward + backward on a row sample of each shape (float64 NumPy, this process's
    threads), reported as GB/s of the same algorithmic bytes the GPU sweep counts, scaled from
    the sample's rows to the shape's.  One JSON line per case."""
    import numpy as np
    import synth
    from oracle import dropout as OD
    from oracle import ops as O
    rng = np.random.default_rng(synth.SEED_SWEEP)
    sample = 64   # rows timed per shape

    def timed(fn, reps=3):
        best = float("inf")
        for _ in range(reps):
            t0 = time.perf_counter()
            fn()
            best = min(best, time.perf_counter() - t0)
        return best

    cores = os.environ.get("OPENBLAS_NUM_THREADS") or str(os.cpu_count())
    for dtn, e in (("f32", 4), ("bf16", 2)):
        for C in synth.SWEEP_COLS:
            x = rng.standard_normal((sample, C))
            d = rng.standard_normal((sample, C))
            gam = 1.0 + 0.1 * rng.standard_normal(C)
            bet = 0.1 * rng.standard_normal(C)
            X = synth.SWEEP_ROWS * C * e

            def rms():
                y, ir = O.rms_norm_fwd(x, gam, 1e-5)
                O.rms_norm_bwd(d, x, gam, ir)

            def ln():
                y, mu, rs = O.layernorm_fwd(x, gam, bet, 1e-5)
                O.layernorm_bwd(d, x, gam, mu, rs)

            def sm():
                y = O.softmax_fwd(x)
                O.softmax_bwd(d, y)

            def silu():
                O.silu_fwd(x)
                O.silu_bwd(d, x)

            def swiglu():
                O.swiglu_fwd(x, d)
                O.swiglu_bwd(d, x, d)

            def drop():
                OD.dropout_fwd(x.reshape(-1), 0.1, 0x5EED, dtype=dtn)
                OD.dropout_bwd(d.reshape(-1), 0.1, 0x5EED, dtype=dtn)

            for name, fn, nbytes in (("rms_norm", rms, 5 * X), ("layernorm", ln, 5 * X), ("softmax", sm, 5 * X),
                                     ("silu", silu, 5 * X), ("swiglu", swiglu, 8 * X), ("dropout p=0.1", drop, 4 * X)):
                t = timed(fn) * synth.SWEEP_ROWS / sample
                print(json.dumps({"impl": "reference", "sweep": f"{name} fwd+bwd {dtn} {synth.SWEEP_ROWS}x{C}",
                                  "seconds": round(t, 4), "bytes": int(nbytes), "gbs": round(nbytes / t / 1e9, 3),
                                  "threads": cores, "sample_rows": sample}), flush=True)
    cfg = synth.BIGVOCAB
    R, V = cfg["rows"], cfg["V"]
    rows = 16
    x = rng.standard_normal((rows, V)) * cfg["std"]
    t = rng.integers(0, V, size=rows)

    def fan():
        _, lse = O.cross_entropy_fwd(x, t)
        ones = np.ones_like(x)
        O.cross_entropy_bwd(x, t, lse, 1.0) + O.scale_bwd(ones, 0.5) + sum(O.mul_bwd(ones, x, x))
    tt = timed(fan) * R / rows
    nbytes = 6 * R * V
    print(json.dumps({"impl": "reference", "sweep": f"fan-out CE + sum(0.5x) + sum(x*x) fwd+bwd {R}x{V}",
                      "seconds": round(tt, 3), "bytes": int(nbytes), "gbs": round(nbytes / tt / 1e9, 3),
                      "threads": cores, "sample_rows": rows}), flush=True)


def run_reference(args, rank, world):
    """The oracle, as it stands, on the host cores.  One untimed full-sequence sample sizes the
    per-step sample: a causal prefix of one sequence (a multiple of 128 positions, at least 128)
    chosen so that the warm-up and timed steps together take about REF_BUDGET_S seconds."""
    if rank != 0:
        return
    import synth
    cfg = synth.BLOCK_CONFIGS[args.workload]
    S = cfg["S"]
    _, t_full, _ = oracle_sample(args.workload, 1)
    per_step = REF_BUDGET_S / max(1, args.warmup + args.steps)
    prefix = int(min(S, max(128, 128 * int(S * per_step / t_full / 128))))
    rates = []
    for i in range(args.warmup + args.steps):
        r, t, n = oracle_sample(args.workload, 1, prefix=prefix)
        if i >= args.warmup:
            rates.append((r, t))
    secs = [t for _, t in rates]
    value = n / statistics.mean(secs)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * statistics.mean(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": REFERENCE_TEXT[args.workload].format(n=n), "global_batch": cfg["B"],
                   "seq_len": cfg["S"], "parallelism": "cpu"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                  "sample": f"per step: the first {n} positions of one sequence (of {cfg['B']} x {S}), "
                                   f"all {cfg['n_layers']} layers, float64 NumPy forward + backward"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ our arm


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import __graft_entry__
    import synth
    from transformer_fwd_bwd_gb300 import xt
    from transformer_fwd_bwd_gb300.block import NativeBlock

    __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = dict(synth.BLOCK_CONFIGS[args.workload], recompute=int(args.recompute))
    T = cfg["B"] * cfg["S"]
    nb = NativeBlock(cfg, device=dev, training=True, base_seed=synth.BASE_SEED_DROPOUT)
    nb.load(synth.block_params(cfg))
    ids_h, tgt_h = synth.block_tokens(cfg, seed=synth.SEED_TOKENS + rank)
    ids = torch.tensor(ids_h, device=dev)
    tgt = torch.tensor(tgt_h, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        nb.zero_grads(stream)
        nb.forward(ids, tgt, stream)
        nb.backward(ids, tgt, stream)

    for _ in range(max(1, args.warmup)):   # eager warm-up: kernel attributes and tensor maps are set up here
        step()
    torch.cuda.synchronize(dev)
    assert xt.device_errors() == 0, "device error flag set during warm-up"

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # ---------------- the step captured as CUDA graphs ----------------
    # The step is enqueued once into a graph and replayed: the same kernels, without host launch
    # gaps, and with every kernel launched as a programmatic dependent of the one before it.
    # Two captures of the same step: `graph` for the throughput (and e2e) measurement, and
    # `graph_prof` with GEMM timing on, for the GEMM roofline: every CTA of every GEMM launch
    # stores %globaltimer when it starts work and when it is done (no event or extra node enters
    # the graph, so the programmatic edges stay); the pass is timed and reported separately.
    def capture(block, profile):
        xt.profile_gemm(400 * cfg["n_layers"] // 12 + 64 if profile else 0)
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        n0 = xt.launch_count()
        with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
            cs = torch.cuda.current_stream(dev)
            block.zero_grads(cs)
            block.forward(ids, tgt, cs)
            block.backward(ids, tgt, cs)
        torch.cuda.synchronize(dev)
        return g, xt.launch_count() - n0

    graph, kernels_per_step = capture(nb, False)  # (profile_gemm(0) clears the records: capture this one first)
    # the timing pass runs the weight-gradient GEMMs on the step's own stream: beside co-running
    # kernels a launch's timestamps would include the time it waits for the SMs they hold
    xt.block_set_overlap(0)
    try:
        graph_prof, _ = capture(nb, True)
    finally:
        xt.block_set_overlap(1)
    for g_ in (graph, graph_prof):
        for _ in range(3):
            g_.replay()
    torch.cuda.synchronize(dev)
    assert xt.device_errors() == 0, "device error flag set during graph warm-up"

    def timed_replays(g_, steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize(dev)
        with ClockSampler(local_rank) as clk:
            e0.record(stream)
            for _ in range(steps):
                g_.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
        barrier()
        return e0.elapsed_time(e1) / steps, clk

    # ---------------- timed region (device-resident inputs) ----------------
    ms, clocks = timed_replays(graph, args.steps)
    launches = kernels_per_step * args.steps
    assert xt.device_errors() == 0, "device error flag set during the timed region"
    loss = float(nb.loss.item())

    # ---------------- GEMM roofline pass: the same step with the GEMM timestamps ----------------
    ms_prof, clocks_prof = timed_replays(graph_prof, args.steps)
    flops, gms, gshapes = xt.profile_gemm_read(shapes=True)   # the last replay's GEMM launches
    xt.profile_gemm(0)
    assert xt.device_errors() == 0, "device error flag set during the profiled pass"
    del graph_prof

    # ---------------- the composed attention path of the same workload ----------------
    # The pages' attention, matmul(softmax(QKᵀ·scale), V) with the probabilities stored, as
    # separate causal-tile GEMMs around the row softmax (the fused kernel is the default path).
    composed = None
    if cfg.get("attention", "auto") != "composed" and cfg["dtype"] == "bf16" and world == 1 and not args.step_only:
        nbc = NativeBlock(dict(cfg, attention="composed"), device=dev, training=True,
                          base_seed=synth.BASE_SEED_DROPOUT)
        nbc.load(synth.block_params(cfg))
        for _ in range(max(1, args.warmup)):
            nbc.zero_grads(stream)
            nbc.forward(ids, tgt, stream)
            nbc.backward(ids, tgt, stream)
        torch.cuda.synchronize(dev)
        graph_c, kernels_c = capture(nbc, False)
        for _ in range(3):
            graph_c.replay()
        ms_c, clocks_c = timed_replays(graph_c, args.steps)
        assert xt.device_errors() == 0, "device error flag set during the composed-attention pass"
        composed = {"value": T / (ms_c / 1000.0), "unit": "tokens/s", "ms_per_step": ms_c,
                    "loss": float(nbc.loss.item()), "gpu_launches_per_step": int(kernels_c),
                    "workspace_gb": round(nbc.ws.numel() / 1e9, 3),
                    "attention": "composed: causal-tile QK^T GEMM, row softmax (probabilities stored, bf16), "
                                 "P@V GEMM; backward through the same ops",
                    "clocks": clocks_c.summary()}
        del graph_c, nbc
        torch.cuda.synchronize(dev)

    ms_max = max_over_ranks(ms, dev)
    value = world * T / (ms_max / 1000.0)

    # ---------------- end to end: host buffers, copies inside the timed region ----------------
    ids_pin = torch.tensor(ids_h).pin_memory()
    tgt_pin = torch.tensor(tgt_h).pin_memory()
    loss_pin = torch.empty(1, dtype=torch.float32).pin_memory()
    e2e_steps = max(3, args.steps // 2)

    def e2e_step():
        ids.copy_(ids_pin, non_blocking=True)      # the graph reads ids / tgt in place
        tgt.copy_(tgt_pin, non_blocking=True)
        graph.replay()
        loss_pin.copy_(nb.loss, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()
        return float(loss_pin[0])

    for _ in range(3):   # untimed: first use of the pinned buffers and of this copy path
        e2e_step()
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, dev)

    if rank != 0:
        return
    peaks, peak_src = measured_peaks()
    gemm_ms_step = float(np.sum(gms))
    tflops = float(np.sum(flops)) / (float(np.sum(gms)) * 1e-3) / 1e12 if len(gms) else None
    if cfg["dtype"] == "f32":
        # tf32 dense peak measured on this GPU (cuBLAS through torch.matmul, fp32 with TF32 on)
        peak = measure_tf32_peak(dev)
        peak_sus, src_txt = None, "measured tf32 burst (torch.matmul fp32 8192^3, TF32 allowed, this run)"
    else:
        peak = float(peaks.get("bf16_tflops", 1900.0))
        peak_sus = float(peaks.get("bf16_tflops_sustained", 1700.0))
        src_txt = f"{peak_src} bf16 burst (MEASURED_PEAKS.json bf16_tflops)"
    roofline = {
        "kernel": "gemm_kernel (tcgen05.mma + TMA, all GEMM launches of the step)",
        "bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
        "frac": (tflops / peak) if tflops else None, "peak_source": src_txt,
        "frac_of_sustained": (tflops / peak_sus) if (tflops and peak_sus) else None,
        "peak_sustained": peak_sus,
        "traffic": None,
        "traffic_note": "DRAM bytes are not measured in this run (ncu only); see profiles/ for captures",
        "launches_per_step": len(gms),
        "share_of_step": gemm_ms_step / ms_prof, "gemm_tflop_per_step": float(np.sum(flops)) / 1e12,
        "measured_in": (f"second pass of {args.steps} replays of the same step, captured with GEMM timing on and "
                        f"the weight-gradient GEMMs on the step's own stream (no co-running kernels): each CTA "
                        f"of each GEMM launch stores %globaltimer after its wait for the preceding kernel and when "
                        f"done; a launch's time is the latest end minus the earliest start (programmatic launch "
                        f"edges intact); that pass ran {ms_prof:.3f} ms/step, the timed pass that gives `value` "
                        f"(weight gradients on a second stream) {ms:.3f} ms/step"),
        "clocks_profiled_pass": clocks_prof.summary(),
        "by_shape": gemm_by_shape(flops, gms, gshapes),
    }
    cpu = cpu_baseline(args.workload, args.sample_seqs) if world == 1 and not args.step_only else None
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": cfg["dtype"], "data": "synthetic (seeded tokens, N(0,0.02) weights)",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "model": args.workload, "global_batch": world * cfg["B"],
                   "seq_len": cfg["S"], "parallelism": f"replicas x{world} (data parallel, no collective)",
                   "activation_recompute": bool(args.recompute), "workspace_gb": round(nb.ws.numel() / 1e9, 3),
                   "l2": "inputs larger than L2 (weights 85M params + GBs of saved activations per step)",
                   "loss": loss},
        "e2e": {"value": world * T / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": int(2 * T * 4),
                "d2h_bytes_per_step": 4},
        "gpu_launches": int(launches),
        "roofline": roofline,
        "composed_attention": composed,
        "cpu_baseline": cpu,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


def measure_tf32_peak(dev):
    """Dense tf32 tensor throughput of this GPU: cuBLAS (torch.matmul) on 8192³ fp32 operands with
    TF32 allowed, best of 10 after 3 untimed, CUDA events on the current stream (TFLOP/s)."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        n = 8192
        a = torch.randn(n, n, device=dev)
        b = torch.randn(n, n, device=dev)
        c = torch.empty(n, n, device=dev)
        for _ in range(3):
            torch.matmul(a, b, out=c)
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            torch.cuda.synchronize(dev)
            best = min(best, e0.elapsed_time(e1))
        del a, b, c
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def gemm_by_shape(flops, gms, shapes, top=12):
    """The GEMM launches of one step grouped by (M, N, K, batches, BN (1000 + BN for the paired-CTA
    kernel), A MN-major, B MN-major, causal mode, 10 x K splits, 1000 for stream-K over every SM,
    1000 + s for s lockstep K slices): launches per step, summed event time (a K split's reduce
    included) and TFLOP/s of each group, largest time first."""
    groups = {}
    for f, t, sh in zip(flops, gms, shapes):
        g = groups.setdefault(tuple(int(x) for x in sh), [0, 0.0, 0.0])
        g[0] += 1
        g[1] += float(t)
        g[2] += float(f)
    rows = sorted(groups.items(), key=lambda kv: -kv[1][1])[:top]
    def sched(c):
        if c >= 1000:
            return "stream_k" if c == 1000 else f"stream_k_slices_{c - 1000}"
        return f"k_split_{c // 10}" if c >= 10 else "tiles"
    return [{"mnk": list(k[:3]), "batches": 1 if 10 <= k[7] < 1000 else k[3], "bn": k[4] % 1000,
             "paired": k[4] > 1000, "a_mn": k[5],
             "b_mn": k[6], "causal": 0 if k[7] >= 10 else k[7], "schedule": sched(k[7]),
             "launches": n, "ms": round(t, 4), "tflops": round(f / (t * 1e-3) / 1e12, 1) if t > 0 else None}
            for k, (n, t, f) in rows]


def run_kernel(args):
    """One kernel family alone on seeded N(0, 1) inputs: 3 untimed launches, then 20 timed with
    CUDA events; prints one JSON line (µs per launch and algorithmic TFLOP/s)."""
    import torch

    import __graft_entry__
    import synth
    from transformer_fwd_bwd_gb300 import xt

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(synth.SEED_SWEEP)

    clocks = []

    def timed(fn, n=200):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(0) as cs:
            e0.record()
            for _ in range(n):
                fn()
            e1.record()
            torch.cuda.synchronize(dev)
        clocks.append(cs.summary())
        assert xt.device_errors() == 0, "device error flag set"
        return e0.elapsed_time(e1) / n * 1e3

    if args.kernel == "attention":
        cfg = synth.BLOCK_CONFIGS[args.workload]
        B, S, H, hd = cfg["B"], cfg["S"], cfg["H"], cfg["hd"]
        d = H * hd
        qkv = torch.randn(B * S, 3 * d, generator=g).to(torch.bfloat16).to(dev)
        dO = torch.randn(B * S, d, generator=g).to(torch.bfloat16).to(dev)
        o = torch.empty(B * S, d, dtype=torch.bfloat16, device=dev)
        o_lo = torch.empty(B * S, d, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(B, H, S, dtype=torch.float32, device=dev)
        dqkv = torch.empty_like(qkv)
        nws = xt.ws_bytes("xt_attention_bwd_workspace_size", B, S, H)
        ws = torch.empty(max(1, nws), dtype=torch.uint8, device=dev)
        q, k, v = qkv[:, :d], qkv[:, d:2 * d], qkv[:, 2 * d:]
        fwd_us = timed(lambda: xt.xt_attention_fwd(q, k, v, o, lse, B, S, H, hd, 1, o_lo=o_lo))
        bwd_us = timed(lambda: xt.xt_attention_bwd(q, k, v, o, dO, lse, dqkv[:, :d], dqkv[:, d:2 * d],
                                                   dqkv[:, 2 * d:], B, S, H, hd, 1, o_lo=o_lo, ws=ws))
        fl = 2 * 2 * S * S * hd / 2 * B * H   # QKᵀ and PV over the causal half
        print(json.dumps({"kernel": "attention", "workload": f"B{B} S{S} H{H}x{hd} causal bf16",
                          "fwd_us": fwd_us, "bwd_us": bwd_us,
                          "fwd_tflops": fl / fwd_us / 1e6, "bwd_tflops": 2 * fl / bwd_us / 1e6, "clocks": clocks}))
    elif args.kernel == "layernorm":
        # as the stack launches it: bf16 rows, float32 residual gradient accumulated, float32 dγ / dβ
        cfg = synth.BLOCK_CONFIGS[args.workload]
        R, Cn = cfg["B"] * cfg["S"], cfg["d"]
        x = torch.randn(R, Cn, generator=g).to(torch.bfloat16).to(dev)
        dy = torch.randn(R, Cn, generator=g).to(torch.bfloat16).to(dev)
        gam = torch.ones(Cn, dtype=torch.bfloat16, device=dev)
        bet = torch.zeros(Cn, dtype=torch.bfloat16, device=dev)
        y = torch.empty_like(x)
        mean = torch.empty(R, dtype=torch.float32, device=dev)
        rstd = torch.empty(R, dtype=torch.float32, device=dev)
        dh = torch.zeros(R, Cn, dtype=torch.float32, device=dev)
        dg = torch.zeros(Cn, dtype=torch.float32, device=dev)
        db = torch.zeros(Cn, dtype=torch.float32, device=dev)
        fwd_us = timed(lambda: xt.xt_layernorm_fwd(x, gam, bet, y, mean, rstd, cfg["eps"]))
        bwd_us = timed(lambda: xt.xt_layernorm_bwd(dy, x, gam, mean, rstd, dh, dg, db, acc_dx=1, acc_param=1))
        fb, bb = 2 * R * Cn * 2 + 8 * R, R * Cn * (2 + 2 + 4 + 4) + 8 * R   # fwd: x, y; bwd: d, x, dh read + write
        print(json.dumps({"kernel": "layernorm", "rows": R, "cols": Cn, "fwd_us": fwd_us, "bwd_us": bwd_us,
                          "fwd_gbs": fb / fwd_us / 1e3, "bwd_gbs": bb / bwd_us / 1e3, "clocks": clocks}))
    elif args.kernel == "gelu":
        cfg = synth.BLOCK_CONFIGS[args.workload]
        n = cfg["B"] * cfg["S"] * cfg["F"]
        a = torch.randn(n, generator=g).to(torch.bfloat16).to(dev)
        d = torch.randn(n, generator=g).to(torch.bfloat16).to(dev)
        y = torch.empty_like(a)
        dx = torch.empty_like(a)
        fwd_us = timed(lambda: xt.xt_gelu_fwd(a, y))
        bwd_us = timed(lambda: xt.xt_gelu_bwd(d, a, dx))
        print(json.dumps({"kernel": "gelu", "n": n, "fwd_us": fwd_us, "bwd_us": bwd_us,
                          "fwd_gbs": 4 * n / fwd_us / 1e3, "bwd_gbs": 6 * n / bwd_us / 1e3, "clocks": clocks}))
    elif args.kernel == "adamw":
        # the optimizer step over the stack's parameter tensors (float32 masters, bf16 copies)
        cfg = synth.BLOCK_CONFIGS[args.workload]
        d, F, V, S, L = cfg["d"], cfg["F"], cfg["V"], cfg["S"], cfg["n_layers"]
        up = 2 * F if cfg["mlp"] == "swiglu" else F
        shapes = [(V, d), (d,), (d,)] + ([(S, d)] if cfg["learned_pos"] else [])
        for _ in range(L):
            shapes += [(d,), (d,), (d,), (d,), (d, 3 * d), (d, d), (d, up), (F, d)]
        mk = lambda sh: (torch.randn(*sh, generator=g) * 0.02).to(dev)  # noqa: E731
        P = [mk(sh) for sh in shapes]
        G = [mk(sh) for sh in shapes]
        M = [torch.zeros_like(x) for x in P]
        Vv = [torch.zeros_like(x) for x in P]
        SH = [torch.empty(x.shape, dtype=torch.bfloat16, device=dev) for x in P]
        nrm = torch.zeros(1, dtype=torch.float32, device=dev)
        ows = xt.adamw_workspace([x.numel() for x in P], dev)
        acfg = xt.adamw_config(1e-4, weight_decay=0.1, max_grad_norm=1.0, grad_scale=0.5, step=1)
        us = timed(lambda: xt.xt_adamw_step(acfg, P, G, M, Vv, shadows=SH, norm_out=nrm, ws=ows))
        n = sum(x.numel() for x in P)
        nbytes = n * (4 + 16 + 12 + 2)   # norm pass reads g; update reads θ, g, m, v, writes θ, m, v, bf16 θ
        peak = measured_peaks()[0].get("hbm_gbs", 6780.0)
        print(json.dumps({"kernel": "adamw", "tensors": len(P), "params": n, "us": us,
                          "gbs": nbytes / us / 1e3, "frac_of_measured_hbm": nbytes / us / 1e3 / peak,
                          "clocks": clocks}))
    elif args.kernel == "fp8gemm":
        # e4m3 GEMM (A [M, K], B [N, K], K contiguous) after per-tensor quantization, bf16 out
        M, N, K, _, _ = (int(x) for x in args.shape.split(","))
        A = torch.randn(M, K, generator=g).to(dev)
        Bm = torch.randn(N, K, generator=g).to(dev)
        Aq = torch.empty(M, K, dtype=torch.uint8, device=dev)
        Bq = torch.empty(N, K, dtype=torch.uint8, device=dev)
        da = torch.empty(1, dtype=torch.float32, device=dev)
        db = torch.empty(1, dtype=torch.float32, device=dev)
        xt.xt_quantize_fp8(A, Aq, da)
        xt.xt_quantize_fp8(Bm, Bq, db)
        C = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        us = timed(lambda: xt.xt_matmul_fp8_fwd(Aq, Bq, C, scale_a=da, scale_b=db))
        qus = timed(lambda: xt.xt_quantize_fp8(A, Aq, da))
        peaks, src = measured_peaks()
        peak = 2.0 * peaks.get("bf16_tflops", 1900.0)   # the bf16 burst measurement × the nominal fp8/bf16 ratio
        tf = 2 * M * N * K / us / 1e6
        print(json.dumps({"kernel": "fp8gemm", "shape": [M, N, K], "us": us, "tflops": tf, "peak_tflops": peak,
                          "frac": tf / peak, "peak_source": f"{src} bf16 burst x 4.5/2.25",
                          "quantize_us": qus, "quantize_gbs": M * K * (4 + 1) / qus / 1e3, "clocks": clocks}))
    elif args.kernel == "ce_fanout":
        # the fused fan-out L = CE(x) + 0.5·Σx + Σx∘x on 128256-wide bf16 logits ~N(0, 2), float32 gradient
        cfg = synth.BIGVOCAB
        R, V = (args.rows or cfg["rows"]), cfg["V"]
        x = (torch.randn(R, V, generator=g) * cfg["std"]).to(torch.bfloat16).to(dev)
        tg = torch.randint(0, V, (R,), generator=g, dtype=torch.int32).to(dev)
        G = torch.empty(R, V, dtype=torch.float32, device=dev)
        lse = torch.empty(R, dtype=torch.float32, device=dev)
        loss = torch.empty(1, dtype=torch.float32, device=dev)
        sums = torch.empty(3, dtype=torch.float32, device=dev)
        fws = xt.workspace(xt.ws_bytes("xt_cross_entropy_fanout_workspace_size", R), dev)
        us = timed(lambda: xt.xt_cross_entropy_fanout_fwd_bwd(x, tg, 0.5, 1.0, lse, loss, sums, G, ws=fws), n=20)
        nbytes = 6 * R * V
        peak = measured_peaks()[0].get("hbm_gbs", 6780.0)
        print(json.dumps({"kernel": "ce_fanout", "rows": R, "V": V, "us": us, "gbs": nbytes / us / 1e3,
                          "frac_of_measured_hbm": nbytes / us / 1e3 / peak, "clocks": clocks}))
    elif args.kernel == "cross_entropy":
        # the tied-logit loss as the stack runs it: bf16 logits [B·S, V], backward in place
        cfg = synth.BLOCK_CONFIGS[args.workload]
        R, V = cfg["B"] * cfg["S"], cfg["V"]
        x = (torch.randn(R, V, generator=g) * 2.0).to(torch.bfloat16).to(dev)
        tg = torch.randint(0, V, (R,), generator=g, dtype=torch.int32).to(dev)
        lse = torch.empty(R, dtype=torch.float32, device=dev)
        loss = torch.empty(1, dtype=torch.float32, device=dev)
        one = torch.ones(1, dtype=torch.float32, device=dev)
        dx = torch.empty_like(x)
        fwd_us = timed(lambda: xt.xt_cross_entropy_fwd(x, tg, lse, loss))
        bwd_us = timed(lambda: xt.xt_cross_entropy_bwd(x, tg, lse, one, dx))
        print(json.dumps({"kernel": "cross_entropy", "rows": R, "V": V, "fwd_us": fwd_us, "bwd_us": bwd_us,
                          "fwd_gbs": 2 * R * V / fwd_us / 1e3, "bwd_gbs": 4 * R * V / bwd_us / 1e3,
                          "clocks": clocks}))
    else:
        M, N, K, ta, tb = (int(x) for x in args.shape.split(","))
        A = (torch.randn(K, M, generator=g) if ta else torch.randn(M, K, generator=g)).to(torch.bfloat16).to(dev)
        Bm = (torch.randn(N, K, generator=g) if tb else torch.randn(K, N, generator=g)).to(torch.bfloat16).to(dev)
        C = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        xt.gemm_set_pairing(args.pairing)
        xt.gemm_set_schedule(args.schedule)
        desc = xt.matmul_desc(M, N, K, trans_a=ta, trans_b=tb, dtype_c=xt.XT_BF16)
        mws = xt.matmul_workspace(desc, dev)
        us = timed(lambda: xt.xt_matmul_fwd(desc, A, Bm, C, ws=mws))
        xt.profile_gemm(8)
        xt.xt_matmul_fwd(desc, A, Bm, C, ws=mws)
        torch.cuda.synchronize(dev)
        _, _, sh = xt.profile_gemm_read(shapes=True)
        xt.profile_gemm(0)
        bn = int(sh[0][4])
        print(json.dumps({"kernel": "gemm", "shape": [M, N, K, ta, tb], "us": us, "tflops": 2 * M * N * K / us / 1e6,
                          "paired": bn > 1000, "bn": bn % 1000, "schedule_code": int(sh[0][7]),
                          "clocks": clocks}))


def run_sweep(args):
    """Isolated memory-bound ops, forward and backward, at rows 8192 × cols ∈ {768, 2048, 4096, 8192} in fp32 and
    bf16 (x and the upstream gradient ~N(0, 1); RoPE with head_dim 128 and position = row mod 1024; dropout at
    p ∈ {0, 0.1, 0.5}), then cross-entropy and the three-branch fan-out on 8192 × 128256 bf16 logits ~N(0, 2).
    Each case: 3 untimed launches, then 30 launches each timed alone with its own CUDA events after 1 GiB has been
    read (so no input, and no dirty line, is left in the 129 MB L2); the median is reported.  GB/s = algorithmic bytes / time,
    `frac` of the measured HBM copy bandwidth."""
    import torch

    import __graft_entry__
    import synth
    from transformer_fwd_bwd_gb300 import tape as TP
    from transformer_fwd_bwd_gb300 import xt

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    peaks, peak_src = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    g = torch.Generator().manual_seed(synth.SEED_SWEEP)

    flush = torch.zeros(256 * 1024 * 1024, dtype=torch.float32, device=dev)   # 1 GiB
    flush_acc = torch.zeros((), dtype=torch.float32, device=dev)

    def timed(fn, n=30):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for e0, e1 in evs:
            # L2 flushed by a 1 GiB read: the lines left behind are clean, so the timed launch pays
            # for no write-back of the flush itself (a 1 GiB write would leave up to 129 MB dirty)
            torch.sum(flush, 0, out=flush_acc)
            e0.record()
            fn()
            e1.record()
        torch.cuda.synchronize(dev)
        assert xt.device_errors() == 0, "device error flag set"
        ts = sorted(e0.elapsed_time(e1) for e0, e1 in evs)
        return ts[len(ts) // 2] * 1e3

    def report(case, us, nbytes):
        gbs = nbytes / us / 1e3
        print(json.dumps({"sweep": case, "us": round(us, 2), "bytes": int(nbytes), "gbs": round(gbs, 1),
                          "frac": round(gbs / hbm, 3), "peak": f"{hbm:.0f} GB/s {peak_src}"}), flush=True)

    R = synth.SWEEP_ROWS
    for dtn, tdt in (("f32", torch.float32), ("bf16", torch.bfloat16)):
        e = 4 if dtn == "f32" else 2
        for C in synth.SWEEP_COLS:
            X = R * C * e
            rn = lambda *shape: torch.randn(*shape, generator=g).to(tdt).to(dev)  # noqa: E731
            x, d = rn(R, C), rn(R, C)
            y, dx = torch.empty_like(x), torch.empty_like(x)
            gam = (1 + 0.1 * torch.randn(C, generator=g)).to(tdt).to(dev)
            bet = (0.1 * torch.randn(C, generator=g)).to(tdt).to(dev)
            st1 = torch.empty(R, dtype=torch.float32, device=dev)
            st2 = torch.empty(R, dtype=torch.float32, device=dev)
            pg = torch.empty(C, dtype=torch.float32, device=dev)
            pb = torch.empty(C, dtype=torch.float32, device=dev)
            nws = xt.workspace(xt.ws_bytes("xt_norm_bwd_workspace_size", R, C), dev)
            cws = xt.workspace(xt.ws_bytes("xt_colsum_workspace_size", R, C), dev)
            tag = f"{dtn} {R}x{C}"
            report(f"rms_norm fwd {tag}", timed(lambda: xt.xt_rms_norm_fwd(x, gam, y, st1, 1e-5)), 2 * X + 4 * R)
            report(f"rms_norm bwd {tag}", timed(lambda: xt.xt_rms_norm_bwd(d, x, gam, st1, dx, pg, ws=nws)),
                   3 * X + 4 * R)
            report(f"layernorm fwd {tag}", timed(lambda: xt.xt_layernorm_fwd(x, gam, bet, y, st1, st2, 1e-5)),
                   2 * X + 8 * R)
            report(f"layernorm bwd {tag}",
                   timed(lambda: xt.xt_layernorm_bwd(d, x, gam, st1, st2, dx, pg, pb, ws=nws)), 3 * X + 8 * R)
            report(f"softmax fwd {tag}", timed(lambda: xt.xt_softmax_fwd(x, y)), 2 * X)
            report(f"softmax bwd {tag}", timed(lambda: xt.xt_softmax_bwd(d, y, dx)), 3 * X)
            report(f"silu fwd {tag}", timed(lambda: xt.xt_silu_fwd(x, y)), 2 * X)
            report(f"silu bwd {tag}", timed(lambda: xt.xt_silu_bwd(d, x, dx)), 3 * X)
            u, du = rn(R, C), torch.empty_like(x)
            report(f"swiglu fwd {tag}", timed(lambda: xt.xt_swiglu_fwd(x, u, y)), 3 * X)
            report(f"swiglu bwd {tag}", timed(lambda: xt.xt_swiglu_bwd(d, x, u, dx, du)), 5 * X)
            hd = synth.SWEEP_ROPE_HD
            S = synth.SWEEP_ROPE_SEQ
            tab = torch.empty(2 * S * hd // 2, dtype=torch.float32, device=dev)
            xt.xt_rope_table(tab, S, hd, 10000.0)
            report(f"rope fwd {tag}", timed(lambda: xt.xt_rope_fwd(x, y, tab, R // S, S, C // hd, hd, C)), 2 * X)
            report(f"rope bwd {tag}", timed(lambda: xt.xt_rope_bwd(d, dx, tab, R // S, S, C // hd, hd, C)), 2 * X)
            report(f"add_bias fwd {tag}", timed(lambda: xt.xt_add_bias_fwd(x, bet, y)), 2 * X + C * e)
            report(f"add_bias bwd (dbias) {tag}", timed(lambda: xt.xt_add_bias_bwd(d, None, pb, ws=cws)), X)
            for pdrop in synth.SWEEP_DROPOUT_P:
                report(f"dropout fwd p={pdrop} {tag}",
                       timed(lambda: xt.xt_dropout_fwd(x, y, pdrop, synth.BASE_SEED_DROPOUT)), 2 * X)
                report(f"dropout bwd p={pdrop} {tag}",
                       timed(lambda: xt.xt_dropout_bwd(d, dx, pdrop, synth.BASE_SEED_DROPOUT)), 2 * X)
            del x, d, y, dx, u, du
            torch.cuda.empty_cache()

    # cross-entropy on 8192 × 128256 bf16 logits, and the fan-out CE(x) + Σ 0.5·x + Σ x∘x into one fp32 gradient
    cfg = synth.BIGVOCAB
    R, V = cfg["rows"], cfg["V"]
    X = (torch.randn(R, V, generator=g) * cfg["std"]).to(torch.bfloat16).to(dev)
    tg = torch.randint(0, V, (R,), generator=g, dtype=torch.int32).to(dev)
    lse = torch.empty(R, dtype=torch.float32, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    one = torch.ones(1, dtype=torch.float32, device=dev)
    G = torch.empty(R, V, dtype=torch.float32, device=dev)
    cws = xt.workspace(xt.ws_bytes("xt_cross_entropy_workspace_size", R), dev)
    n = R * V
    report(f"cross_entropy fwd bf16 {R}x{V}", timed(lambda: xt.xt_cross_entropy_fwd(X, tg, lse, loss, ws=cws)), 2 * n)
    report(f"cross_entropy bwd bf16 -> f32 grad {R}x{V}",
           timed(lambda: xt.xt_cross_entropy_bwd(X, tg, lse, one, G)), 2 * n + 4 * n)

    def fanout():
        x = TP.leaf(X, grad_dtype=torch.float32)
        L = TP.add(TP.add(TP.cross_entropy(x, tg), TP.sum_all(TP.scale(x, 0.5))), TP.sum_all(TP.mul(x, x)))
        TP.backward(L)
    report(f"fan-out CE + sum(0.5x) + sum(x*x), tape fwd+bwd, fp32 grad {R}x{V} (vs the fused minimum)",
           timed(fanout, n=5), 2 * n + 4 * n)
    # one pass: rows split across a cluster of CTAs (forward and backward, the gradient in place)
    Xc = X.clone()
    report(f"cross_entropy fwd+bwd one pass (rows split over a cluster), bf16 in place {R}x{V}",
           timed(lambda: xt.xt_cross_entropy_fwd_bwd(Xc, tg, lse, loss, one, Xc, ws=cws)), 2 * n + 2 * n)
    del Xc
    report(f"cross_entropy fwd+bwd one pass (rows split over a cluster), bf16 -> f32 grad {R}x{V}",
           timed(lambda: xt.xt_cross_entropy_fwd_bwd(X, tg, lse, loss, one, G, ws=cws)), 2 * n + 4 * n)
    sums = torch.empty(3, dtype=torch.float32, device=dev)
    fws = xt.workspace(xt.ws_bytes("xt_cross_entropy_fanout_workspace_size", R), dev)
    # the 12-layer stack's vocabulary: in place (one CTA per row) and into a float32 gradient
    # (rows split over a cluster)
    Vs = synth.BLOCK_CONFIGS["gpt12"]["V"]
    Xs = (torch.randn(R, Vs, generator=g) * cfg["std"]).to(torch.bfloat16).to(dev)
    tgs = torch.randint(0, Vs, (R,), generator=g, dtype=torch.int32).to(dev)
    Gs = torch.empty(R, Vs, dtype=torch.float32, device=dev)
    ns = R * Vs
    report(f"cross_entropy fwd+bwd one pass, bf16 in place {R}x{Vs}",
           timed(lambda: xt.xt_cross_entropy_fwd_bwd(Xs, tgs, lse, loss, one, Xs, ws=cws)), 4 * ns)
    report(f"cross_entropy fwd+bwd one pass (rows split over a cluster), bf16 -> f32 grad {R}x{Vs}",
           timed(lambda: xt.xt_cross_entropy_fwd_bwd(Xs, tgs, lse, loss, one, Gs, ws=cws)), 6 * ns)
    del Xs, Gs

    def fanout_fused():
        x = TP.leaf(X, grad_dtype=torch.float32)
        TP.backward(TP.cross_entropy_fanout(x, tg, 0.5, 1.0))
    report(f"fan-out CE + sum(0.5x) + sum(x*x), fused node (one pass), tape fwd+bwd, fp32 grad {R}x{V} "
           f"(vs the fused minimum)", timed(fanout_fused, n=20), 2 * n + 4 * n)
    report(f"fan-out fused kernel alone, fp32 grad {R}x{V} (vs the fused minimum)",
           timed(lambda: xt.xt_cross_entropy_fanout_fwd_bwd(X, tg, 0.5, 1.0, lse, loss, sums, G, ws=fws)),
           2 * n + 4 * n)


def main():
    args = parse_args()
    if args.sweep and args.impl == "reference":
        run_reference_sweep(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.kernel:
        run_kernel(args)
        return
    if args.oracle_sample:
        r, t, n = oracle_sample(args.workload, args.sample_seqs)
        reps = 1
        if t < 2.0:   # a small workload: repeat to about 10 s of CPU work, report the median
            reps = max(1, min(2000, int(10.0 / max(t, 1e-4))))
            r, t, n = oracle_sample(args.workload, args.sample_seqs, reps=reps)
        print(json.dumps({"value": r, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                          "cpu": cpu_model(),
                          "sample": f"{n} tokens ({args.sample_seqs} sequence(s)) of the same workload, all layers, "
                                    f"float64 NumPy forward + backward, {t * 1e3:.3f} ms"
                                    + (f" (median of {reps} repetitions)" if reps > 1 else "")}))
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "ours":
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        else:
            dist.init_process_group("gloo")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
