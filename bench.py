#!/usr/bin/env python3
"""Throughput of the tensor-parallel MLP block (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step = tpmlp_forward then tpmlp_backward (all six GEMMs and both bias
gradients) over one batch of seeded synthetic input of the named workload
(default: the 175B-class layer, T=2048 tokens, h=12288, f=49152, t=8).  The
value is fwd+bwd TFLOP/s (12*T*h*f FLOP per step) over all ranks; tokens/s and
the fraction of the dense bf16 peak ride along.  Prints one JSON line.

--workload may also name one of the tensor-parallel linear layers (the
attention projections, e.g. qkv_175b: the 175B-class QKV projection 12288 x
36864, column parallel, t=8; attn_out_175b: its 12288 x 12288 output
projection, row parallel).  One step is then that layer's forward and
backward (3 GEMMs of 2*T*in*out FLOP and the bias gradient).

--sp-layer wraps the MLP workload in the sequence-parallel sublayer
Out = X + Dropout(MLP(LN(X))) (LayerNorm and dropout per token chunk); the
FLOP count stays the block's 12*T*h*f (the LayerNorm and dropout passes are
timed but counted as no FLOP).

--cublas adds an informative comparison: torch.matmul / torch.mm (cuBLAS) on
the block's six GEMM shapes, unsharded, back to back as one step for as many
steps as the timed region (weight gradients with fp32 output where torch.mm
takes out_dtype), with its own clock record ("cublas_reference"), and the
whole block composed from PyTorch ops (cuBLAS GEMMs, PyTorch's GeLU and its
backward, column sums; "cublas_reference.torch_block").

After the main timed loop a sustained sub-record ("sustained") times at least
3 s of back-to-back steps with its own clock record, long enough for the
GPU's power cap to set the clock.  The roofline fraction of the main line is
taken against the burst bf16 peak when its timed region lasted under 2 s and
against the sustained peak otherwise; both fractions ride along.

--impl reference times the fp64 CPU oracle on the host cores instead, on a
bounded token sample of the same layer per step (same metric and unit).
Under torchrun with N > 1 every rank runs an independent replica of the
block (weak scaling; the block needs no data exchange between replicas).
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

METRIC = "TP-MLP fwd+bwd TFLOP/s and tokens/s on 1 GB300; % of BF16 dense peak"
SP_EPS, SP_P, SP_SEED = 1e-5, 0.1, 1234
LINEAR_METRIC = ("TP linear layer (attention projection) fwd+bwd TFLOP/s and tokens/s on 1 GB300; "
                 "% of BF16 dense peak")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PRE_STEPS = 3  # profiled steps before the timed region that pick the kernel kinds timed live
# A timed region shorter than BURST_MAX_S runs before the power cap pulls the
# clock down, so its kernels are compared with the burst peak; a longer one
# with the sustained peak.  The sustained sub-record times at least
# SUSTAINED_MIN_S of back-to-back steps after the main loop.
BURST_MAX_S = 2.0
SUSTAINED_MIN_S = 3.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gpt_175b")
    ap.add_argument("--tokens", type=int, help="override the workload's token count")
    ap.add_argument("--hidden", type=int, help="override h")
    ap.add_argument("--ffn", type=int, help="override f")
    ap.add_argument("--t", type=int, help="override the shard count")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sp-layer", action="store_true",
                    help="run the sequence-parallel sublayer Out = X + Dropout(MLP(LN(X))) around "
                         "the MLP workload (dropout p = 0.1, eps = 1e-5)")
    ap.add_argument("--sp-explicit-copy", action="store_true",
                    help="sequence-parallel workloads: gather the token chunks into one tensor and "
                         "scatter the outputs back with explicit copies (tpmlp_sp_gather / "
                         "tpmlp_sp_scatter) around the un-chunked block, instead of addressing the "
                         "chunks through per-chunk tensor maps (the ablation of the copy-free path)")
    ap.add_argument("--recompute", action="store_true",
                    help="selective recompute: keep only Y between passes, rebuild H in backward")
    ap.add_argument("--split-min-kblocks", type=int, default=None,
                    help="tail-split depth threshold of the GEMMs (0 = off; library default 128)")
    ap.add_argument("--head-prefetch", type=int, default=None,
                    help="K steps of the next tile the GEMMs prefetch into L2 (library default)")
    ap.add_argument("--wide-tiles", type=int, default=None, choices=[0, 1, 2, 3],
                    help="GEMM tile width: 0 = 256-wide, 1 = 512-wide where the waves fill as "
                         "well, 2 = 512-wide wherever allowed, 3 = 512-wide for GEMMs of at least "
                         "256 K steps (library default)")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of one step captured in a CUDA graph (the per-kernel "
                         "times then come from eager steps run after the timed region)")
    ap.add_argument("--cublas", action="store_true",
                    help="also time cuBLAS on the block's six GEMM shapes (unsharded, back to back) "
                         "and the whole block composed from PyTorch ops (informative comparisons)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sustained", action="store_true",
                    help="skip the >= 3 s power-capped sub-record after the main loop")
    return ap.parse_args()


def pick_workload(args):
    """The named workload, with any size overrides applied (for profiling
    smaller cases of the same kernels)."""
    from dataclasses import replace
    from tensor_transformer_mlp_gemm_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    over = {}
    if args.tokens is not None:
        over.update(micro_batch=1, seq=args.tokens)
    if args.hidden is not None:
        over["hidden"] = args.hidden
    if args.ffn is not None:
        over["ffn"] = args.ffn
    if args.t is not None:
        over["t"] = args.t
        over["seq_chunks"] = min(w.seq_chunks, args.t)
    if over:
        w = replace(w, name=w.name + "(" + ",".join(f"{k}={v}" for k, v in over.items()) + ")",
                    **over)
    return w


def pick_linear_workload(args):
    from dataclasses import replace
    from tensor_transformer_mlp_gemm_gb300.inputs import LINEAR_WORKLOADS
    w = LINEAR_WORKLOADS[args.workload]
    over = {}
    if args.tokens is not None:
        over["tokens"] = args.tokens
    if args.t is not None:
        over["t"] = args.t
        over["seq_chunks"] = min(w.seq_chunks, args.t)
    if over:
        w = replace(w, name=w.name + "(" + ",".join(f"{k}={v}" for k, v in over.items()) + ")",
                    **over)
    return w


def is_linear(args) -> bool:
    from tensor_transformer_mlp_gemm_gb300.inputs import LINEAR_WORKLOADS
    return args.workload in LINEAR_WORKLOADS


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# The files that decide what the GEMM kernels do and how they are launched
# (tile raster, operand descriptors): the recorded DRAM traffic stays valid
# while these are unchanged.
GEMM_SOURCES = ("gemm.cuh", "gemm_params.h", "ptx.cuh", "philox.cuh", "gemm_fwd.cu", "gemm_dgrad.cu",
                "gemm_wgrad.cu", "gemm_fwd_dropout.cu", "tpmlp.cu", "abi_internal.h",
                "block_internal.h")


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tensor_transformer_mlp_gemm_gb300", "csrc")
    for name in GEMM_SOURCES:
        h.update(name.encode())
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, or None when the
    kernels have changed since those counters were taken (or for another
    workload)."""
    try:
        with open(os.path.join(ROOT, "profiles", "gemm_traffic.json")) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("source_hash") != kernel_source_hash() or workload != "gpt_175b":
        return None
    return d.get("dram_bytes_per_launch", {}).get(kernel)


def workload_config(w, l2_note):
    return {"workload": f"{w.name}: T={w.tokens} (mb {w.micro_batch} x seq {w.seq}), "
                        f"h={w.hidden}, f={w.ffn}, t={w.t}, seq_chunks={w.seq_chunks}",
            "tokens": w.tokens, "hidden": w.hidden, "ffn": w.ffn, "t": w.t,
            "seq_chunks": w.seq_chunks, "sigma_w": w.sigma_w, "seed": 0, "l2": l2_note}


def linear_config(w, l2_note):
    return {"workload": f"{w.name}: {w.split}-parallel linear, T={w.tokens}, in={w.in_features}, "
                        f"out={w.out_features}, t={w.t}, seq_chunks={w.seq_chunks}",
            "tokens": w.tokens, "in_features": w.in_features, "out_features": w.out_features,
            "split": w.split, "t": w.t, "seq_chunks": w.seq_chunks, "sigma_w": w.sigma_w,
            "seed": 0, "l2": l2_note}


# ---- clocks -----------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def gpu_selector(torch, dev_index):
    try:
        props = torch.cuda.get_device_properties(dev_index)
        uuid = str(getattr(props, "uuid", "") or "")
        if uuid:
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[dev_index]
    return str(dev_index)


def cublas_reference(w, torch, dev, steps=300, warmup=10):
    """torch.matmul (cuBLAS) on the MLP block's six GEMM shapes, unsharded, bf16
    in and out (fp32 out for the weight gradients where torch.mm takes
    out_dtype): Y = X.A, Z = H.B, dH = dZ.B^T, dX = dY.A^T, dB = H^T.dZ,
    dA = X^T.dY, run back to back as one step and repeated for as many steps
    as the timed region, so that cuBLAS sees the same power-capped clocks as
    the library's step.  CUDA events around each GEMM; clocks sampled during
    the loop."""
    T, h, f = w.tokens, w.hidden, w.ffn
    bf = torch.bfloat16
    X = torch.randn(T, h, device=dev, dtype=bf)
    A = torch.randn(h, f, device=dev, dtype=bf)
    B = torch.randn(f, h, device=dev, dtype=bf)
    Hm = torch.randn(T, f, device=dev, dtype=bf)
    dZ = torch.randn(T, h, device=dev, dtype=bf)
    shapes = {"column_fwd (X.A)": (X, A), "row_fwd (H.B)": (Hm, B), "dgrad_h (dZ.B^T)": (dZ, B.t()),
              "dgrad_x (dY.A^T)": (Hm, A.t()), "wgrad_b (H^T.dZ)": (Hm.t(), dZ),
              "wgrad_a (X^T.dY)": (X.t(), Hm)}
    outs = {k: torch.empty(a.shape[0], b.shape[1], device=dev, dtype=bf) for k, (a, b) in shapes.items()}
    flop = 2.0 * T * h * f
    names = list(shapes)
    # The weight gradients leave as fp32, like the library's; torch.mm's out_dtype
    # form keeps cuBLAS's fp32 accumulator instead of rounding it to bf16.
    wgrad_fp32 = True
    try:
        a, b = shapes["wgrad_b (H^T.dZ)"]
        torch.mm(a[:128, :128], b[:128, :128], out_dtype=torch.float32)
    except Exception:
        wgrad_fp32 = False

    def gemm(k):
        a, b = shapes[k]
        if wgrad_fp32 and k.startswith("wgrad"):
            return torch.mm(a, b, out_dtype=torch.float32)
        return torch.matmul(a, b, out=outs[k])

    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in names] for _ in range(steps)]
    for _ in range(warmup):
        for k in names:
            gemm(k)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(gpu_selector(torch, dev.index or 0))
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for s in range(steps):
        for n, k in enumerate(names):
            ev[s][n][0].record()
            gemm(k)
            ev[s][n][1].record()
    e1.record()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    per = {}
    for n, k in enumerate(names):
        ms = sum(ev[s][n][0].elapsed_time(ev[s][n][1]) for s in range(steps)) / steps
        per[k] = flop / (ms / 1e3) / 1e12
    ms_step = e0.elapsed_time(e1) / steps
    del X, A, B, Hm, dZ, outs
    torch.cuda.empty_cache()
    return {"tflops": per, "step_tflops": 6 * flop / (ms_step / 1e3) / 1e12, "ms_per_step": ms_step,
            "steps": steps, "clocks": clocks, "wgrad_out": "fp32" if wgrad_fp32 else "bf16",
            "note": "torch.matmul / torch.mm, unsharded shapes, bf16 out (weight gradients as "
                    "wgrad_out), no fused epilogues, six GEMMs back to back per step"}


def torch_block_reference(w, inputs, torch, dev, steps=300, warmup=10):
    """The same block composed from PyTorch CUDA ops, unsharded: cuBLAS GEMMs
    (the biases in their epilogue through addmm), PyTorch's tanh-GeLU and its
    backward, fp32 column sums.  Forward Y = X.A + b1, H = GeLU(Y), Z = H.B + b2;
    backward dH = dZ.B^T, dY = GeLU'(Y) * dH, dX = dY.A^T, dB = H^T.dZ and
    dA = X^T.dY (fp32 where torch.mm takes out_dtype), db1, db2.  Same seeded
    inputs, timed over as many steps as the timed region, clocks sampled."""
    import torch.nn.functional as F
    X, A, b1, B, b2, dZ = (inputs[k].to(dev) for k in ("X", "A", "b1", "B", "b2", "dZ"))
    try:
        torch.mm(X[:128, :128], A[:128, :128], out_dtype=torch.float32)
        fp32 = True
    except Exception:
        fp32 = False

    def wgrad(a, b):
        return torch.mm(a, b, out_dtype=torch.float32) if fp32 else torch.mm(a, b)

    def step():
        Y = torch.addmm(b1, X, A)
        H = F.gelu(Y, approximate="tanh")
        Z = torch.addmm(b2, H, B)
        dH = torch.mm(dZ, B.t())
        dY = torch.ops.aten.gelu_backward(dH, Y, approximate="tanh")
        dX = torch.mm(dY, A.t())
        dB = wgrad(H.t(), dZ)
        dA = wgrad(X.t(), dY)
        db1 = dY.sum(0, dtype=torch.float32)
        db2 = dZ.sum(0, dtype=torch.float32)
        return Z, dX, dA, dB, db1, db2

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(gpu_selector(torch, dev.index or 0))
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / steps
    del X, A, b1, B, b2, dZ
    torch.cuda.empty_cache()
    return {"value": w.flops / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "steps": steps, "clocks": clocks, "wgrad_out": "fp32" if fp32 else "bf16",
            "note": "the block from PyTorch ops (addmm, gelu tanh, gelu_backward, mm, sum), "
                    "unsharded, same inputs"}


def theoretical_peak_tflops(torch, dev):
    """SMs x 8192 dense bf16 FLOP/clk x maximum SM clock."""
    try:
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.max.sm", "--format=csv,noheader,nounits",
                              "-i", str(dev.index or 0)], capture_output=True, text=True, timeout=20)
        mhz = float(out.stdout.strip().splitlines()[0])
        return {"tflops": sms * 8192 * mhz * 1e6 / 1e12, "sms": sms, "max_sm_mhz": mhz}
    except Exception:
        return None


# ---- CPU oracle ----------------------------------------------------------------------------

class OracleSample:
    """The fp64 oracle on the first T_s tokens of the workload (same weights)."""

    def __init__(self, w, inputs):
        import numpy as np
        import oracle
        from tensor_transformer_mlp_gemm_gb300.inputs import column_shards, row_shards
        self.oracle = oracle
        self.cores = len(os.sched_getaffinity(0))
        oracle.set_threads(self.cores)
        self.w = w
        # fp64 copies prepared once, outside any timing (input conversion only)
        self.A = [np.ascontiguousarray(a.double().numpy()) for a in column_shards(inputs["A"], w.t)]
        self.B = [np.ascontiguousarray(b.double().numpy()) for b in row_shards(inputs["B"], w.t)]
        self.b1 = inputs["b1"].double().numpy()
        self.b2 = inputs["b2"].double().numpy()
        self.X = inputs["X"].double().numpy()
        self.dZ = inputs["dZ"].double().numpy()

    def run(self, tokens: int) -> float:
        X = self.X[:tokens]
        dZ = self.dZ[:tokens]
        t0 = time.perf_counter()
        self.oracle.forward_backward(X, self.A, self.b1, self.B, self.b2, dZ)
        return time.perf_counter() - t0

    def calibrate(self, target_s: float, start: int | None = None, cap: int | None = None) -> int:
        tok = start or max(8, self.cores)
        cap = cap or self.w.tokens
        tok = min(tok, cap)
        dt = self.run(tok)
        if dt <= 0:
            return tok
        want = int(tok * target_s / dt)
        want = max(self.cores, (want // self.cores) * self.cores) if want >= self.cores else max(1, want)
        return max(1, min(cap, want))


    def flops(self, tokens: int) -> float:
        return 12.0 * tokens * self.w.hidden * self.w.ffn

    def describe(self) -> str:
        return f"h={self.w.hidden}, f={self.w.ffn}, t={self.w.t}"


class LinearOracleSample(OracleSample):
    """The fp64 oracle of a linear layer on the first T_s tokens (same weights)."""

    def __init__(self, w, inputs):
        import numpy as np
        import oracle
        from tensor_transformer_mlp_gemm_gb300.inputs import column_shards, row_shards
        self.oracle = oracle
        self.cores = len(os.sched_getaffinity(0))
        oracle.set_threads(self.cores)
        self.w = w
        f64 = lambda x: np.ascontiguousarray(x.double().numpy())
        if w.split == "column":
            self.W = [f64(x) for x in column_shards(inputs["W"], w.t)]
            self.X = f64(inputs["X"])
            self.dY = [f64(x) for x in column_shards(inputs["dY"], w.t)]
        else:
            self.W = [f64(x) for x in row_shards(inputs["W"], w.t)]
            self.X = [f64(x) for x in column_shards(inputs["X"], w.t)]
            self.dY = f64(inputs["dY"])
        self.b = f64(inputs["b"])

    def run(self, tokens: int) -> float:
        t0 = time.perf_counter()
        if self.w.split == "column":
            self.oracle.column_linear(self.X[:tokens], self.W, self.b,
                                      [d[:tokens] for d in self.dY])
        else:
            self.oracle.row_linear([x[:tokens] for x in self.X], self.W, self.b,
                                   self.dY[:tokens])
        return time.perf_counter() - t0

    def flops(self, tokens: int) -> float:
        return 6.0 * tokens * self.w.in_features * self.w.out_features

    def describe(self) -> str:
        w = self.w
        return f"{w.split} split, in={w.in_features}, out={w.out_features}, t={w.t}"


class SpOracleSample(OracleSample):
    """The fp64 oracle of the sequence-parallel sublayer on the first T_s tokens."""

    def __init__(self, w, inputs):
        super().__init__(w, inputs)
        self.gamma = inputs["gamma"].double().numpy()
        self.beta = inputs["beta"].double().numpy()

    def run(self, tokens: int) -> float:
        t0 = time.perf_counter()
        self.oracle.sp_layer(self.X[:tokens], self.gamma, self.beta, SP_EPS, self.A, self.b1,
                             self.B, self.b2, SP_P, SP_SEED, dOut=self.dZ[:tokens])
        return time.perf_counter() - t0

    def describe(self) -> str:
        return f"LN + MLP + dropout + residual, h={self.w.hidden}, f={self.w.ffn}, t={self.w.t}"


def oracle_sample(w, inputs, sp_layer=False):
    if hasattr(w, "split"):
        return LinearOracleSample(w, inputs)
    return SpOracleSample(w, inputs) if sp_layer else OracleSample(w, inputs)


def cpu_baseline(w, inputs, target_s: float, sp_layer=False) -> dict:
    smp = oracle_sample(w, inputs, sp_layer)
    tok = smp.calibrate(target_s)
    dt = smp.run(tok)
    flops = smp.flops(tok)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": smp.cores, "kind": "oracle",
            "tokens_per_s": tok / dt, "seconds": dt,
            "sample": f"fp64 oracle fwd+bwd on the first {tok} of {w.tokens} tokens of the same "
                      f"layer ({smp.describe()}), same weights; "
                      f"{flops / 1e9:.1f} GFLOP in {dt:.1f} s"}


# ---- distributed ----------------------------------------------------------------------------

def dist_setup(torch):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return dist, rank, world, local
    return None, rank, world, local


def barrier(dist, torch):
    if dist is not None:
        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(dist, torch, x: float) -> float:
    if dist is None:
        return x
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- arms -------------------------------------------------------------------------------------

def run_reference(args, torch):
    """The oracle arm: fp64 CPU oracle, rank 0 only, bounded token samples."""
    from tensor_transformer_mlp_gemm_gb300.inputs import make_inputs
    dist, rank, world, _ = dist_setup(torch)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    if is_linear(args):
        from tensor_transformer_mlp_gemm_gb300.inputs import make_linear_inputs
        w = pick_linear_workload(args)
        inputs = make_linear_inputs(w, 0)
        metric, config = LINEAR_METRIC, linear_config(w, "host memory (CPU oracle)")
    else:
        from tensor_transformer_mlp_gemm_gb300.inputs import make_sp_inputs
        w = pick_workload(args)
        inputs = make_sp_inputs(w, 0) if args.sp_layer else make_inputs(w, 0)
        metric, config = METRIC, workload_config(w, "host memory (CPU oracle)")
        if args.sp_layer:
            config = {**config, **sp_config()}
    smp = oracle_sample(w, inputs, args.sp_layer)
    per_step = max(0.5, 150.0 / max(1, args.steps + args.warmup))
    tok = smp.calibrate(per_step, start=min(w.tokens, max(4, smp.cores // 2)))
    for _ in range(args.warmup):
        smp.run(tok)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        smp.run(tok)
    dt = time.perf_counter() - t0
    flops = smp.flops(tok) * args.steps
    value = flops / dt / 1e12
    line = {"impl": "reference", "metric": metric, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config,
            "tokens_per_s": tok * args.steps / dt,
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": smp.cores,
                             "kind": "oracle",
                             "sample": f"each step: fp64 oracle fwd+bwd on the first {tok} of "
                                       f"{w.tokens} tokens of the layer, same weights"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


class MlpRunner:
    """One step = tpmlp_forward + tpmlp_backward of the MLP block."""

    def __init__(self, args, dev):
        from tensor_transformer_mlp_gemm_gb300 import binding
        from tensor_transformer_mlp_gemm_gb300.block import DeviceBlock
        from tensor_transformer_mlp_gemm_gb300.inputs import make_inputs
        self.binding = binding
        self.w = w = pick_workload(args)
        self.inputs = make_inputs(w, 0)
        self.recompute = bool(args.recompute)
        self.blk = DeviceBlock(w, self.inputs, device=dev, recompute=args.recompute)
        T, h, f = w.tokens, w.hidden, w.ffn
        self.tokens = T
        self.metric = METRIC
        self.flops_step = 12.0 * T * h * f
        self.gemm_kinds = ("column_fwd", "row_fwd", "dgrad_h", "dgrad_x", "wgrad_b", "wgrad_a")
        self.gemm_flops = 2.0 * T * h * f  # every GEMM launch
        # bias-gradient kernels per step: db1 adds the dH GEMM's fp32 column sums
        # of each 32-row group (read ceil(T/32) x f x 4 bytes, write f x 4); db2
        # sums dZ (read T x h x 2, write h x 4)
        self.colsum_bytes = ((T + 31) // 32) * f * 4 + f * 4 + T * h * 2 + h * 4
        self.l2_note = (f"inputs larger than L2 (bf16 weights {2 * h * f * 2 / 1e9:.2f} GB, "
                        f"activations {3 * T * f * 2 / 1e9:.2f} GB per step)")
        self.ins, self.outs = ("X", "dZ"), ("Z", "dX")  # per-step uploads; fwd, bwd results

    def config(self):
        return {**workload_config(self.w, self.l2_note),
                "activation_recompute": self.recompute}

    def buffers(self, name):
        return getattr(self.blk, name)

    def step(self, stream):
        self.blk.step(stream)

    def forward(self, B, stream):
        b, blk, w = self.binding, self.blk, self.w
        if self.recompute:
            b.tpmlp_forward_recompute(blk.dims, B["X"], blk.A, blk.b1, blk.B, blk.b2, w.t, B["Z"],
                                      blk.saved_y, blk.scratch, stream)
        else:
            b.tpmlp_forward(blk.dims, B["X"], blk.A, blk.b1, blk.B, blk.b2, w.t, B["Z"], blk.ws,
                            stream)

    def backward(self, B, stream):
        b, blk = self.binding, self.blk
        if self.recompute:
            b.tpmlp_backward_recompute(blk.dims, B["dZ"], B["X"], blk.A, blk.B, blk.saved_y,
                                       blk.scratch, B["dX"], blk.dA, blk.db1, blk.dB, blk.db2,
                                       stream)
        else:
            b.tpmlp_backward(blk.dims, B["dZ"], B["X"], blk.A, blk.B, blk.ws, B["dX"], blk.dA,
                             blk.db1, blk.dB, blk.db2, stream)


class MlpCopyRunner(MlpRunner):
    """The sequence-parallel block with explicit copies: X and dZ arrive as
    token chunks, are gathered into one [T, h] tensor each, the block runs
    un-chunked, and Z and dX are scattered back to chunks."""

    def __init__(self, args, dev):
        super().__init__(args, dev)
        import torch
        from dataclasses import replace
        from tensor_transformer_mlp_gemm_gb300.block import DeviceBlock
        w = self.w
        if w.seq_chunks < 2:
            raise SystemExit("--sp-explicit-copy needs a workload with token chunks")
        self.chunked = self.blk            # its X, dZ, Z, dX chunk buffers face the caller
        self.blk = DeviceBlock(replace(w, seq_chunks=1), self.inputs, device=dev,
                               recompute=args.recompute)
        self.cdims = self.chunked.dims
        self.h = w.hidden
        self.torch = torch

    def config(self):
        c = super().config()
        c["sp_addressing"] = "explicit gather / scatter copies around the un-chunked block"
        return c

    def buffers(self, name):
        return getattr(self.chunked, name)

    def step(self, stream):
        self.forward({"X": self.chunked.X, "Z": self.chunked.Z}, stream)
        self.backward({"dZ": self.chunked.dZ, "X": self.chunked.X, "dX": self.chunked.dX},
                      stream)

    def forward(self, B, stream):
        b, blk = self.binding, self.blk
        b.tpmlp_sp_gather(self.cdims, B["X"], self.h, blk.X[0], stream)
        super().forward({"X": blk.X, "Z": blk.Z}, stream)
        b.tpmlp_sp_scatter(self.cdims, blk.Z[0], self.h, B["Z"], stream)

    def backward(self, B, stream):
        b, blk = self.binding, self.blk
        b.tpmlp_sp_gather(self.cdims, B["dZ"], self.h, blk.dZ[0], stream)
        super().backward({"dZ": blk.dZ, "X": blk.X, "dX": blk.dX}, stream)
        b.tpmlp_sp_scatter(self.cdims, blk.dX[0], self.h, B["dX"], stream)


def sp_config():
    return {"sublayer": "Out = X + Dropout(MLP(LN(X))), LayerNorm and dropout per token chunk",
            "layernorm_eps": SP_EPS, "dropout_p": SP_P, "dropout_seed": SP_SEED,
            "flop_count": "the block's 12*T*h*f; LayerNorm and dropout passes timed, no FLOP"}


class SpRunner(MlpRunner):
    """One step = tpmlp_sp_forward + tpmlp_sp_backward of the sublayer."""

    def __init__(self, args, dev):
        from tensor_transformer_mlp_gemm_gb300 import binding
        from tensor_transformer_mlp_gemm_gb300.inputs import make_sp_inputs
        from tensor_transformer_mlp_gemm_gb300.sp import DeviceSPLayer
        self.binding = binding
        self.w = w = pick_workload(args)
        self.inputs = make_sp_inputs(w, 0)
        self.recompute = False
        self.lay = DeviceSPLayer(w, self.inputs, device=dev, eps=SP_EPS, dropout_p=SP_P,
                                 seed=SP_SEED)
        T, h, f = w.tokens, w.hidden, w.ffn
        self.tokens = T
        self.metric = METRIC
        self.flops_step = 12.0 * T * h * f
        self.gemm_kinds = ("column_fwd", "row_fwd", "dgrad_h", "dgrad_x", "wgrad_b", "wgrad_a")
        self.gemm_flops = 2.0 * T * h * f
        # bias-gradient kernels: only db1's finish here (db2 comes out of the dropout pass)
        self.colsum_bytes = ((T + 31) // 32) * f * 4 + f * 4
        # LayerNorm forward reads X, writes LN(X); backward reads X, dLN(X), dOut and writes
        # dX; dgamma and dbeta come out of the same pass (h <= 4096; wider rows re-read X and
        # dLN(X) in a second pass, not counted: algorithmic bytes only)
        self.ln_fwd_bytes = 2 * T * h * 2
        self.ln_bwd_bytes = 4 * T * h * 2
        # dropout backward reads dOut and the mask's bits, writes dZ (and db2 from it)
        self.dropout_bytes = 2 * T * h * 2 + T * ((h + 31) // 32) * 4 + h * 4
        self.l2_note = (f"inputs larger than L2 (bf16 weights {2 * h * f * 2 / 1e9:.2f} GB, "
                        f"activations {(3 * T * f + 4 * T * h) * 2 / 1e9:.2f} GB per step)")
        self.ins, self.outs = ("X", "dOut"), ("Out", "dX")

    def config(self):
        return {**workload_config(self.w, self.l2_note), **sp_config()}

    def buffers(self, name):
        return getattr(self.lay, name)

    def step(self, stream):
        self.lay.step(stream)

    def forward(self, B, stream):
        self.lay.forward(stream, X=B["X"], Out=B["Out"])

    def backward(self, B, stream):
        self.lay.backward(stream, dOut=B["dOut"], X=B["X"], dX=B["dX"])


class LinearRunner:
    """One step = forward + backward of one tensor-parallel linear layer."""

    def __init__(self, args, dev):
        from tensor_transformer_mlp_gemm_gb300.inputs import make_linear_inputs
        from tensor_transformer_mlp_gemm_gb300.linear import DeviceLinear
        self.w = w = pick_linear_workload(args)
        self.inputs = make_linear_inputs(w, 0)
        self.lin = DeviceLinear(w, self.inputs, device=dev)
        T, din, dout = w.tokens, w.in_features, w.out_features
        self.tokens = T
        self.metric = LINEAR_METRIC
        self.flops_step = 6.0 * T * din * dout
        self.gemm_kinds = ("linear_fwd", "linear_dgrad", "linear_wgrad")
        self.gemm_flops = 2.0 * T * din * dout
        # column sums: read dY [T, out] bf16, write db fp32, per step
        self.colsum_bytes = T * dout * 2 + dout * 4
        self.l2_note = (f"inputs larger than L2 (bf16 weight {din * dout * 2 / 1e9:.2f} GB, "
                        f"activations {T * (din + 2 * dout) * 2 / 1e9:.2f} GB per step)")
        self.ins, self.outs = ("X", "dY"), ("Y", "dX")

    def config(self):
        return linear_config(self.w, self.l2_note)

    def buffers(self, name):
        return getattr(self.lin, name)

    def step(self, stream):
        self.lin.step(stream)

    def forward(self, B, stream):
        self.lin.forward(stream, X=B["X"], Y=B["Y"])

    def backward(self, B, stream):
        self.lin.backward(stream, dY=B["dY"], X=B["X"], dX=B["dX"])


def run_ours(args, torch):
    from tensor_transformer_mlp_gemm_gb300.build import build
    dist, rank, world, local = dist_setup(torch)
    if rank == 0:
        build()
    if dist is not None:
        dist.barrier()
    from tensor_transformer_mlp_gemm_gb300 import binding

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.split_min_kblocks is not None:
        binding.tpmlp_set_split_min_kblocks(args.split_min_kblocks)
    if args.head_prefetch is not None:
        binding.tpmlp_set_head_prefetch(args.head_prefetch)
    if args.wide_tiles is not None:
        binding.tpmlp_set_wide_tiles(args.wide_tiles)
    if is_linear(args):
        run = LinearRunner(args, dev)
    elif args.sp_layer:
        run = SpRunner(args, dev)
    elif args.sp_explicit_copy:
        run = MlpCopyRunner(args, dev)
    else:
        run = MlpRunner(args, dev)
    w = run.w
    stream = torch.cuda.current_stream(dev)
    T = run.tokens
    flops_step = run.flops_step

    # warm-up, then the timed device-resident loop
    for _ in range(args.warmup):
        run.step(stream)
    st = binding.tpmlp_sync_check(stream)
    if st != binding.TPMLP_OK:
        raise RuntimeError(f"warm-up failed: {binding.tpmlp_status_string(st)}")
    graph = None
    if args.graph:
        # one whole step captured once; every timed step is a replay of it
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run.step(torch.cuda.current_stream(dev))
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize(dev)
    timed_kinds = None
    if graph is None:
        # The timed region records CUDA events around the launches of the
        # kernel kind with the most device time in a short profiled pass (the
        # dominant kernel); the other kinds' launches get no event records
        # there, which small layers would see in their step time.
        binding.tpmlp_profile_begin(16 * PRE_STEPS + 16)
        for _ in range(PRE_STEPS):
            run.step(stream)
        pre_ms, _ = binding.tpmlp_profile_end()
        timed_kinds = sorted(pre_ms, key=lambda k: -pre_ms[k])[:1]
        timed_kinds = [k for k in timed_kinds if pre_ms[k] > 0]
    barrier(dist, torch)
    sampler = ClockSampler(gpu_selector(torch, local))
    sampler.start()
    time.sleep(0.5)
    if timed_kinds:
        binding.tpmlp_profile_begin_kinds(4 * args.steps + 16, timed_kinds)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(dist, torch)
    e0.record(stream)
    for _ in range(args.steps):
        if graph is None:
            run.step(stream)
        else:
            graph.replay()
    e1.record(stream)
    barrier(dist, torch)
    clocks = sampler.stop()
    live_ms, live_count = binding.tpmlp_profile_end() if timed_kinds else ({}, {})
    # every kind's time from eager steps after the timed region (the
    # per-kernel table and shares), scaled to the timed steps; the kinds timed
    # live keep their timed-region figures
    prof_steps = min(args.steps, 50)
    binding.tpmlp_profile_begin(16 * prof_steps + 16)
    for _ in range(prof_steps):
        run.step(stream)
    kms, kcount = binding.tpmlp_profile_end()
    scale = args.steps / prof_steps
    kms = {k: v * scale for k, v in kms.items()}
    kcount = {k: int(round(v * scale)) for k, v in kcount.items()}
    for k in (timed_kinds or []):
        if live_count.get(k):
            kms[k] = live_ms[k]
            kcount[k] = live_count[k]
    st = binding.tpmlp_sync_check(stream)
    if st != binding.TPMLP_OK:
        raise RuntimeError(f"timed loop failed: {binding.tpmlp_status_string(st)}")
    ms = max_over_ranks(dist, torch, e0.elapsed_time(e1))
    value = flops_step * args.steps * world / (ms / 1e3) / 1e12
    tokens_s = T * args.steps * world / (ms / 1e3)

    peaks, peak_src = load_peaks()
    # the peak that matches how long the timed region ran
    timed_s = ms / 1e3
    peak_key = "bf16_tflops_sustained" if timed_s >= BURST_MAX_S else "bf16_tflops"
    # dominant kernel: the kernel kind with the largest share of device time
    total_k = sum(kms.values())
    kernels = {}
    for name in kms:
        if kcount[name]:
            kernels[name] = {"launches": kcount[name], "ms_per_launch": kms[name] / kcount[name],
                             "share": kms[name] / total_k if total_k else None}
    # dominant kernel: the kind timed live
    dom = max(timed_kinds or kernels, key=lambda k: kms[k])
    for k in kernels:
        kernels[k]["timed"] = ("live, in the timed region" if k in (timed_kinds or [])
                               else f"{prof_steps} eager steps after the timed region")
    if dom in run.gemm_kinds:
        achieved = run.gemm_flops / (kernels[dom]["ms_per_launch"] / 1e3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved,
                "peak": peaks[peak_key], "unit": "TFLOP/s",
                "frac": achieved / peaks[peak_key],
                "frac_of_burst": achieved / peaks["bf16_tflops"],
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                "traffic": measured_traffic(dom, w.name),
                "peak_source": f"{peak_src} {peak_key}: the timed region lasted {timed_s:.2f} s "
                               f"({'at least' if timed_s >= BURST_MAX_S else 'under'} "
                               f"{BURST_MAX_S:g} s)",
                "flops_per_launch": run.gemm_flops}
    else:
        achieved = run.colsum_bytes / 1e9 / (kms[dom] / args.steps / 1e3)
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                "peak_source": f"{peak_src} hbm_gbs"}
    if "bias_grad" in kernels:
        cs_ms = kms["bias_grad"] / args.steps
        kernels["bias_grad"]["gb_per_s"] = run.colsum_bytes / (cs_ms / 1e3) / 1e9
        kernels["bias_grad"]["frac_of_hbm"] = kernels["bias_grad"]["gb_per_s"] / peaks["hbm_gbs"]
    for name, attr in (("layernorm_fwd", "ln_fwd_bytes"), ("layernorm_bwd", "ln_bwd_bytes"),
                       ("dropout_bwd", "dropout_bytes")):
        if name in kernels and hasattr(run, attr):
            per_step = kms[name] / args.steps
            kernels[name]["gb_per_s"] = getattr(run, attr) / (per_step / 1e3) / 1e9
            kernels[name]["frac_of_hbm"] = kernels[name]["gb_per_s"] / peaks["hbm_gbs"]
    for name in run.gemm_kinds:
        if name in kernels:
            kernels[name]["tflops"] = run.gemm_flops / (kernels[name]["ms_per_launch"] / 1e3) / 1e12
    launches_per_step = sum(kcount.values()) / args.steps

    # The same eager steps without the per-kernel event pairs (two event
    # records per launch cost host time that layers of a few hundred tokens see
    # in their step time); reported beside the main line, not instead of it.
    plain_events = None
    if graph is None:
        n_plain = min(args.steps, 200)
        e6 = torch.cuda.Event(enable_timing=True)
        e7 = torch.cuda.Event(enable_timing=True)
        barrier(dist, torch)
        e6.record(stream)
        for _ in range(n_plain):
            run.step(stream)
        e7.record(stream)
        barrier(dist, torch)
        ms_plain = max_over_ranks(dist, torch, e6.elapsed_time(e7))
        plain_events = {"value": flops_step * n_plain * world / (ms_plain / 1e3) / 1e12,
                        "unit": "TFLOP/s", "ms_per_step": ms_plain / n_plain, "steps": n_plain}

    # Sustained sub-record: at least SUSTAINED_MIN_S of back-to-back steps, long
    # enough for the power cap to set the clock, with its own clock record.
    sustained = None
    if not args.no_sustained:
        n_sus = max(args.steps, int(SUSTAINED_MIN_S * 1e3 / (ms / args.steps)) + 1)
        sampler_s = ClockSampler(gpu_selector(torch, local))
        sampler_s.start()
        time.sleep(0.5)
        e4 = torch.cuda.Event(enable_timing=True)
        e5 = torch.cuda.Event(enable_timing=True)
        barrier(dist, torch)
        e4.record(stream)
        for _ in range(n_sus):
            if graph is None:
                run.step(stream)
            else:
                graph.replay()
        e5.record(stream)
        barrier(dist, torch)
        clocks_s = sampler_s.stop()
        st = binding.tpmlp_sync_check(stream)
        if st != binding.TPMLP_OK:
            raise RuntimeError(f"sustained loop failed: {binding.tpmlp_status_string(st)}")
        ms_s = max_over_ranks(dist, torch, e4.elapsed_time(e5))
        v_s = flops_step * n_sus * world / (ms_s / 1e3) / 1e12
        sustained = {"value": v_s, "unit": "TFLOP/s", "steps": n_sus, "seconds": ms_s / 1e3,
                     "ms_per_step": ms_s / n_sus,
                     "tokens_per_s": T * n_sus * world / (ms_s / 1e3),
                     "frac_of_sustained_peak": v_s / world / peaks["bf16_tflops_sustained"],
                     "frac_of_burst_peak": v_s / world / peaks["bf16_tflops"],
                     "clocks": clocks_s,
                     "gpu_launches": int(round(launches_per_step * n_sus))}

    # End to end through the C ABI with host buffers.  Every step uploads its
    # inputs (the block: X and dZ; a linear layer: X and dY) from pinned host
    # memory and downloads its forward and backward results.  Uploads and
    # downloads run on two more streams with double-buffered device
    # activations, so the upload of step i+1 overlaps step i's kernels and the
    # downloads of step i overlap step i+1's, as a training loop that
    # prefetches its next batch would.
    e2e = None
    if not args.no_e2e:
        up_stream = torch.cuda.Stream(dev)
        down_stream = torch.cuda.Stream(dev)
        names = run.ins + run.outs
        host_in = {k: [x.cpu().pin_memory() for x in run.buffers(k)] for k in run.ins}
        host_out = {k: [torch.empty_like(x, device="cpu").pin_memory() for x in run.buffers(k)]
                    for k in run.outs}
        bufs = []
        for b in range(2):
            bufs.append({k: [torch.empty_like(x) for x in run.buffers(k)] for k in names})
        ev = {k: [torch.cuda.Event() for _ in range(2)]
              for k in ("in_ready", "fwd_done", "bwd_done", "out_done")}
        fwd_out, bwd_out = run.outs

        def e2e_steps(n):
            for i in range(n):
                b = i & 1
                B = bufs[b]
                with torch.cuda.stream(up_stream):
                    if i >= 2:  # step i-2 is done with this buffer set
                        up_stream.wait_event(ev["out_done"][b])
                    for k in run.ins:
                        for d, h in zip(B[k], host_in[k]):
                            d.copy_(h, non_blocking=True)
                    ev["in_ready"][b].record(up_stream)
                stream.wait_event(ev["in_ready"][b])
                run.forward(B, stream)
                ev["fwd_done"][b].record(stream)
                run.backward(B, stream)
                ev["bwd_done"][b].record(stream)
                with torch.cuda.stream(down_stream):
                    down_stream.wait_event(ev["fwd_done"][b])
                    for h, d in zip(host_out[fwd_out], B[fwd_out]):
                        h.copy_(d, non_blocking=True)
                    down_stream.wait_event(ev["bwd_done"][b])
                    for h, d in zip(host_out[bwd_out], B[bwd_out]):
                        h.copy_(d, non_blocking=True)
                    ev["out_done"][b].record(down_stream)

        e2e_steps(2)
        torch.cuda.synchronize(dev)
        barrier(dist, torch)
        e2 = torch.cuda.Event(enable_timing=True)
        e3 = torch.cuda.Event(enable_timing=True)
        e2.record(stream)
        up_stream.wait_event(e2)  # the first upload starts inside the timed region
        down_stream.wait_event(e2)
        e2e_steps(args.e2e_steps)
        stream.wait_stream(up_stream)
        stream.wait_stream(down_stream)  # ... and the last download ends inside it
        e3.record(stream)
        barrier(dist, torch)
        st = binding.tpmlp_sync_check(stream)
        if st != binding.TPMLP_OK:
            raise RuntimeError(f"e2e loop failed: {binding.tpmlp_status_string(st)}")
        for k in run.outs:
            if not torch.equal(host_out[k][0], run.buffers(k)[0].cpu()):
                raise RuntimeError(f"e2e output {k} differs from the device-resident step")
        ms_e2e = max_over_ranks(dist, torch, e2.elapsed_time(e3))
        e2e = {"value": flops_step * args.e2e_steps * world / (ms_e2e / 1e3) / 1e12,
               "unit": "TFLOP/s",
               "h2d_bytes_per_step": sum(x.numel() * x.element_size()
                                         for k in run.ins for x in host_in[k]),
               "d2h_bytes_per_step": sum(x.numel() * x.element_size()
                                         for k in run.outs for x in host_out[k]),
               "tokens_per_s": T * args.e2e_steps * world / (ms_e2e / 1e3),
               "steps": args.e2e_steps,
               "overlap": "uploads and downloads on two more streams, double-buffered activations"}

    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline(w, run.inputs, args.cpu_seconds, args.sp_layer)
        cublas = None
        if args.cublas and hasattr(w, "hidden"):
            cublas = cublas_reference(w, torch, dev, steps=args.steps)
            if not args.sp_layer:
                cublas["torch_block"] = torch_block_reference(w, run.inputs, torch, dev,
                                                              steps=args.steps)
        theo = theoretical_peak_tflops(torch, dev)
        line = {"metric": run.metric, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": run.config(),
                "tokens_per_s": tokens_s,
                "pct_of_bf16_peak": {"burst": value / world / peaks["bf16_tflops"],
                                     "sustained": value / world / peaks["bf16_tflops_sustained"],
                                     "source": peak_src,
                                     "theoretical": (value / world / theo["tflops"]) if theo else None,
                                     "theoretical_peak": theo},
                "roofline": roof, "kernels": kernels, "sustained": sustained,
                "eager_without_kernel_events": plain_events,
                "cpu_baseline": cpu, "e2e": e2e,
                "cublas_reference": cublas,
                "clocks": clocks, "gpu_launches": int(sum(kcount.values())),
                "cuda_graph": bool(args.graph),
                "kernel_timing": (f"CUDA events around each launch of {timed_kinds} inside the "
                                  f"timed region (the kind with the most device time in a "
                                  f"{PRE_STEPS}-step profiled pass before it); the other kinds from "
                                  f"{prof_steps} eager steps after it"
                                  if graph is None else
                                  "CUDA events around each launch of eager steps run after the "
                                  "timed region (replays of the captured step carry no events)"),
                "gpu_launches_per_step": launches_per_step}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse_args()
    import torch
    if args.impl == "reference":
        run_reference(args, torch)
    else:
        run_ours(args, torch)


if __name__ == "__main__":
    main()
