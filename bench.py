#!/usr/bin/env python3
"""Throughput of the MLP training step on GB300, as one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Workloads (synthetic, seeded inputs; see synth.py):
  stack         11 MLP blocks over 262,144 tokens, MSE loss, fwd + bwd + momentum SGD
                (default: the largest single-GPU configuration)
  mlp784_epoch  784-256-10 MLP, ReLU hidden, bf16 tensor-core path, one epoch of 6,000
                images = 46 steps of batch 128 + 1 of 112
  mlp784_fp32   same network, fp32 SIMT path, one step of batch 128
  mlp_wide      1024-8192-8192-1000 MLP, batch 16,384, bf16 operands, fp32 master weights
  mlp784_epoch_f16, mlp_wide_f16
                the same two workloads with fp16 operands (FP16 in, FP32 accumulate)
  block         one RMSNorm -> gate -> LeakyReLU^2 -> down -> residual block, fwd + bwd,
                65,536 tokens x 512
  attn_prep     fused attention preprocessing (RMSNorm -> QKV -> QK norm -> RoPE -> gain),
                65,536 tokens x 512, 8 query / 4 key-value heads of 64
  hbm           the memory-bound kernels (SGD, MSE, softmax cross entropy, column sum,
                input cast) once each at full-config sizes; value = their total bytes
                per second

A bench "step" is one pass of the whole training step of the workload over its
batch (for mlp784_epoch: the whole epoch).  The timed region is K steps, each
bracketed by CUDA events on the launching stream, with an L2 flush (a 256 MiB
write) between steps outside the events, and a barrier plus device
synchronisation on both sides; the value is the maximum over ranks.  With N > 1
every rank runs an independent replica (the step has no data-parallel
exchange), so scaling is weak.

`--impl reference` times the fp64 CPU oracle (the deliberately slow checker)
on the same workload, each step a bounded sample, on the host cores of rank 0.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "training samples/s (tokens/s) per step on 1 GB300; % of BF16 tensor/HBM roofline"
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ environment

def rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.15)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ roofline helpers

def parse_kernel(name):
    """'gemm_tc_bn256[M,N,K]' -> ('gemm_tc_bn256', (M, N, K))."""
    if "[" in name:
        base, rest = name.split("[", 1)
        return base, tuple(int(v) for v in rest.rstrip("]").split(","))
    return name, ()


def algorithmic_work(name):
    """(bound, units per launch) from the kernel's recorded shape.

    GEMMs: 2 M N K flops.  Memory-bound kernels: the bytes they must move.
    """
    base, sh = parse_kernel(name)
    if base == "gemm_simt":
        M_, N, K = sh
        return "alu", 2.0 * M_ * N * K   # fp32 FMA on the CUDA cores, not the tensor cores
    if base.startswith("gemm"):
        M_, N, K = sh
        return "tensor", 2.0 * M_ * N * K
    if base == "step_program":
        steps, flops_per_step, _ = sh          # whole training steps, GEMM flops only
        return "tensor", float(steps) * flops_per_step
    if base.startswith("block_fwd"):
        T, d, h = sh
        return "tensor", 4.0 * T * d * h
    if base.startswith("block_bwd_act"):
        T, d, h = sh
        return "tensor", 2.0 * T * d * h      # dA = dY W_down^T; the u recompute is not credited
    if base.startswith("attn_prep_gemm"):
        M_, N, K = sh
        return "tensor", 2.0 * M_ * N * K     # the QKV projection; the epilogue is not credited
    if base == "row_rstd":
        T, d = sh[0], sh[1]
        return "hbm", 2.0 * T * d + 4.0 * T
    if base == "rmsnorm_bwd":
        return "hbm", 4100.0 * sh[0]          # per token: dn', x, dy, dx bf16 + rstd
    if base == "sgd":
        return "hbm", 22.0 * sh[0]        # read w, g, v; write w, v (fp32) + bf16 shadow
    if base == "cast":
        return "hbm", 3.0 * sh[0]         # byte in, bf16 out
    if base == "xent":
        B, C = sh[0], sh[1]
        return "hbm", B * C * (4.0 + 2.0) + 8.0 * B
    if base == "colsum":
        r, c = sh[0], sh[1]
        return "hbm", 2.0 * r * c + 4.0 * c
    if base == "mse":
        return "hbm", 6.0 * sh[0]
    return "hbm", 0.0


# ------------------------------------------------------------------ workloads

class Workload:
    name = ""
    unit = "samples/s"
    samples_per_step = 1
    dtype = "bf16"
    config = {}
    # a step of tens of milliseconds, repeated back to back for seconds: the
    # tensor-core roofline takes the sustained (power-capped) peak
    sustained = False
    # algorithmic (credited) GEMM flops of one bench step; recomputation is
    # not credited
    credited_flops_per_step = 0.0

    def setup(self):
        raise NotImplementedError

    def step(self):
        raise NotImplementedError

    def step_e2e(self):
        raise NotImplementedError

    h2d_bytes = 0
    d2h_bytes = 0
    launches_per_step = 0
    # End to end with the next step's input copies overlapping the current
    # step (a data loader's prefetch): (host attribute, device attribute) of
    # every input the step reads, and the result read back after each step.
    # Only for workloads whose inputs and working set are far above L2.
    e2e_inputs = ()

    def e2e_result(self):
        """(device tensor, pinned host tensor) of the per-step result."""
        raise NotImplementedError

    def check(self):
        pass


def capture_graph(wl):
    """A CUDA graph of one eager step of the workload (its current buffers)."""
    import torch
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            wl.step_eager()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def e2e_slots(wl):
    """Two input-buffer sets, each with a graph of the step over it: slot 0 is
    the workload's own, slot 1 a second copy of every input."""
    import torch
    own = {d: getattr(wl, d) for _, d in wl.e2e_inputs}
    slots = [(own, wl.graph)]
    second = {d: torch.empty_like(t).copy_(t) for d, t in own.items()}
    for d, t in second.items():
        setattr(wl, d, t)
    wl.step_eager()  # warm the second buffers' tensor maps outside the capture
    torch.cuda.synchronize()
    slots.append((second, capture_graph(wl)))
    for d, t in own.items():
        setattr(wl, d, t)
    return slots


def timed_e2e_pipelined(wl, slots, steps, sync_barrier):
    """Wall time (ms, CUDA events) of `steps` end-to-end steps: every step
    copies its inputs from pinned host memory (a second stream, into the slot
    the step before last has released), runs the step's graph once its copies
    have landed, and reads its result back; step k + 1's copies overlap step
    k's kernels."""
    import torch
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    freed = [torch.cuda.Event(), torch.cuda.Event()]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    dev_out, host_out = wl.e2e_result()
    sync_barrier()
    start.record(comp)
    copy.wait_event(start)
    for k in range(steps):
        i = k & 1
        bufs, graph = slots[i]
        with torch.cuda.stream(copy):
            if k >= 2:
                copy.wait_event(freed[i])
            for h, d in wl.e2e_inputs:
                bufs[d].copy_(getattr(wl, h), non_blocking=True)
            ready[i].record(copy)
        comp.wait_event(ready[i])
        graph.replay()
        freed[i].record(comp)
        host_out.copy_(dev_out, non_blocking=True)
    end.record(comp)
    sync_barrier()
    return start.elapsed_time(end)


class MLP784Epoch(Workload):
    """784-256-10, bf16 (or fp16) tensor-core path, one epoch (6,000 images,
    47 steps); the fp32 form is one step of 128 on the SIMT path."""
    name = "mlp784_epoch"
    unit = "samples/s"
    dtype = "bf16"

    def __init__(self, prec_name="bf16", n_images=6000, batch=128):
        self.prec_name = prec_name
        if prec_name == "fp32":
            self.name = "mlp784_fp32"
            self.dtype = "f32"
        elif prec_name == "fp16":
            self.name = "mlp784_epoch_f16"
            self.dtype = "f16"
        self.n_images = n_images
        self.batch = batch
        self.n_steps = (n_images + batch - 1) // batch
        self.samples_per_step = n_images
        self.config = {"workload": "784-256-10 MLP, ReLU hidden, %s operands, fp32 accumulation "
                                   "and master weights; one epoch = %d synthetic images "
                                   "(%d steps of batch %d, last partial), lr 0.1, momentum 0.9"
                       % (prec_name, n_images, (n_images + batch - 1) // batch, batch),
                       "dims": [784, 256, 10], "batch": batch, "images_per_epoch": n_images,
                       "train_steps_per_bench_step": (n_images + batch - 1) // batch,
                       "cuda_graph": True, "l2": "flushed between timed steps (256 MiB write)"}

    def setup(self):
        import torch
        import mlp_step_gb300 as M
        from mlp_step_gb300 import synth
        self.M = M
        dims = [784, 256, 10]
        prec = {"bf16": M.MLP_PREC_BF16, "fp16": M.MLP_PREC_FP16}.get(self.prec_name,
                                                                      M.MLP_PREC_FP32)
        p0 = synth.mlp_flat_params(dims)
        self.net = M.MLP(dims, prec=prec, max_batch=self.batch, params=torch.from_numpy(p0))
        xb = synth.images_u8(self.n_images, 784)
        y = synth.labels(self.n_images, 10)
        self.x_host = torch.from_numpy(xb).pin_memory()
        self.y_host = torch.from_numpy(y).pin_memory()
        self.x = self.x_host.cuda()
        self.y = self.y_host.cuda()
        self.n_steps = (self.n_images + self.batch - 1) // self.batch
        # per training step of b rows: forward and weight-gradient GEMMs of
        # both layers, and the hidden layer's input gradient (the first
        # layer's input gradient is not computed)
        self.credited_flops_per_step = float(sum(
            2.0 * min(self.batch, self.n_images - i * self.batch) * (
                2 * (784 * 256 + 256 * 10) + 256 * 10) for i in range(self.n_steps)))
        self.losses = torch.zeros(self.n_steps, dtype=torch.float32, device="cuda")
        self.losses_host = torch.zeros(self.n_steps, dtype=torch.float32).pin_memory()
        self.h2d_bytes = xb.nbytes + y.nbytes
        self.d2h_bytes = self.n_steps * 4
        # warm the kernels once eagerly (tensor maps, function attributes), then
        # capture the epoch into one CUDA graph
        self._epoch()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        c0 = M.launch_count()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(self.graph, stream=s):
                self._epoch()
        torch.cuda.current_stream().wait_stream(s)
        self.launches_per_step = M.launch_count() - c0
        torch.cuda.synchronize()
        # the end-to-end form as one graph as well: the input copies from
        # pinned host memory, the epoch and the read-back of its losses
        self.graph_e2e = torch.cuda.CUDAGraph()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(self.graph_e2e, stream=s):
                self._e2e_eager()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.train_step_launches = self._count_train_step_launches(dims, prec, p0, xb, y)

    def _count_train_step_launches(self, dims, prec, p0, xb, y):
        """Kernel launches of one training step of batch 128: the library's
        train-step call (one step program where it fits) against the same step
        through the separate public calls (forward, softmax cross entropy,
        backward, momentum SGD)."""
        import torch
        M = self.M
        if prec == M.MLP_PREC_FP32:
            return None
        net = M.MLP(dims, prec=prec, max_batch=self.batch, params=torch.from_numpy(p0))
        x = torch.from_numpy(xb[:self.batch]).cuda()
        lab = torch.from_numpy(y[:self.batch]).cuda()
        loss = torch.zeros(1, device="cuda")
        logits = torch.zeros(self.batch, 10, device="cuda")
        dl = torch.zeros(self.batch, 16, dtype=net.shadow.dtype, device="cuda")
        ws = torch.empty(M.softmax_xent_workspace_bytes(self.batch, 10), dtype=torch.uint8,
                         device="cuda")

        def unfused_step():
            net.forward(x, logits)
            M.softmax_xent_fwd_bwd(logits, lab, loss, dlogits=dl, workspace=ws)
            net.backward(dl, self.batch)
            net.sgd_step(0.1, 0.9)

        # the first call of each form also writes the handle's ones columns
        # once; count a later one
        net.train_step(x, lab, 0.1, 0.9, loss_out=loss)
        unfused_step()
        c0 = M.launch_count()
        net.train_step(x, lab, 0.1, 0.9, loss_out=loss)
        fused = M.launch_count() - c0
        c0 = M.launch_count()
        unfused_step()
        unfused = M.launch_count() - c0
        torch.cuda.synchronize()
        return {"fused": fused, "unfused": unfused,
                "unfused_calls": "mlp_forward, softmax_xent_fwd_bwd, mlp_backward, mlp_sgd_step"}

    def _e2e_eager(self):
        self.x.copy_(self.x_host, non_blocking=True)
        self.y.copy_(self.y_host, non_blocking=True)
        self._epoch()
        self.losses_host.copy_(self.losses, non_blocking=True)

    def _epoch(self):
        # the library's epoch call: the same steps in order, the full-size ones
        # in one launch where the step program fits
        self.net.train_epoch(self.x, self.y, 0.1, 0.9, self.batch, losses_out=self.losses)

    def step(self):
        self.graph.replay()

    def step_eager(self):
        self._epoch()

    def step_e2e(self):
        self.graph_e2e.replay()

    def check(self):
        import torch
        torch.cuda.synchronize()
        last = self.losses.cpu().numpy()
        assert np.all(np.isfinite(last)), "non-finite loss"
        assert self.M.get_device_status() == self.M.MLP_OK

    # --- reference arm and CPU baseline: the fp64 oracle
    def oracle_sample(self, budget_s):
        import oracle
        from mlp_step_gb300 import synth
        dims = [784, 256, 10]
        p = synth.mlp_flat_params(dims).astype(np.float64)
        v = np.zeros_like(p)
        xb = synth.images_u8(self.n_images, 784).astype(np.float32) / np.float32(255)
        y = synth.labels(self.n_images, 10)
        t0 = time.perf_counter()
        done = 0
        steps = 0
        while True:
            for i in range(self.n_steps):
                a = i * self.batch
                b = min(self.n_images, a + self.batch)
                _, p, v, _ = oracle.mlp_train_step(dims, p, v, xb[a:b].astype(np.float64),
                                                   y[a:b], 0.1, 0.9,
                                                   points={"bf16": 1, "fp16": 2}.get(
                                                       self.prec_name, 0))
                done += b - a
                steps += 1
                if time.perf_counter() - t0 >= budget_s:
                    break
            if time.perf_counter() - t0 >= budget_s:
                break
        dt = time.perf_counter() - t0
        return done, dt, "%d oracle training steps (%d images of the epoch's stream), fp64" % (
            steps, done)


class WideMLP(Workload):
    """1024-8192-8192-1000, batch 16,384, bf16 (or fp16) operands, fp32 master
    weights."""
    name = "mlp_wide"
    unit = "samples/s"
    dtype = "bf16"

    def __init__(self, batch=16384, prec_name="bf16"):
        self.dims = [1024, 8192, 8192, 1000]
        self.batch = batch
        self.prec_name = prec_name
        if prec_name == "fp16":
            self.name = "mlp_wide_f16"
            self.dtype = "f16"
        self.samples_per_step = self.batch
        self.sustained = True
        d = self.dims
        fwd = sum(2.0 * batch * d[i] * d[i + 1] for i in range(3))
        dx = sum(2.0 * batch * d[i] * d[i + 1] for i in range(1, 3))
        self.credited_flops_per_step = 2 * fwd + dx   # forward, dW, dX of layers 2 and 3
        self.config = {"workload": "1024-8192-8192-1000 MLP, ReLU, " + prec_name +
                                   " weights/activations, "
                                   "fp32 master weights and accumulation, batch 16384, inputs "
                                   "N(0,1), labels uniform 0..999, SGD momentum lr 0.01 m 0.9; "
                                   "one full fwd + bwd + update step" + (
                                       "" if batch == 16384 else " (batch %d)" % batch),
                       "dims": self.dims, "batch": self.batch, "cuda_graph": True,
                       "l2": "flushed between timed steps (256 MiB write); working set > L2"}

    def setup(self):
        import torch
        import mlp_step_gb300 as M
        from mlp_step_gb300 import synth
        self.M = M
        p0 = synth.mlp_flat_params(self.dims)
        f16 = self.prec_name == "fp16"
        self.net = M.MLP(self.dims, prec=M.MLP_PREC_FP16 if f16 else M.MLP_PREC_BF16,
                         max_batch=self.batch, params=torch.from_numpy(p0))
        X = synth.normal_f32((self.batch, self.dims[0]), synth.STREAM_X)
        y = synth.labels(self.batch, self.dims[-1])
        self.x_host = torch.from_numpy(X).to(torch.float16 if f16 else torch.bfloat16).pin_memory()
        self.y_host = torch.from_numpy(y).pin_memory()
        self.x = self.x_host.cuda()
        self.y = self.y_host.cuda()
        self.loss = torch.zeros(4, device="cuda")
        self.loss_host = torch.zeros(4).pin_memory()
        self.h2d_bytes = self.x_host.numel() * 2 + self.y_host.numel() * 4
        self.d2h_bytes = 4
        self.step_eager()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        c0 = M.launch_count()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(self.graph, stream=s):
                self.step_eager()
        torch.cuda.current_stream().wait_stream(s)
        self.launches_per_step = M.launch_count() - c0
        torch.cuda.synchronize()

    def step_eager(self):
        self.net.train_step(self.x, self.y, 0.01, 0.9, loss_out=self.loss)

    def step(self):
        self.graph.replay()

    def step_e2e(self):
        self.x.copy_(self.x_host, non_blocking=True)
        self.y.copy_(self.y_host, non_blocking=True)
        self.graph.replay()
        self.loss_host.copy_(self.loss, non_blocking=True)

    e2e_inputs = (("x_host", "x"), ("y_host", "y"))

    def e2e_result(self):
        return self.loss, self.loss_host

    def check(self):
        import torch
        torch.cuda.synchronize()
        assert np.isfinite(self.loss[0].item()), "non-finite loss"
        assert self.M.get_device_status() == self.M.MLP_OK

    def oracle_sample(self, budget_s):
        import oracle
        from mlp_step_gb300 import synth
        p = synth.mlp_flat_params(self.dims).astype(np.float64)
        v = np.zeros_like(p)
        rows = 4
        X = synth.normal_f32((rows, self.dims[0]), synth.STREAM_X).astype(np.float64)
        y = synth.labels(rows, self.dims[-1])
        t0 = time.perf_counter()
        done = 0
        steps = 0
        while True:
            _, p, v, _ = oracle.mlp_train_step(self.dims, p, v, X, y, 0.01, 0.9)
            done += rows
            steps += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        dt = time.perf_counter() - t0
        return done, dt, ("%d oracle training steps of batch %d (fp64; the full-batch step "
                          "would take hours)" % (steps, rows))


class BlockStep(Workload):
    """One MLP block forward + backward over 65,536 tokens (d 512, hidden 1536)."""
    name = "block"
    unit = "tokens/s"
    dtype = "bf16"

    def __init__(self, T=65536):
        self.T, self.d, self.h = T, 512, 1536
        self.samples_per_step = T
        # six GEMMs of 2 T d h: gate and down forward; dA, dW_down, dW_gate, dn
        self.credited_flops_per_step = 6 * 2.0 * T * 512 * 1536
        self.config = {"workload": "transformer MLP block fwd+bwd: x[%d tokens, 512] bf16 "
                                   "N(0,1), RMSNorm (eps 1e-6, gain 1) -> W_gate 512x1536 -> "
                                   "LeakyReLU(0.5)^2 -> W_down 1536x512 -> residual, weights "
                                   "N(0,0.02), upstream grad N(0,1); the 1536-wide "
                                   "intermediate stays on chip in the forward" % T,
                       "tokens": T, "d": 512, "hidden": 1536, "cuda_graph": True,
                       "l2": "flushed between timed steps (256 MiB write)"}

    def setup(self):
        import torch
        import mlp_step_gb300 as M
        from mlp_step_gb300 import synth
        self.M = M
        T, d, h = self.T, self.d, self.h
        bf = torch.bfloat16
        self.x_host = torch.from_numpy(synth.normal_f32((T, d), synth.STREAM_BLOCK_X)).to(bf)
        self.x_host = self.x_host.pin_memory()
        self.dy_host = torch.from_numpy(synth.normal_f32((T, d), synth.STREAM_BLOCK_DY)).to(bf)
        self.dy_host = self.dy_host.pin_memory()
        self.x = self.x_host.cuda()
        self.dy = self.dy_host.cuda()
        self.wg = torch.from_numpy(synth.normal_f32((d, h), synth.STREAM_BLOCK_WG,
                                                    std=0.02)).to(bf).cuda()
        self.wd = torch.from_numpy(synth.normal_f32((h, d), synth.STREAM_BLOCK_WD,
                                                    std=0.02)).to(bf).cuda()
        self.y = torch.empty(T, d, dtype=bf, device="cuda")
        self.r = torch.empty(T, device="cuda")
        self.dx = torch.empty(T, d, dtype=bf, device="cuda")
        self.dwg = torch.empty(d, h, device="cuda")
        self.dwd = torch.empty(h, d, device="cuda")
        self.ws = torch.empty(M.mlp_block_workspace_bytes(T, d, h), dtype=torch.uint8,
                              device="cuda")
        self.dx_host = torch.empty(4, dtype=bf).pin_memory()
        self.h2d_bytes = 2 * T * d * 2
        self.d2h_bytes = 8
        self.step_eager()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        c0 = M.launch_count()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(self.graph, stream=s):
                self.step_eager()
        torch.cuda.current_stream().wait_stream(s)
        self.launches_per_step = M.launch_count() - c0
        torch.cuda.synchronize()

    def step_eager(self):
        M = self.M
        M.mlp_block_fwd(self.x, self.wg, self.wd, self.y, self.r)
        M.mlp_block_bwd(self.x, self.r, self.wg, self.wd, self.dy, self.dx, self.dwg, self.dwd,
                        self.ws)

    def step(self):
        self.graph.replay()

    def step_e2e(self):
        self.x.copy_(self.x_host, non_blocking=True)
        self.dy.copy_(self.dy_host, non_blocking=True)
        self.graph.replay()
        self.dx_host.copy_(self.dx[0, :4], non_blocking=True)

    e2e_inputs = (("x_host", "x"), ("dy_host", "dy"))

    def e2e_result(self):
        return self.dx[0, :4], self.dx_host

    def check(self):
        import torch
        torch.cuda.synchronize()
        assert torch.isfinite(self.dwg).all(), "non-finite gradient"
        assert self.M.get_device_status() == self.M.MLP_OK

    def oracle_sample(self, budget_s):
        import oracle
        from mlp_step_gb300 import synth
        T = 64
        x = synth.normal_f32((T, self.d), synth.STREAM_BLOCK_X).astype(np.float64)
        dy = synth.normal_f32((T, self.d), synth.STREAM_BLOCK_DY).astype(np.float64)
        wg = synth.normal_f32((self.d, self.h), synth.STREAM_BLOCK_WG, std=0.02)
        wd = synth.normal_f32((self.h, self.d), synth.STREAM_BLOCK_WD, std=0.02)
        t0 = time.perf_counter()
        done = 0
        n = 0
        while True:
            oracle.block_fwd(x, wg, wd, 1e-6, 0.5)
            oracle.block_bwd(x, wg, wd, dy, 1e-6, 0.5)
            done += T
            n += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        dt = time.perf_counter() - t0
        return done, dt, "%d oracle block fwd+bwd passes over %d tokens (fp64)" % (n, T)


class AttnPrep(Workload):
    """Fused attention preprocessing over 65,536 tokens: RMSNorm -> QKV
    projection -> QK norm -> partial RoPE -> q gain."""
    name = "attn_prep"
    unit = "tokens/s"
    dtype = "bf16"

    def __init__(self, T=65536, seq_len=1024, n_q=8, n_kv=4, rope_dims=32):
        self.T, self.d, self.L = T, 512, seq_len
        self.n_q, self.n_kv, self.R = n_q, n_kv, rope_dims
        self.N = (n_q + 2 * n_kv) * 64
        self.samples_per_step = T
        self.credited_flops_per_step = 2.0 * T * 512 * self.N
        self.config = {"workload": "fused attention preprocessing: x[%d tokens, 512] bf16 N(0,1) "
                                   "(%d sequences of %d), RMSNorm (eps 1e-6, gain 1) -> W_qkv "
                                   "512x%d (%d query, %d key, %d value heads of 64, N(0, 512^-1/2)) "
                                   "-> QK RMSNorm -> rotate-half RoPE on %d of 64 dims (base "
                                   "10000) -> q gain U(0.5, 1.5); forward only"
                                   % (T, T // seq_len, seq_len, self.N, n_q, n_kv, n_kv,
                                      rope_dims),
                       "tokens": T, "d": 512, "n_q_heads": n_q, "n_kv_heads": n_kv,
                       "head_dim": 64, "rope_dims": rope_dims, "seq_len": seq_len,
                       "cuda_graph": True, "l2": "flushed between timed steps (256 MiB write)"}

    def setup(self):
        import torch
        import mlp_step_gb300 as M
        from mlp_step_gb300 import synth
        self.M = M
        bf = torch.bfloat16
        self.x_host = torch.from_numpy(synth.normal_f32((self.T, self.d),
                                                        synth.STREAM_GENERIC + 40)).to(bf)
        self.x_host = self.x_host.pin_memory()
        self.x = self.x_host.cuda()
        self.w = torch.from_numpy(synth.normal_f32((self.d, self.N), synth.STREAM_GENERIC + 41,
                                                   std=self.d ** -0.5)).to(bf).cuda()
        self.gain = torch.from_numpy(synth.uniform_f32((self.n_q,), synth.STREAM_GENERIC + 42,
                                                       lo=0.5, hi=1.5)).cuda()
        self.out = torch.empty(self.T, self.N, dtype=bf, device="cuda")
        self.r = torch.empty(self.T, device="cuda")
        self.out_host = torch.empty(4, dtype=bf).pin_memory()
        self.h2d_bytes = self.T * self.d * 2
        self.d2h_bytes = 8
        self.step_eager()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        c0 = M.launch_count()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(self.graph, stream=s):
                self.step_eager()
        torch.cuda.current_stream().wait_stream(s)
        self.launches_per_step = M.launch_count() - c0
        torch.cuda.synchronize()

    def step_eager(self):
        self.M.mlp_attn_prep_fwd(self.x, self.w, self.gain, self.out, self.r, self.n_q,
                                 self.n_kv, self.R, self.L)

    def step(self):
        self.graph.replay()

    def step_e2e(self):
        self.x.copy_(self.x_host, non_blocking=True)
        self.graph.replay()
        self.out_host.copy_(self.out[0, :4], non_blocking=True)

    e2e_inputs = (("x_host", "x"),)

    def e2e_result(self):
        return self.out[0, :4], self.out_host

    def check(self):
        import torch
        torch.cuda.synchronize()
        assert torch.isfinite(self.out.float()).all(), "non-finite output"
        assert self.M.get_device_status() == self.M.MLP_OK

    def oracle_sample(self, budget_s):
        import oracle
        from mlp_step_gb300 import synth
        T = 256
        x = synth.normal_f32((T, self.d), synth.STREAM_GENERIC + 40).astype(np.float64)
        w = synth.normal_f32((self.d, self.N), synth.STREAM_GENERIC + 41, std=self.d ** -0.5)
        g = synth.uniform_f32((self.n_q,), synth.STREAM_GENERIC + 42, lo=0.5, hi=1.5)
        t0 = time.perf_counter()
        done = 0
        n = 0
        while True:
            oracle.attn_prep(x, w, g, self.n_q, self.n_kv, 64, self.R, self.L)
            done += T
            n += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        dt = time.perf_counter() - t0
        return done, dt, "%d oracle passes over %d tokens (fp64)" % (n, T)


class StackStep(Workload):
    """11 blocks over 262,144 tokens, MSE loss, full fwd + bwd + momentum SGD."""
    name = "stack"
    unit = "tokens/s"
    dtype = "bf16"

    def __init__(self, n_blocks=11, T=262144):
        self.nb, self.T, self.d, self.h = n_blocks, T, 512, 1536
        self.samples_per_step = T
        self.sustained = True
        # six 2 T d h GEMMs per block, less the first block's input-gradient
        # GEMM, which the step does not run (the stack input's gradient is
        # not an output)
        self.credited_flops_per_step = (n_blocks * 6 - 1) * 2.0 * T * 512 * 1536
        self.config = {"workload": "stack of %d MLP blocks (d 512, hidden 1536, "
                                   "LeakyReLU(0.5)^2, RMSNorm pre-norm, residual) over %d tokens "
                                   "bf16, MSE loss vs N(0,1) targets, full fwd + bwd + "
                                   "flat-buffer SGD-momentum step (lr 0.02, m 0.95)"
                                   % (n_blocks, T),
                       "blocks": n_blocks, "tokens": T, "d": 512, "hidden": 1536,
                       "cuda_graph": True, "l2": "working set far above L2; flushed as well"}

    def setup(self):
        import torch
        import mlp_step_gb300 as M
        from mlp_step_gb300 import synth
        self.M = M
        nb, T, d, h = self.nb, self.T, self.d, self.h
        bf = torch.bfloat16
        self.x_host = torch.from_numpy(synth.normal_f32((T, d), synth.STREAM_BLOCK_X)).to(bf)
        self.x_host = self.x_host.pin_memory()
        self.t_host = torch.from_numpy(synth.normal_f32((T, d), synth.STREAM_TARGET)).to(bf)
        self.t_host = self.t_host.pin_memory()
        self.x = self.x_host.cuda()
        self.t = self.t_host.cuda()
        P = M.mlp_stack_param_count(nb, d, h)
        self.params = torch.from_numpy(synth.normal_f32((P,), synth.STREAM_BLOCK_WG,
                                                        std=0.02)).cuda()
        self.vel = torch.zeros_like(self.params)
        self.grads = torch.zeros_like(self.params)
        self.shadow = self.params.to(bf)
        self.ws = torch.empty(M.mlp_stack_workspace_bytes(nb, T, d, h), dtype=torch.uint8,
                              device="cuda")
        self.loss = torch.zeros(4, device="cuda")
        self.loss_host = torch.zeros(4).pin_memory()
        self.h2d_bytes = 2 * T * d * 2
        self.d2h_bytes = 4
        self.step_eager()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        c0 = M.launch_count()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(self.graph, stream=s):
                self.step_eager()
        torch.cuda.current_stream().wait_stream(s)
        self.launches_per_step = M.launch_count() - c0
        torch.cuda.synchronize()

    def step_eager(self):
        self.M.mlp_stack_train_step(self.nb, self.T, self.d, self.h, self.x, self.t, self.params,
                                    self.vel, self.grads, self.shadow, 0.02, 0.95, self.loss,
                                    self.ws)

    def step(self):
        self.graph.replay()

    def step_e2e(self):
        self.x.copy_(self.x_host, non_blocking=True)
        self.t.copy_(self.t_host, non_blocking=True)
        self.graph.replay()
        self.loss_host.copy_(self.loss, non_blocking=True)

    e2e_inputs = (("x_host", "x"), ("t_host", "t"))

    def e2e_result(self):
        return self.loss, self.loss_host

    def check(self):
        import torch
        torch.cuda.synchronize()
        assert np.isfinite(self.loss[0].item()), "non-finite loss"
        assert self.M.get_device_status() == self.M.MLP_OK

    def oracle_sample(self, budget_s):
        import oracle
        from mlp_step_gb300 import synth
        T = 16
        x = synth.normal_f32((T, self.d), synth.STREAM_BLOCK_X).astype(np.float64)
        t = synth.normal_f32((T, self.d), synth.STREAM_TARGET).astype(np.float64)
        P = self.nb * 2 * self.d * self.h
        p = synth.normal_f32((P,), synth.STREAM_BLOCK_WG, std=0.02).astype(np.float64)
        t0 = time.perf_counter()
        done = 0
        n = 0
        while True:
            _, g, _ = oracle.stack_fwd_bwd(x, p, self.nb, self.d, self.h, 1e-6, 0.5, t)
            p, _ = oracle.sgd_momentum(p, g, np.zeros_like(p), 0.02, 0.95)
            done += T
            n += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        dt = time.perf_counter() - t0
        return done, dt, ("%d oracle stack steps over %d tokens (%d blocks, fp64)"
                          % (n, T, self.nb))


class HbmKernels(Workload):
    """The step's memory-bound kernels, each at the size it runs at in the
    largest configurations (every buffer above L2): momentum SGD over the
    stack's 17,301,504 parameters with the bf16 shadow, the mean-squared loss
    over 262,144 x 512, softmax cross entropy over 16,384 x 1000 with bf16 dZ,
    a bf16 column sum over 16,384 x 8192 and the input cast of 262,144 images
    of 1,024 bytes to bf16.  The bench step runs each once; the per-kernel
    GB/s come from the library's event timing."""
    name = "hbm"
    unit = "GB/s"
    dtype = "f32"

    def __init__(self):
        # algorithmic bytes of one step (GB): sgd 22 B per parameter; mse 6 B per
        # element; xent 4 B read + 2 B written per logit, 8 B per row; column
        # sum 2 B per element + 4 B per column; cast 1 B read + 2 B written per
        # byte; the small net's two forward GEMMs read the cast input once and
        # write their bf16 / fp32 outputs
        nb = {"sgd": 22.0 * 17301504, "mse": 6.0 * 262144 * 512,
              "xent": 6.0 * 16384 * 1000 + 8.0 * 16384, "colsum": 2.0 * 16384 * 8192 + 4 * 8192,
              "cast": 3.0 * 262144 * 1024,
              "gemm": 2.0 * 262144 * 1024 + 2.0 * 262144 * 16 * 2 + 4.0 * 262144 * 16}
        self.samples_per_step = sum(nb.values()) / 1e9
        self.config = {"workload": "memory-bound kernels at full-config sizes: sgd 17,301,504 "
                                   "params (+bf16 shadow), mse 262144x512 bf16, softmax xent "
                                   "16384x1000 fp32 -> bf16 dZ, column sum 16384x8192 bf16, "
                                   "cast 262144x1024 u8 -> bf16 (+ the 1024-16-16 net's two "
                                   "small forward GEMMs that read it); value = algorithmic "
                                   "bytes of the step / step time",
                       "algorithmic_bytes": nb,
                       "cuda_graph": True, "l2": "every buffer above L2; flushed as well"}

    def setup(self):
        import torch
        import mlp_step_gb300 as M
        from mlp_step_gb300 import synth
        self.M = M
        bf = torch.bfloat16
        n = 17301504
        self.w = torch.from_numpy(synth.normal_f32((n,), synth.STREAM_BLOCK_WG, std=0.02)).cuda()
        self.g = torch.from_numpy(synth.normal_f32((n,), synth.STREAM_GENERIC + 50,
                                                   std=1e-3)).cuda()
        self.v = torch.zeros_like(self.w)
        self.wb = self.w.to(bf)
        T, d = 262144, 512
        self.y = torch.from_numpy(synth.normal_f32((T, d), synth.STREAM_BLOCK_X)).to(bf).cuda()
        self.t = torch.from_numpy(synth.normal_f32((T, d), synth.STREAM_TARGET)).to(bf).cuda()
        self.dy = torch.empty_like(self.y)
        self.mse_ws = torch.empty(M.mse_workspace_bytes(T * d), dtype=torch.uint8, device="cuda")
        self.loss = torch.zeros(4, device="cuda")
        B, C = 16384, 1000
        self.z = torch.from_numpy(synth.normal_f32((B, C), synth.STREAM_GENERIC + 51,
                                                   std=3.0)).cuda()
        self.lab = torch.from_numpy(synth.labels(B, C)).cuda()
        self.dz = torch.empty(B, 1024, dtype=bf, device="cuda")
        self.loss_xent = torch.zeros(4, device="cuda")
        self.xent_ws = torch.empty(M.softmax_xent_workspace_bytes(B, C), dtype=torch.uint8,
                                   device="cuda")
        self.cs_x = torch.from_numpy(synth.uniform_f32((16384, 8192),
                                                       synth.STREAM_GENERIC + 52)).to(bf).cuda()
        self.cs_out = torch.empty(8192, device="cuda")
        self.cs_ws = torch.empty(max(M.mlp_colsum_workspace_bytes(16384, 8192), 16),
                                 dtype=torch.uint8, device="cuda")
        self.net = M.MLP([1024, 16, 16], prec=M.MLP_PREC_BF16, max_batch=262144)
        self.img = torch.from_numpy(synth.images_u8(262144, 1024)).cuda()
        self.logits = torch.empty(262144, 16, device="cuda")
        self.step_eager()
        torch.cuda.synchronize()
        self.graph = capture_graph(self)
        c0 = M.launch_count()
        self.step_eager()
        self.launches_per_step = M.launch_count() - c0
        torch.cuda.synchronize()

    def step_eager(self):
        M = self.M
        M.sgd_momentum_step(self.w, self.g, self.v, 1e-3, 0.9, w_bf16=self.wb)
        M.mse_loss_fwd_bwd(self.y, self.t, self.loss, self.dy, self.mse_ws)
        M.softmax_xent_fwd_bwd(self.z, self.lab, self.loss_xent, dlogits=self.dz,
                               workspace=self.xent_ws, classes=1000)
        M.mlp_colsum(self.cs_x, self.cs_out, workspace=self.cs_ws)
        self.net.forward(self.img, self.logits)

    def step(self):
        self.graph.replay()

    def step_e2e(self):
        self.graph.replay()

    def check(self):
        import torch
        torch.cuda.synchronize()
        assert self.M.get_device_status() == self.M.MLP_OK

    def oracle_sample(self, budget_s):
        import oracle
        from mlp_step_gb300 import synth
        n = 1 << 20
        w = synth.normal_f32((n,), synth.STREAM_BLOCK_WG, std=0.02).astype(np.float64)
        g = synth.normal_f32((n,), synth.STREAM_GENERIC + 50, std=1e-3).astype(np.float64)
        v = np.zeros(n)
        t0 = time.perf_counter()
        done = 0
        while time.perf_counter() - t0 < budget_s:
            w, v = oracle.sgd_momentum(w, g, v, 1e-3, 0.9)
            done += 22.0 * n
        dt = time.perf_counter() - t0
        return done / 1e9, dt, "oracle momentum SGD over 2^20 parameters (22 B each), fp64"


WORKLOADS = {
    "mlp784_epoch": lambda: MLP784Epoch("bf16"),
    "mlp784_fp32": lambda: MLP784Epoch("fp32", n_images=128),
    "mlp784_epoch_f16": lambda: MLP784Epoch("fp16"),
    "mlp_wide": WideMLP,
    "mlp_wide_f16": lambda: WideMLP(prec_name="fp16"),
    "block": BlockStep,
    "attn_prep": AttnPrep,
    "stack": StackStep,
    "hbm": HbmKernels,
}
SIZED = {"block": lambda T: BlockStep(T=T), "stack": lambda T: StackStep(T=T),
         "mlp_wide": lambda B: WideMLP(batch=B)}


# ------------------------------------------------------------------ measurement

def timed_loop(fn, steps, flush, sync_barrier, per_step=None):
    """Sum of per-step CUDA-event durations (ms) over `steps` calls of fn
    (the durations themselves appended to per_step when given)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    sync_barrier()
    for s, e in evs:
        flush.zero_()
        s.record()
        fn()
        e.record()
    sync_barrier()
    ts = [s.elapsed_time(e) for s, e in evs]
    if per_step is not None:
        per_step.extend(ts)
    return sum(ts)


def kernel_profile(wl, steps):
    """Per-kernel average durations from the library's event timing (eager)."""
    import torch
    M = wl.M
    M.timing_enable(True)
    for _ in range(steps):
        wl.step_eager()
    torch.cuda.synchronize()
    rep = M.timing_report()
    M.timing_enable(False)
    return rep


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary under profiles/, if it
    was captured on the kernel source that is built now (else None)."""
    import glob
    import hashlib
    if kernel == "gemm_simt":
        fname = "k_gemm_simt.cu"
    elif kernel.startswith("gemm") or kernel == "step_program" or kernel.startswith("attn_prep"):
        fname = "k_gemm_tc.cu"
    elif kernel.startswith("block") or kernel.startswith("rmsnorm"):
        fname = "k_block.cu"
    else:
        fname = "k_elementwise.cu"
    src = os.path.join(ROOT, "mlp_step_gb300", "csrc", fname)
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    for f in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        for line in open(f):
            parts = line.split()
            if len(parts) == 5 and parts[0] == "traffic:" and parts[1] == kernel and \
                    parts[2] == workload and parts[4] == sha:
                return float(parts[3])
    return None


def fp32_alu_tflops():
    """Peak fp32 FMA rate of the CUDA cores: SMs x 128 fp32 lanes x 2 flops per
    clock at the maximum SM clock (2070 MHz on the GB300)."""
    try:
        import torch
        sms = torch.cuda.get_device_properties(0).multi_processor_count
    except Exception:
        sms = 152
    return sms * 128 * 2 * 2.070e9 / 1e12


def roofline_entry(rep, peaks, peaks_kind, sustained=False, f16=False):
    """Roofline of the dominant kernel.  f16: the contraction runs on fp16
    operands, whose nominal dense rate equals bf16's, so the measured bf16
    peak is its denominator (times 1.0)."""
    if not rep:
        return None
    # dominant kernel kind = largest total time, aggregated over shapes
    by_base = {}
    for name, (n, ms) in rep.items():
        base, _ = parse_kernel(name)
        by_base.setdefault(base, []).append((name, n, ms))
    base = max(by_base, key=lambda b: sum(ms for _, _, ms in by_base[b]))
    entries = by_base[base]
    launches = sum(n for _, n, _ in entries)
    total_ms = sum(ms for _, _, ms in entries)
    work = 0.0
    bound = "hbm"
    for name, n, _ in entries:
        bound, w = algorithmic_work(name)
        work += w * n
    avg_ms = total_ms / launches
    per_launch = work / launches
    if bound == "tensor":
        achieved = per_launch / (avg_ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        unit = "TFLOP/s"
    elif bound == "alu":
        achieved = per_launch / (avg_ms * 1e-3) / 1e12
        peak = round(fp32_alu_tflops(), 2)
        unit = "TFLOP/s"
    else:
        achieved = per_launch / (avg_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    share = total_ms / sum(ms for _, ms in rep.values())
    return {"bound": bound, "kernel": base, "achieved": round(achieved, 3), "peak": peak,
            "unit": unit, "frac": round(achieved / peak, 5), "traffic": None,
            "peak_kind": ("derived: SMs x 128 fp32 lanes x 2 flops x 2070 MHz" if bound == "alu" else
                          peaks_kind + (" sustained" if sustained and bound == "tensor" else
                                        (" burst" if bound == "tensor" else "")) +
                          (" bf16 x 1.0 (nominal dense fp16 = bf16 rate)"
                           if bound == "tensor" and f16 else "")),
            "launches_profiled": launches, "avg_launch_ms": round(avg_ms, 6),
            "share_of_kernel_time": round(share, 4),
            "work_per_launch": per_launch}


def max_over_ranks(dist, values, device="cpu"):
    """Element-wise maximum of a list of floats over all ranks (the timing
    contract takes the slowest replica); identity without a process group."""
    if dist is None:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def run_ours(args, wl):
    import torch
    rank, world, local = rank_info()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    def sync_barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    wl.setup()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    wl.check()

    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        step_ms = []
        dev_ms = timed_loop(wl.step, args.steps, flush, sync_barrier, step_ms)
        wall = time.perf_counter() - t0
    wl.check()
    if wl.e2e_inputs:
        slots = e2e_slots(wl)
        for _ in range(2):  # warm-up of the pipelined form
            timed_e2e_pipelined(wl, slots, 2, sync_barrier)
        e2e_ms = timed_e2e_pipelined(wl, slots, args.steps, sync_barrier)
        e2e_mode = ("pipelined: step k+1's host-to-device copies overlap step k on a second "
                    "stream (inputs and working set far above L2, no flush)")
    else:
        e2e_ms = timed_loop(wl.step_e2e, args.steps, flush, sync_barrier)
        e2e_mode = "serial: copies, step, read-back per step; L2 flushed between steps"
    wl.check()

    dev_ms, e2e_ms = max_over_ranks(dist, [dev_ms, e2e_ms],
                                    device="cuda" if dist is not None and
                                    dist.get_backend() == "nccl" else "cpu")

    ms_per_step = dev_ms / args.steps
    value = wl.samples_per_step * world / (ms_per_step * 1e-3)
    e2e_value = wl.samples_per_step * world / (e2e_ms / args.steps * 1e-3)

    peaks, peaks_kind = load_peaks()
    rep = kernel_profile(wl, max(3, min(args.steps, 20)))
    roof = roofline_entry(rep, peaks, peaks_kind, sustained=wl.sustained, f16=wl.dtype == "f16")
    if roof is not None:
        roof["traffic"] = recorded_traffic(roof["kernel"], wl.name)
    step_roof = None
    if wl.credited_flops_per_step:
        # the whole step against the tensor peak: credited GEMM flops per step
        # over the device-timed step (every kernel of the step in the time)
        alu = wl.dtype == "f32"
        peak = round(fp32_alu_tflops(), 2) if alu else \
            peaks["bf16_tflops_sustained" if wl.sustained else "bf16_tflops"]
        ach = wl.credited_flops_per_step / (ms_per_step * 1e-3) / 1e12
        step_roof = {"bound": "alu" if alu else "tensor", "achieved": round(ach, 3),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(ach / peak, 5),
                     "credited_flops_per_step": wl.credited_flops_per_step,
                     "peak_kind": ("derived: SMs x 128 fp32 lanes x 2 flops x 2070 MHz" if alu
                                   else peaks_kind + (" sustained" if wl.sustained
                                                      else " burst"))}

    med = float(np.median(step_ms))
    cv = float(np.std(step_ms) / np.mean(step_ms)) if len(step_ms) > 1 else 0.0
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": wl.unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "ms_per_step_median": round(med, 6), "ms_per_step_cv": round(cv, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic", "config": dict(wl.config, parallelism="replicas" if world > 1
                                            else "single GPU"),
        "clocks": clk.summary(),
        "e2e": {"value": round(e2e_value, 3), "unit": wl.unit,
                "h2d_bytes_per_step": wl.h2d_bytes, "d2h_bytes_per_step": wl.d2h_bytes,
                "mode": e2e_mode},
        "gpu_launches": wl.launches_per_step * args.steps,
        "roofline": roof,
        "step_roofline": step_roof,
        "kernels": {k: [n, round(ms / n, 6)] for k, (n, ms) in sorted(rep.items())},
        "wall_s_timed_region": round(wall, 4),
    }
    if getattr(wl, "train_step_launches", None):
        out["train_step_launches"] = wl.train_step_launches
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.set_threads(os.cpu_count())
        done, dt, sample = wl.oracle_sample(args.cpu_seconds)
        out["cpu_baseline"] = {"value": round(done / dt, 3), "unit": wl.unit,
                               "cores": os.cpu_count(), "kind": "oracle", "sample": sample}
        if wl.name == "mlp784_fp32":
            # the single-step configuration is also timed on one host thread
            oracle.set_threads(1)
            done, dt, sample = wl.oracle_sample(args.cpu_seconds)
            out["cpu_baseline_1thread"] = {"value": round(done / dt, 3), "unit": wl.unit,
                                           "cores": 1, "kind": "oracle", "sample": sample}
            oracle.set_threads(os.cpu_count())
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args, wl):
    rank, world, _ = rank_info()
    if rank != 0:
        return
    per = []
    done_total = 0
    sample = ""
    for i in range(args.warmup + args.steps):
        done, dt, sample = wl.oracle_sample(args.ref_seconds)
        if i >= args.warmup:
            per.append((done, dt))
            done_total += done
    secs = sum(dt for _, dt in per)
    value = done_total / secs
    out = {"metric": METRIC, "impl": "reference", "value": round(value, 3), "unit": wl.unit,
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1e3 * secs / args.steps, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": wl.config,
           "cpu_baseline": {"value": round(value, 3), "unit": wl.unit, "cores": os.cpu_count(),
                            "kind": "oracle", "sample": "each step: " + sample},
           "e2e": {"value": round(value, 3), "unit": wl.unit, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="stack", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=1.0,
                    help="CPU seconds of oracle work per reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="tokens (block, stack) or batch (mlp_wide): smaller profiling cases")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    _, world, _ = rank_info()
    if args.gpus > 1 and world == 1 and "RANK" not in os.environ:
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               "--nproc-per-node", str(args.gpus), "--master-addr", "127.0.0.1",
               "--master-port", "29517", os.path.abspath(__file__)] + sys.argv[1:]
        sys.exit(subprocess.call(cmd))
    if args.tokens and args.workload in SIZED:
        wl = SIZED[args.workload](args.tokens)
    else:
        wl = WORKLOADS[args.workload]()
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
