#!/usr/bin/env python
"""Benchmark: bf16 GEMM throughput at M = N = K = 8192 on GB300 (one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

A step is one call of the library's public entry point, ``gemm_run`` (C ABI),
on the workload: C[8192 x 8192] = A[8192 x 8192] . B[8192 x 8192], bf16
inputs drawn N(0, 1) from fixed seeds, fp32 accumulation, bf16 output.  The
inputs (384 MB with C) are larger than the 129 MB L2, so no flush is needed
between steps.  ``value`` is TFLOP/s (2*M*N*K per step) with the inputs
resident in HBM; ``e2e`` is the same metric when every step also copies A and
B from pinned host memory and reads C back (steps pipelined over two buffer
sets, so one step's copies overlap the previous step's computation).

With N > 1 (torchrun, one process per GPU) every rank runs an independent
replica of the workload (the GEMM needs no exchange between GPUs) and the
value is the work of all ranks over the slowest rank's time.

``--impl reference`` times the float64 CPU oracle on the host cores on a
bounded sample of the same workload (whole rows of C) and prints the same
metric; under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "bf16 GEMM TFLOP/s at M=N=K=8192 and % of GB300 dense bf16 roofline"

WORKLOADS = {
    # name: (M, N, K, b_layout, epilogue(bias, relu), out, a_std, b_std)
    "square8192_bf16": (8192, 8192, 8192, "kn", (False, False), "bf16", 1.0, 1.0),
    "square4096_bf16": (4096, 4096, 4096, "kn", (False, False), "bf16", 1.0, 1.0),
    "square2048_bf16": (2048, 2048, 2048, "kn", (False, False), "bf16", 1.0, 1.0),
    "square1024_bf16": (1024, 1024, 1024, "kn", (False, False), "bf16", 1.0, 1.0),
    # the small single GEMM: fp32 output, no epilogue
    "square512_f32": (512, 512, 512, "kn", (False, False), "f32", 1.0, 1.0),
    "square8192_nk_bf16": (8192, 8192, 8192, "nk", (False, False), "bf16", 1.0, 1.0),
    "square4096_nk_bf16": (4096, 4096, 4096, "nk", (False, False), "bf16", 1.0, 1.0),
    "qkv_8192x4096x12288": (8192, 12288, 4096, "kn", (False, False), "bf16", 1.0, 4096 ** -0.5),
    "ffn_up_8192x4096x14336": (8192, 14336, 4096, "kn", (True, True), "bf16", 1.0, 4096 ** -0.5),
    "ffn_down_8192x14336x4096": (8192, 4096, 14336, "kn", (True, False), "bf16", 1.0, 14336 ** -0.5),
    "conv_im2col_100352x2304x256": (100352, 256, 2304, "nk", (False, False), "bf16", 1.0, (2 / 2304) ** 0.5),
    # the same convolution as an implicit GEMM: gemm_conv2d on the NHWC activations
    "conv_implicit_32x56x56x256_3x3": (100352, 256, 2304, "nk", (False, False), "bf16", 1.0, (2 / 2304) ** 0.5),
    # ... with per-channel bias, ReLU and the 2 x 2 max-pool fused (gemm_conv2d_maxpool)
    "conv_pool_32x56x56x256_3x3": (100352, 256, 2304, "nk", (True, True), "bf16", 1.0, (2 / 2304) ** 0.5),
    "odd_3000x5000x2048": (3000, 5000, 2048, "kn", (False, False), "bf16", 1.0, 1.0),
    # fused attention forward, B 4 x H 32 x S 4096 x D 128 (M = B*H*S query rows, N = D, K = S keys)
    "attention_b4h32s4096d128": (4 * 32 * 4096, 128, 4096, "nk", (False, False), "bf16", 1.0, 1.0),
    "attention_causal_b4h32s4096d128": (4 * 32 * 4096, 128, 4096, "nk", (False, False), "bf16", 1.0, 1.0),
    "attention_b4h32s4096d64": (4 * 32 * 4096, 64, 4096, "nk", (False, False), "bf16", 1.0, 1.0),
    # fp8 operands (both K-major: B stored N x K), bf16 output
    "square8192_e4m3": (8192, 8192, 8192, "nk", (False, False), "bf16", 1.0, 1.0),
    "square8192_e5m2": (8192, 8192, 8192, "nk", (False, False), "bf16", 1.0, 1.0),
    # fp32 operands multiplied at tf32 precision (B stored N x K), bf16 output
    "square8192_tf32": (8192, 8192, 8192, "nk", (False, False), "bf16", 1.0, 1.0),
    # A stored K x M (the transposed operand, plan flag GEMM_A_KM)
    "square8192_transa_bf16": (8192, 8192, 8192, "kn", (False, False), "bf16", 1.0, 1.0),
    "odd_4095": (4095, 4095, 4095, "kn", (False, False), "bf16", 1.0, 1.0),
    "odd_1000": (1000, 1000, 1000, "kn", (False, False), "bf16", 1.0, 1.0),
    # decode-like Linear layers: W stored out x in, bias, M tokens
    "linear_m1_4096x14336": (1, 14336, 4096, "nk", (True, False), "bf16", 1.0, 4096 ** -0.5),
    "linear_m16_4096x14336": (16, 14336, 4096, "nk", (True, False), "bf16", 1.0, 4096 ** -0.5),
    "linear_m128_4096x14336": (128, 14336, 4096, "nk", (True, False), "bf16", 1.0, 4096 ** -0.5),
    "linear_m1_4096x4096": (1, 4096, 4096, "nk", (True, False), "bf16", 1.0, 4096 ** -0.5),
    "linear_m2_4096x14336": (2, 14336, 4096, "nk", (True, False), "bf16", 1.0, 4096 ** -0.5),
    "linear_m4_4096x14336": (4, 14336, 4096, "nk", (True, False), "bf16", 1.0, 4096 ** -0.5),
    "linear_m8_4096x14336": (8, 14336, 4096, "nk", (True, False), "bf16", 1.0, 4096 ** -0.5),
    "linear_m4_4096x4096": (4, 4096, 4096, "nk", (True, False), "bf16", 1.0, 4096 ** -0.5),
    "linear_m16_4096x4096": (16, 4096, 4096, "nk", (True, False), "bf16", 1.0, 4096 ** -0.5),
    "linear_m128_4096x4096": (128, 4096, 4096, "nk", (True, False), "bf16", 1.0, 4096 ** -0.5),
    # the same decode layers with e4m3 weights and activations (per-tensor scales belong in alpha)
    "linear_m1_4096x14336_e4m3": (1, 14336, 4096, "nk", (True, False), "bf16", 1.0, 1.0),
    "linear_m4_4096x14336_e4m3": (4, 14336, 4096, "nk", (True, False), "bf16", 1.0, 1.0),
    "linear_m16_4096x14336_e4m3": (16, 14336, 4096, "nk", (True, False), "bf16", 1.0, 1.0),
    "linear_m128_4096x14336_e4m3": (128, 14336, 4096, "nk", (True, False), "bf16", 1.0, 1.0),
}
DEFAULT_WORKLOAD = "square8192_bf16"
KERNEL_NAME = "gemm_tc_kernel"
SMI_QUERY = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of `x` over the ranks of the default process group
    (the slowest rank's time); `x` itself when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: every rank ran `steps` independent replica steps; the
    job took as long as its slowest rank."""
    return world * flops_per_step * steps / (max_ms * 1e-3) / 1e12


# sources each profiled kernel depends on: its translation unit, the shared
# headers and the dispatcher that sets its launch parameters
KERNEL_SOURCES = {
    "tc": ["kernels_tc.cu", "ptx.cuh", "internal.h", "gemm_api.cu"],
    "skinny": ["kernels_skinny.cu", "ptx.cuh", "internal.h", "gemm_api.cu"],
    "gemv": ["kernels_gemv.cu", "ptx.cuh", "internal.h", "gemm_api.cu"],
    "attn": ["kernels_attn.cu", "ptx.cuh", "internal.h", "gemm_api.cu"],
}


def kernel_source_hash(files) -> str:
    h = hashlib.sha256()
    for name in files:
        h.update((ROOT / "dnn_linear_layers_gb300" / "csrc" / name).read_bytes())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the top kernel from the committed ncu summary,
    valid only if that kernel's sources are unchanged since it was taken."""
    f = ROOT / "profiles" / "traffic.json"
    try:
        d = json.loads(f.read_text())
        e = d[workload]
        if e.get("source_hash") == kernel_source_hash(KERNEL_SOURCES[e["sources"]]):
            return float(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    def __init__(self, index: int, period_ms: int = 100):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu={SMI_QUERY}", "--format=csv,noheader,nounits",
                 f"-lms={period_ms}"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, max_mhz_hint=None):
        sms, maxes, reasons, powers = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            try:
                sm, mx = float(f[2]), float(f[3])
            except ValueError:
                continue
            sms.append(sm); maxes.append(mx)
            try:
                powers.append(float(f[4]))
            except ValueError:
                pass
            for n, v in zip(names, f[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": max_mhz_hint, "reasons": [], "samples": 0}
        # samples under load: the upper half by power (the tool starts before the load)
        loaded = sms
        if powers and len(powers) == len(sms) and len(sms) >= 4:
            cut = statistics.median(powers)
            loaded = [s for s, p in zip(sms, powers) if p >= cut] or sms
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms), "power_w_max": max(powers) if powers else None}


def fp8_dtype(name):
    """torch dtype of a workload's operands when they are not 16-bit (fp8, or fp32 read as tf32)."""
    import torch
    return {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2,
            "tf32": torch.float32}.get(name.rsplit("_", 1)[-1])


# nominal dense tensor rate of each operand type relative to bf16 (fp8 4.5 / 2.25, tf32 1.1 / 2.25)
PEAK_RATIO = {"e4m3": 2.0, "e5m2": 2.0, "tf32": 1.1 / 2.25}


def attn_shape(name):
    """(B, H, S, D) of an attention workload, from its name (..._b4h32s4096d128)."""
    m = re.search(r"_b(\d+)h(\d+)s(\d+)d(\d+)$", name)
    return tuple(int(x) for x in m.groups())


def attention_flops(name: str) -> float:
    """4 D FLOPs per visible (query, key) pair: 2 D for the score, 2 D for P V."""
    causal = "causal" in name
    B, H, S, D = attn_shape(name)
    pairs = S * (S + 1) / 2 if causal else S * S
    return 4.0 * B * H * D * pairs


def make_inputs(name, device, seed=0):
    import torch
    from dnn_linear_layers_gb300.inputs import normal_bf16
    M, N, K, lay, (has_bias, relu), out, a_std, b_std = WORKLOADS[name]
    if name.startswith(("attention_",)):
        # q (B, H, S, D) and k, v stacked: (2, B, H, S, D); N(0, 1) bf16
        B, H, S, D = attn_shape(name)
        q = normal_bf16((B, H, S, D), 3 * seed)
        kv = torch.stack([normal_bf16((B, H, S, D), 3 * seed + 1), normal_bf16((B, H, S, D), 3 * seed + 2)])
        return q, kv, None
    f8 = fp8_dtype(name)
    if f8 is not None and name.endswith("_tf32"):   # N(0,1) fp32
        A = normal_bf16((M, K), 3 * seed, a_std, dtype=torch.float32)
        B = normal_bf16((N, K), 3 * seed + 1, b_std, dtype=torch.float32)
        return A, B, None
    if f8 is not None:   # N(0,1) drawn as bf16, then rounded to the fp8 format; bf16 bias
        A = normal_bf16((M, K), 3 * seed, a_std).to(f8)
        B = normal_bf16((N, K), 3 * seed + 1, b_std).to(f8)
        bias = normal_bf16((N,), 3 * seed + 2, 0.02) if has_bias else None
        return A, B, bias
    if "_transa_" in name:   # A as stored: K x M
        A = normal_bf16((K, M), 3 * seed, a_std)
        B = normal_bf16((N, K) if lay == "nk" else (K, N), 3 * seed + 1, b_std)
        return A, B, None
    if name.startswith(("conv_implicit", "conv_pool")):
        # x (NHWC 32x56x56x256, ReLU(N(0,1))) and w[f][r][s][c] as they are
        from dnn_linear_layers_gb300.inputs import conv_tensors
        x, w = conv_tensors(seed=seed)
        bias = normal_bf16((N,), 3 * seed + 2, 0.02) if has_bias else None
        return x, w, bias
    if name.startswith("conv_im2col"):
        # activations ReLU(N(0,1)) NHWC 32x56x56x256, weights w[f][r][s][c]; the
        # im2col matrix is built on the GPU by the library (setup, untimed)
        from dnn_linear_layers_gb300 import gemm as G
        from dnn_linear_layers_gb300.inputs import conv_tensors
        x, w = conv_tensors(seed=seed)
        dev = device if device is not None else torch.device("cuda", 0)
        A = G.im2col(x.to(dev), 3, 3, 1, 1).cpu()
        return A, w.reshape(w.shape[0], -1).contiguous(), None
    A = normal_bf16((M, K), 3 * seed, a_std)
    B = normal_bf16((N, K) if lay == "nk" else (K, N), 3 * seed + 1, b_std)
    bias = normal_bf16((N,), 3 * seed + 2, 0.02) if has_bias else None
    return A, B, bias


class Workload:
    """One workload on one GPU: inputs resident in HBM (rotating copies when
    they are smaller than twice the L2), a plan, and the K timed steps
    captured once into a CUDA graph."""

    def __init__(self, name, dev, local_rank, args):
        import torch
        from dnn_linear_layers_gb300 import gemm as G
        from dnn_linear_layers_gb300 import roofline as R
        self.name = name
        self.dev = dev
        self.args = args
        M, N, K, lay, (has_bias, relu), out, _, _ = WORKLOADS[name]
        self.M, self.N, self.K, self.lay, self.has_bias, self.relu = M, N, K, lay, has_bias, relu
        self.out_dtype = torch.float32 if out == "f32" else torch.bfloat16
        self.A_h, self.B_h, self.bias_h = make_inputs(name, dev, seed=0)
        A, B = self.A_h.to(dev), self.B_h.to(dev)
        self.bias = self.bias_h.to(dev) if self.bias_h is not None else None
        self.pool = name.startswith("conv_pool")
        self.attn = name.startswith("attention_")
        self.causal = "causal" in name
        self.conv = name.startswith(("conv_implicit", "conv_pool"))
        self.f8 = fp8_dtype(name)
        # the pooled convolution writes a quarter of the output rows; attention writes O like q
        C = (torch.empty(tuple(A.shape), dtype=self.out_dtype, device=dev) if self.attn else
             torch.empty((M // 4 if self.pool else M, N), dtype=self.out_dtype, device=dev))
        self.A, self.B, self.C = A, B, C
        # Linear-layer weights are constant model parameters: say so to the plan
        self.plan = G.Plan(local_rank, lay, b_const=name.startswith("linear_"),
                           a_layout="km" if "_transa_" in name else "mk")
        if args.kernel != "auto":
            self.plan.set_kernel({"pair": G.KERNEL_TC_PAIR, "single": G.KERNEL_TC_SINGLE, "skinny": G.KERNEL_SKINNY,
                                  "gemv": G.KERNEL_GEMV, "warp_mma": G.KERNEL_WARP_MMA}[args.kernel])
        for kv in args.opt or []:          # scheduling options (sweeps): NAME=VALUE, NAME as in GEMM_OPT_NAME
            key, val = kv.split("=")
            self.plan.set_option(getattr(G, "OPT_" + key.upper()), int(val))
        self.stream = torch.cuda.current_stream(dev)
        self.flops = attention_flops(name) if self.attn else 2.0 * M * N * K
        if self.attn:   # q, k, v read once, o written once
            self.nbytes = float(A.numel() * 2 + B.numel() * 2 + C.numel() * C.element_size())
        elif self.conv:   # activations, weights and output once each (no im2col matrix exists)
            self.nbytes = float(A.numel() * 2 + B.numel() * 2 + C.numel() * C.element_size() +
                                (N * 2 if has_bias else 0))
        else:
            es = A.element_size()
            self.nbytes = R.gemm_bytes(M, N, K, es, es, C.element_size(), 2 if has_bias else 0)
        # Workloads smaller than twice the L2 rotate through enough copies of their
        # operands that each step reads HBM, not the previous step's L2 lines.
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.n_copies = 1 if self.nbytes >= 2 * self.l2 else int(2 * self.l2 // self.nbytes) + 2
        self.copies = [(A, B, C)] + [(A.clone(), B.clone(), torch.empty_like(C)) for _ in range(self.n_copies - 1)]
        self.counter = 0
        self.graph = None

    def call(self, a, b, c):
        if self.attn:
            self.plan.attention(a, b[0], b[1], c, causal=self.causal)
        elif self.pool:
            self.plan.conv2d_maxpool(a, b, c, self.bias, self.relu, pad=1)
        elif self.conv:
            self.plan.conv2d(a, b, c, self.bias, self.relu, pad=1)
        else:
            self.plan.run(a, b, c, self.bias, self.relu)      # on torch's current stream

    def step(self):
        a, b, c = self.copies[self.counter % self.n_copies]
        self.counter += 1
        self.call(a, b, c)

    def prepare(self):
        """Warm-up steps, then capture the K timed steps into a CUDA graph, so
        the GPU runs them back to back with no host launch gaps between steps
        (short decode-like kernels would otherwise time the Python launch path)."""
        import torch
        args, dev = self.args, self.dev
        for _ in range(args.warmup):
            self.step()
        torch.cuda.synchronize()
        assert self.plan.status() == 0, "device status after warm-up"
        launches0 = self.plan.launch_count
        if not args.no_graph:
            try:
                side = torch.cuda.Stream(dev)
                side.wait_stream(torch.cuda.current_stream(dev))
                with torch.cuda.stream(side):
                    self.step()
                torch.cuda.current_stream(dev).wait_stream(side)
                torch.cuda.synchronize()
                launches0 = self.plan.launch_count
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=side):
                    for _ in range(args.steps):
                        self.step()
                torch.cuda.synchronize()
                self.graph = graph
            except Exception as exc:  # capture unsupported: time eager launches instead
                self.graph = None
                print(f"# graph capture failed ({exc}); timing eager launches", file=sys.stderr)
                torch.cuda.synchronize()
        self.launches_per_run = self.plan.launch_count - launches0

    def timed_run(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            for _ in range(self.args.steps):
                self.step()

    def time(self, world, sampler=None):
        """Device time (ms) of the K steps on the launching stream, and the
        number of this library's kernels they launched.  With a clock sampler,
        the GPU is first kept busy for a second (untimed) so the clocks settle."""
        import torch
        import torch.distributed as dist
        self.timed_run()
        torch.cuda.synchronize()
        t_end = time.time() + (1.0 if sampler else 0.0)
        while time.time() < t_end:
            self.timed_run()
            torch.cuda.synchronize()
        launches0 = self.plan.launch_count
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True); t1 = torch.cuda.Event(enable_timing=True)
        t0.record(self.stream)
        self.timed_run()
        t1.record(self.stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        launches = self.launches_per_run if self.graph is not None else self.plan.launch_count - launches0
        st = self.plan.status()
        assert st == 0, f"device status {st}"
        return t0.elapsed_time(t1), launches

    def roofline(self, kernel_ms):
        """(tensor_bound, achieved, peak, unit, peak_source, roofline_time_s, peak_src_kind)."""
        from dnn_linear_layers_gb300 import roofline as R
        peaks, src = R.load_peaks()
        kind = self.name.rsplit("_", 1)[-1]
        # an fp8 or tf32 contraction takes the measured bf16 peak times the nominal ratio of the two rates
        t_peak = peaks["bf16_tflops"] * (PEAK_RATIO[kind] if self.f8 is not None else 1.0)
        t_roof = R.roofline_time(self.flops, self.nbytes, t_peak * 1e12, peaks["hbm_gbs"] * 1e9)
        tensor_bound = self.flops / (t_peak * 1e12) >= self.nbytes / (peaks["hbm_gbs"] * 1e9)
        if tensor_bound:
            achieved, peak, unit = self.flops / (kernel_ms * 1e-3) / 1e12, t_peak, "TFLOP/s"
            peak_src = (f"MEASURED_PEAKS.json bf16_tflops (burst) x {PEAK_RATIO[kind]:.4g}, the nominal {kind} / "
                        "bf16 ratio" if self.f8 is not None else "MEASURED_PEAKS.json bf16_tflops (burst)")
        else:
            achieved, peak, unit = self.nbytes / (kernel_ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s"
            peak_src = "MEASURED_PEAKS.json hbm_gbs"
        return tensor_bound, achieved, peak, unit, peak_src, t_roof, src

    def kernel_name(self):
        from dnn_linear_layers_gb300 import gemm as G
        if self.attn:
            return "attention"
        return {G.KERNEL_TC_PAIR: "tc_pair", G.KERNEL_TC_SINGLE: "tc_single", G.KERNEL_SKINNY: "skinny",
                G.KERNEL_GEMV: "gemv", G.KERNEL_WARP_MMA: "warp_mma"}.get(self.plan.last_kernel,
                                                                          str(self.plan.last_kernel))

    def close(self):
        self.plan.close()


# Decode-like Linear layers timed after the headline in the same process and
# reported under "secondary" (the memory-bound half of the target).
SECONDARY = ("linear_m1_4096x14336", "linear_m4_4096x14336", "linear_m16_4096x14336")


def secondary_lines(dev, local_rank, args, world):
    out = {}
    for name in SECONDARY:
        w = Workload(name, dev, local_rank, args)
        w.prepare()
        sampler = ClockSampler(local_rank) if not args.no_clocks else None
        total_ms, launches = w.time(world, sampler)
        if sampler:
            sampler.stop()
        total_ms = max_over_ranks(total_ms, dev)
        kernel_ms = total_ms / args.steps
        tb, achieved, peak, unit, peak_src, t_roof, src = w.roofline(kernel_ms)
        out[name] = {"value": round(w.nbytes * args.steps * world / (total_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                     "ms_per_step": round(total_ms / args.steps, 5), "kernel": w.kernel_name(),
                     "roofline": {"bound": "tensor" if tb else "hbm", "achieved": round(achieved, 2), "peak": peak,
                                  "unit": unit, "frac": round(achieved / peak, 4),
                                  "peak_source": f"measured ({peak_src})" if src == "measured" else "fallback",
                                  "algorithmic_bytes": w.nbytes, "traffic": profiled_traffic(name)},
                     "config": {"M": w.M, "N": w.N, "K": w.K, "b_layout": w.lay, "epilogue": "bias",
                                "l2": f"{w.n_copies} rotating operand copies"},
                     "gpu_launches": int(launches),
                     "clocks": sampler.summary() if sampler else None}
        w.close()
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    name = args.workload
    w = Workload(name, dev, local_rank, args)
    M, N, K = w.M, w.N, w.K
    w.prepare()
    sampler = ClockSampler(local_rank) if not args.no_clocks else None
    total_ms, launches = w.time(world, sampler)
    if sampler:
        sampler.stop()
    # steps run back to back on one stream: the average launch lasts total / K
    # (for single-kernel steps; with packing, a step also holds the copies)
    kernel_ms = total_ms / args.steps
    total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(w.flops, args.steps, world, total_ms)

    # ---- end to end: pinned host inputs -> device -> the library call -> host
    # result, every step.  Steps are pipelined over two device buffer sets and
    # three streams (copy in, compute, copy out): the copies of one step overlap
    # the computation of the one before, as a serving loop would run them.
    A, B, C, stream = w.A, w.B, w.C, w.stream
    A_p = w.A_h.pin_memory(); B_p = w.B_h.pin_memory()
    C_p = [torch.empty(tuple(C.shape), dtype=C.dtype).pin_memory() for _ in range(2)]
    A_e = [torch.empty_like(A) for _ in range(2)]
    B_e = [torch.empty_like(B) for _ in range(2)]
    C_e = [torch.empty_like(C) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of buffer set b are on the device
    ev_comp = [torch.cuda.Event() for _ in range(2)]    # its result is computed (inputs free)
    ev_out = [torch.cuda.Event() for _ in range(2)]     # its result is on the host (output free)
    e2e_count = [0]

    def e2e_step():
        i = e2e_count[0]
        e2e_count[0] += 1
        b = i & 1
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[b])
            A_e[b].copy_(A_p, non_blocking=True)
            B_e[b].copy_(B_p, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])
        w.call(A_e[b], B_e[b], C_e[b])            # on torch's current stream
        ev_comp[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            C_p[b].copy_(C_e[b], non_blocking=True)
            ev_out[b].record(s_out)

    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    for _ in range(0 if args.no_e2e else 2):
        e2e_step()
    torch.cuda.synchronize()
    e2e_count[0] = 0
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for _ in range(0 if args.no_e2e else e2e_steps):
        e2e_step()
    stream.wait_stream(s_out)                     # the last result is on the host
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, dev)
    e2e_value = job_throughput(w.flops, e2e_steps, world, e2e_ms) if not args.no_e2e else None
    assert w.plan.status() == 0

    tensor_bound, achieved, peak, r_unit, peak_src, t_roof, src = w.roofline(kernel_ms)
    secondary = (secondary_lines(dev, local_rank, args, world)
                 if name == DEFAULT_WORKLOAD and not args.no_secondary else None)
    kind = name.rsplit("_", 1)[-1]
    f8, attn = w.f8, w.attn
    has_bias, relu, lay, l2, n_copies, nbytes = w.has_bias, w.relu, w.lay, w.l2, w.n_copies, w.nbytes
    result = None
    if rank == 0:
        cpu = None if args.no_cpu_baseline else cpu_baseline(name, w.A_h, w.B_h, w.bias_h, args.cpu_seconds)
        clocks = sampler.summary() if sampler else {"sm_mhz": None, "sm_max_mhz": None, "reasons": []}
        result = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": kind if f8 is not None else "bf16",
            "data": ("synthetic: N(0,1) fp32 (torch CPU generator, fixed seeds), resident in HBM" if kind == "tf32"
                     else "synthetic: N(0,1) drawn as bf16 (torch CPU generator, fixed seeds), rounded to "
                     f"{kind}, resident in HBM" if f8 is not None else
                     "synthetic: N(0,1) bf16 (torch CPU generator, fixed seeds), resident in HBM"),
            "config": {"workload": name,
                       **({"B": attn_shape(name)[0], "H": attn_shape(name)[1], "Sq": attn_shape(name)[2],
                           "Sk": attn_shape(name)[2], "D": attn_shape(name)[3], "causal": "causal" in name,
                           "scale": "1/sqrt(D)"} if attn else
                          {"M": M, "N": N, "K": K, "b_layout": lay, "a_layout": "km" if "_transa_" in name else "mk",
                           "epilogue": ("bias" if has_bias else "") + ("+relu" if relu else "") or "none"}),
                       "out": "f32" if w.out_dtype == torch.float32 else "bf16", "accumulate": "fp32",
                       "parallelism": f"replicas x{world}",
                       "l2": (f"inputs larger than L2 ({nbytes / 1e6:.1f} MB > {l2 / 1e6:.0f} MB), no flush"
                              if n_copies == 1 else
                              f"{n_copies} rotating operand copies ({n_copies * nbytes / 1e6:.0f} MB > 2 x L2)"),
                       "kernel": w.kernel_name(),
                       "timing": "CUDA graph of the K steps, one replay" if w.graph is not None else "eager launches"},
            "roofline": {"bound": "tensor" if tensor_bound else "hbm",
                         "achieved": round(achieved, 2), "peak": peak, "unit": r_unit,
                         "frac": round(achieved / peak, 4),
                         "frac_of_roofline_time": round(t_roof / (kernel_ms * 1e-3), 4),
                         "peak_source": f"measured ({peak_src})" if src == "measured" else "fallback",
                         "traffic": profiled_traffic(name),
                         "algorithmic_bytes": nbytes, "flops_per_launch": w.flops,
                         "kernel_ms": round(kernel_ms, 5)},
            "e2e": {"value": round(e2e_value, 2) if e2e_value else None, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": int(A_p.numel() * A_p.element_size() + B_p.numel() * B_p.element_size()),
                    "d2h_bytes_per_step": int(C_p[0].numel() * C_p[0].element_size()), "steps": e2e_steps,
                    "pipelined": "copies of a step overlap the previous step's computation (two buffer sets, "
                                 "three streams)"},
            "gpu_launches": int(launches),
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        if secondary is not None:
            result["secondary"] = secondary
        print(json.dumps(result), flush=True)
    w.close()
    if world > 1:
        dist.destroy_process_group()
    return result


def _oracle_rows_timer(name, A, B, bias):
    """Callable timing the oracle on n seeded whole rows of C: returns (seconds, n)."""
    import numpy as np
    import oracle
    M, N, K, lay, (has_bias, relu), *_ = WORKLOADS[name]
    threads = len(os.sched_getaffinity(0))
    if name.startswith("attention_"):
        # float64 attention of n seeded heads (numpy); each head is a unit of work
        Bb, Hh, S, D = attn_shape(name)
        causal = "causal" in name
        rng = np.random.default_rng(0)

        def run_attn(n):
            heads = rng.choice(Bb * Hh, size=min(Bb * Hh, max(1, n)), replace=False)
            qf = A.reshape(Bb * Hh, S, D); kf = B[0].reshape(Bb * Hh, S, D); vf = B[1].reshape(Bb * Hh, S, D)
            t = time.perf_counter()
            for hd in heads:
                oracle.attention(qf[hd], kf[hd], vf[hd], causal=causal)
            return time.perf_counter() - t, len(heads)

        return run_attn, threads
    if name.startswith(("conv_implicit", "conv_pool")):
        # the direct seven-loop convolution at n seeded output positions (one thread)
        Nb, H, W, _ = A.shape
        rng = np.random.default_rng(0)

        def run_conv(n):
            idx = rng.choice(M, size=min(M, n), replace=False)
            pos = [(int(i) // (H * W), (int(i) // W) % H, int(i) % W) for i in idx]
            t = time.perf_counter()
            oracle.conv2d_at(A, B, 1, pos)
            return time.perf_counter() - t, len(pos)

        return run_conv, 1
    Af = oracle._f64(A); Bf = oracle._f64(B)   # fp8 bytes decoded by the oracle's own decoders
    if "_transa_" in name:                      # A is stored K x M
        Af = np.ascontiguousarray(Af.T)
    bf = bias.double().numpy() if bias is not None else None
    rng = np.random.default_rng(0)

    def run(n):
        rows = rng.choice(M, size=min(M, n), replace=False)
        t = time.perf_counter()
        oracle.gemm_rows(Af, Bf, rows, bias=bf, relu=relu, b_nk=(lay == "nk"), threads=threads)
        return time.perf_counter() - t, len(rows)

    return run, threads


def oracle_unit(name):
    """(FLOPs per unit of oracle work, units in the workload, unit description)."""
    M, N, K, *_ = WORKLOADS[name]
    if name.startswith("attention_"):
        Bb, Hh, S, D = attn_shape(name)
        return attention_flops(name) / (Bb * Hh), Bb * Hh, f"heads ({S} x {S} scores, D {D})"
    return 2.0 * N * K, M, f"rows of C (each {N} x {K} MACs)"


def cpu_baseline(name, A, B, bias, seconds: float):
    """Oracle (float64 triple loop, OpenMP over rows) on whole rows of C, about `seconds` of work."""
    per, total, what = oracle_unit(name)
    run, threads = _oracle_rows_timer(name, A, B, bias)
    cal = 1 if name.startswith("attention_") else threads
    dt, n = run(cal)                            # calibration: one row per thread (one head)
    n = int(max(cal, min(total, cal * max(1, round(seconds / max(dt, 1e-3))))))
    dt, n = run(n)
    return {"value": round(per * n / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "sample": f"{n} of {total} {what}, {dt:.1f} s",
            "seconds": round(dt, 2)}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return None
    name = args.workload
    M, N, K, lay, (has_bias, relu), *_ = WORKLOADS[name]
    A, B, bias = make_inputs(name, None, seed=0)
    per, total, what = oracle_unit(name)
    run, threads = _oracle_rows_timer(name, A, B, bias)
    cal = 1 if name.startswith("attention_") else threads
    dt, n = run(cal)
    # size every step so the whole run stays within about two minutes
    per_step = min(max(90.0 / (args.warmup + args.steps), 0.05), args.cpu_seconds)
    n = int(max(cal, min(total, cal * max(1, round(per_step / max(dt, 1e-3))))))
    vals, times = [], []
    for i in range(args.warmup + args.steps):
        dt, n_done = run(n)
        if i >= args.warmup:
            vals.append(per * n_done / dt / 1e12); times.append(dt)
    value = round(statistics.median(vals), 6)
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * statistics.median(times), 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic: same inputs as the GPU arm", "config": {"workload": name, "M": M, "N": N, "K": K},
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                            "sample": f"{n} of {total} {what} per step"},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling runs)")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of a graph replay")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the decode-layer lines appended to the default workload's result")
    ap.add_argument("--opt", action="append", metavar="NAME=VALUE",
                    help="set a plan scheduling option (sweeps), e.g. stream_k=0 or group_m=16")
    ap.add_argument("--kernel", choices=["auto", "pair", "single", "skinny", "gemv", "warp_mma"], default="auto",
                    help="force a kernel (sweeps); the default lets the library choose")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
