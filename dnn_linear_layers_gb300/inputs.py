"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module draws random numbers and names workloads; it holds none of the
GEMM's arithmetic, imports neither the CUDA library nor the oracle, and both
sides consume exactly the tensors it returns.

Recipe: a ``torch.Generator('cpu')`` seeded per tensor; ``torch.randn`` in
float32 scaled by the standard deviation, then rounded to bf16 (round to
nearest even); integer data from ``torch.randint`` (exact in bf16).  Tensors
are generated on the host so both sides see identical bits.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


def normal_bf16(shape, seed: int, std: float = 1.0, dtype=torch.bfloat16) -> torch.Tensor:
    g = torch.Generator("cpu").manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(dtype)


def relu_normal_bf16(shape, seed: int, dtype=torch.bfloat16) -> torch.Tensor:
    """Non-negative activations: ReLU(N(0,1)) (the output of a previous ReLU layer)."""
    return normal_bf16(shape, seed, 1.0, dtype).clamp_min(0)


def int_bf16(shape, seed: int, lo: int = -4, hi: int = 4, dtype=torch.bfloat16) -> torch.Tensor:
    """Uniform integers in [lo, hi], exactly representable in bf16/fp16."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    return torch.randint(lo, hi + 1, tuple(shape), generator=g, dtype=torch.int32).to(dtype)


@dataclass
class GemmCase:
    """One GEMM / Linear problem: C[M,N] = A[M,K] . B (+bias) (ReLU)."""
    name: str
    M: int
    N: int
    K: int
    b_nk: bool = False          # B stored N x K (a Linear weight W, out x in)
    bias: bool = False
    relu: bool = False
    out: str = "bf16"           # "bf16" or "f32"
    in_dtype: str = "bf16"      # "bf16" or "f16"
    a_std: float = 1.0
    b_std: float = 1.0
    bias_std: float = 0.02
    integer: bool = False
    a_relu: bool = False        # activations are ReLU(N(0,1))
    seed: int = 0
    tags: tuple = field(default_factory=tuple)

    def tensors(self):
        """Host tensors (A, B, bias-or-None) for this case."""
        dt = torch.bfloat16 if self.in_dtype == "bf16" else torch.float16
        b_shape = (self.N, self.K) if self.b_nk else (self.K, self.N)
        s = self.seed * 3
        if self.integer:
            A = int_bf16((self.M, self.K), s, dtype=dt)
            B = int_bf16(b_shape, s + 1, dtype=dt)
            bias = int_bf16((self.N,), s + 2, dtype=dt) if self.bias else None
        else:
            if self.a_relu:
                A = relu_normal_bf16((self.M, self.K), s, dtype=dt)
            else:
                A = normal_bf16((self.M, self.K), s, self.a_std, dtype=dt)
            B = normal_bf16(b_shape, s + 1, self.b_std, dtype=dt)
            bias = normal_bf16((self.N,), s + 2, self.bias_std, dtype=dt) if self.bias else None
        return A, B, bias

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


def square(n: int, integer: bool = False, out: str = "bf16", seed: int = 0) -> GemmCase:
    return GemmCase(f"square{n}{'_int' if integer else ''}", n, n, n, out=out,
                    integer=integer, seed=seed)


# Workload families (shapes, distributions and layouts of the pages' layers).
SMALL_F32 = GemmCase("gemm512_f32out", 512, 512, 512, out="f32", seed=0)

SQUARE_SIZES = (1024, 2048, 4096, 8192)

TOKENS = 8192          # batch 4 x sequence 2048
D_MODEL = 4096
D_FF = 14336


def transformer_cases(seed: int = 0):
    """QKV projection, FFN up (bias+ReLU), FFN down (bias); weights N(0, 1/in),
    stored in x out (the K x N operand), bias N(0, 0.02^2)."""
    return [
        GemmCase("qkv_4096x12288", TOKENS, 3 * D_MODEL, D_MODEL, b_std=D_MODEL ** -0.5, seed=seed),
        GemmCase("ffn_up_4096x14336_bias_relu", TOKENS, D_FF, D_MODEL, bias=True, relu=True,
                 b_std=D_MODEL ** -0.5, seed=seed + 1),
        GemmCase("ffn_down_14336x4096_bias", TOKENS, D_MODEL, D_FF, bias=True,
                 b_std=D_FF ** -0.5, seed=seed + 2),
    ]


# 3x3 convolution, stride 1, pad 1, batch 32, 56x56, 256 -> 256 channels.
CONV = dict(Nb=32, H=56, W=56, Cin=256, Cout=256, R=3, S=3, pad=1)


def conv_tensors(Nb=32, H=56, W=56, Cin=256, Cout=256, R=3, S=3, seed: int = 0):
    """NHWC activations ReLU(N(0,1)) and weights w[f][r][s][c] ~ N(0, 2/(R*S*Cin))."""
    x = relu_normal_bf16((Nb, H, W, Cin), 3 * seed)
    w = normal_bf16((Cout, R, S, Cin), 3 * seed + 1, (2.0 / (R * S * Cin)) ** 0.5)
    return x, w


def skinny_cases(seed: int = 0):
    """Decode-like Linear layers: W (out x in) stored as given, x ~ N(0,1),
    W ~ N(0, 1/4096), bias N(0, 0.02^2)."""
    cases = []
    for (n, k) in ((D_FF, D_MODEL), (D_MODEL, D_MODEL)):
        for m in (1, 16, 128):
            cases.append(GemmCase(f"linear_m{m}_{k}x{n}", m, n, k, b_nk=True, bias=True,
                                  b_std=D_MODEL ** -0.5, seed=seed))
    return cases


def odd_cases(seed: int = 0):
    return [GemmCase("odd1000", 1000, 1000, 1000, seed=seed),
            GemmCase("odd4095", 4095, 4095, 4095, seed=seed),
            GemmCase("odd3000x5000x2048", 3000, 5000, 2048, seed=seed)]
