"""GPU parity for tf32 operands (GEMM_TF32_*: fp32 A and B in memory,
multiplied by the tensor cores at tf32 precision -- 8-bit exponent, 10-bit
mantissa -- with fp32 accumulation) against the float64 oracle.

Bounds, with S = sum_k |a_ik b_kj| and K the reduction length:
* integer inputs in [-4, 4] are tf32 values, every product and partial sum is
  an integer below 2^24: exact;
* inputs already on the tf32 grid: each product of two 11-bit significands is
  exact in fp32, so only the accumulation rounds: |err| <= K 2^-23 S (one unit
  of 2^-23 per addition, which also covers an accumulator that truncates);
* arbitrary fp32 inputs: reading each operand as tf32 moves it by less than
  2^-10 of itself (truncation; 2^-11 when rounded), so a product moves by less
  than (2^-9 + 2^-20) of itself: |err| <= (2^-9 + 2^-20 + K 2^-23) S + 1e-6.
The middle case is the one that tells a tf32 product from a narrower one (bf16
operands would miss its bound by about 60x).
"""
import numpy as np
import pytest
import torch

import oracle
from dnn_linear_layers_gb300 import gemm as G

from parity import alloc_with_guard, guard_intact

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def plan():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dnn_linear_layers_gb300 import build
    build.build()
    p = G.Plan(0, "nk")
    yield p
    p.close()


def to_tf32_grid(x: torch.Tensor) -> torch.Tensor:
    """Round fp32 values to the nearest tf32 value (ties to even): keep the top
    10 of the 23 stored mantissa bits."""
    u = x.contiguous().view(torch.int32).numpy().astype(np.int64) & 0xFFFFFFFF
    lsb = (u >> 13) & 1
    r = ((u + 0xFFF + lsb) & ~0x1FFF) & 0xFFFFFFFF
    return torch.from_numpy(r.astype(np.uint32).view(np.int32)).view(torch.float32).reshape(x.shape)


def inputs(M, N, K, kind, seed, bias=False):
    g = torch.Generator().manual_seed(seed)
    if kind == "int":
        A = torch.randint(-4, 5, (M, K), generator=g).float()
        W = torch.randint(-4, 5, (N, K), generator=g).float()
        b = torch.randint(-4, 5, (N,), generator=g).to(torch.bfloat16) if bias else None
    else:
        A = torch.randn(M, K, generator=g)
        W = torch.randn(N, K, generator=g)
        if kind == "grid":
            A, W = to_tf32_grid(A), to_tf32_grid(W)
        b = (0.02 * torch.randn(N, generator=g)).to(torch.bfloat16) if bias else None
    return A, W, b


def run(plan, M, N, K, kind, out=torch.float32, kernel=G.KERNEL_AUTO, bias=False, relu=False, seed=0,
        lda_pad=0):
    A, W, b = inputs(M, N, K, kind, seed, bias)
    if lda_pad:
        full = torch.zeros(M, K + lda_pad)
        full[:, :K] = A
        Ad = full.cuda()[:, :K]
    else:
        Ad = A.cuda()
    buf, C, iv, bits = alloc_with_guard(M, N, out)
    plan.set_kernel(kernel)
    plan.run(Ad, W.cuda(), C, b.cuda() if b is not None else None, relu=relu)
    assert plan.status() == 0
    if kernel == G.KERNEL_AUTO and K > 0:
        assert plan.last_kernel == G.KERNEL_TC_PAIR
    assert guard_intact(buf, M, N, iv, bits)
    ref, S = oracle.gemm(A, W, bias=b, relu=relu, b_nk=True, with_mag=True)
    got = C.double().cpu().numpy()
    if kind == "int":
        want = ref if out == torch.float32 else oracle.bf16_round(ref)
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"{len(bad)} mismatches, first {bad[0]}: {got[tuple(bad[0])]} vs {want[tuple(bad[0])]}"
        return 0.0
    rel = (K * 2.0 ** -23) if kind == "grid" else (2.0 ** -9 + 2.0 ** -20 + K * 2.0 ** -23)
    bound = rel * S + 1e-6
    if out == torch.bfloat16:
        bound = bound + oracle.ulp_bf16(ref)
    err = np.abs(got - ref)
    worst = float((err / bound).max())
    assert np.all(err <= bound), f"worst err/bound {worst:.3f}"
    return worst


@pytest.mark.parametrize("kernel", [G.KERNEL_TC_SINGLE, G.KERNEL_TC_PAIR])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_tf32_integer_exact_ragged(plan, kernel, out):
    run(plan, 600, 700, 333, "int", out=out, kernel=kernel, seed=1)


@pytest.mark.parametrize("shape", [(1, 8, 4), (16, 300, 40), (129, 257, 100), (513, 520, 1000)])
def test_tf32_shapes_with_epilogue_integer_exact(plan, shape):
    M, N, K = shape
    run(plan, M, N, K, "int", out=torch.bfloat16, bias=True, relu=True, seed=sum(shape))


@pytest.mark.parametrize("kernel", [G.KERNEL_TC_SINGLE, G.KERNEL_TC_PAIR])
def test_tf32_grid_inputs_round_only_in_the_sum(plan, kernel):
    run(plan, 1000, 1100, 700, "grid", kernel=kernel, seed=2)


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_tf32_float_within_tolerance(plan, out):
    run(plan, 1000, 1100, 2000, "float", out=out, bias=True, seed=3)


def test_tf32_misaligned_pitch_is_packed(plan):
    run(plan, 250, 260, 270, "int", lda_pad=1, seed=4)        # 271 fp32 per row: not a 16-byte multiple


def test_tf32_k0_and_large(plan):
    run(plan, 100, 200, 0, "int", bias=True, seed=5)
    run(plan, 2048, 2304, 1024, "int", seed=6)


def test_tf32_refusals():
    """tf32 runs on the tensor-core kernels only (every operand layout: see the
    layout tests); the small-M kernel and the convolution refuse it."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    A = torch.zeros(64, 32, device="cuda")
    C = torch.zeros(64, 16, device="cuda")
    with G.Plan(0, "nk") as p:
        p.set_kernel(G.KERNEL_SKINNY)
        with pytest.raises(G.GemmError) as e:
            p.run(A, torch.zeros(16, 32, device="cuda"), C)
        assert e.value.code == G.ERR_UNSUPPORTED
        p.set_kernel(G.KERNEL_AUTO)
        x = torch.zeros(1, 8, 8, 64, device="cuda")
        w = torch.zeros(64, 3, 3, 64, device="cuda")
        y = torch.zeros(64, 64, device="cuda")
        with pytest.raises(G.GemmError) as e:
            p.conv2d(x, w, y, pad=1)
        assert e.value.code == G.ERR_UNSUPPORTED


def test_tf32_extended_epilogue_integer_exact(plan):
    # alpha * acc * scale + bias + beta * C_old, ReLU; bf16 scale and bias vectors
    A, W, _ = inputs(260, 300, 64, "int", 7)
    g = torch.Generator().manual_seed(8)
    scale = torch.randint(-4, 5, (300,), generator=g).to(torch.bfloat16)
    bias = torch.randint(-4, 5, (300,), generator=g).to(torch.bfloat16)
    C0 = torch.randint(-4, 5, (260, 300), generator=g).float()
    C = C0.cuda().clone()
    plan.set_kernel(G.KERNEL_AUTO)
    plan.run(A.cuda(), W.cuda(), C, bias.cuda(), relu=True, alpha=2.0, beta=-1.0, scale=scale.cuda())
    assert plan.status() == 0
    ref, _ = oracle.gemm_ex(A, W, alpha=2.0, beta=-1.0, C0=C0, scale=scale, bias=bias, relu=True, b_nk=True)
    assert (C.double().cpu().numpy() == ref).all()
