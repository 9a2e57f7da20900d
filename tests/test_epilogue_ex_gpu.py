"""The extended epilogue (gemm_run_ex, gemm_conv2d with gemm_epilogue_args_t)
on the GPU against the oracle's gemm_ex:

    C = relu?( alpha * (A.B) * scale[j] + bias[j] + beta * C_old[i][j] )

Integer inputs with power-of-two alpha and scale keep every intermediate an
exact integer below 2^24, so the fp32 output must equal the oracle exactly and
a bf16 output must equal its round-to-nearest-even; float inputs are checked
against the propagated tolerance.  Covers the paired, single-CTA and small-M
kernels, both B layouts, C updated in place, C packed through the workspace
(misaligned pitch), K = 0 and the implicit convolution.
"""
import numpy as np
import pytest
import torch

import oracle
from dnn_linear_layers_gb300 import gemm as G
from dnn_linear_layers_gb300.inputs import int_bf16

pytestmark = pytest.mark.gpu

OUT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dnn_linear_layers_gb300 import build
    build.build()


def ints(shape, seed, lo=-4, hi=4):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g)


def expect(C_ref, out):
    return oracle.bf16_round(C_ref) if out == "bf16" else C_ref


CASES = [  # kernel, M, N, K, layout
    (G.KERNEL_TC_PAIR, 300, 264, 130, "kn"),
    (G.KERNEL_TC_PAIR, 257, 200, 72, "nk"),
    (G.KERNEL_TC_SINGLE, 129, 136, 64, "kn"),
    (G.KERNEL_SKINNY, 64, 300, 130, "nk"),
    (G.KERNEL_SKINNY, 7, 129, 200, "kn"),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("relu", [False, True])
def test_run_ex_exact_integers(case, out, relu):
    kernel, M, N, K, lay = case
    seed = M + N + K + (7 if relu else 0)
    A = ints((M, K), seed).to(torch.bfloat16)
    B = ints((N, K) if lay == "nk" else (K, N), seed + 1).to(torch.bfloat16)
    C0 = ints((M, N), seed + 2, -60, 60)
    e = ints((N,), seed + 3, 0, 2)
    scale = (2.0 ** e).to(torch.bfloat16)
    bias = ints((N,), seed + 4, -20, 20).to(torch.bfloat16)
    alpha, beta = 2.0, -0.5 if out == "f32" else -1.0
    C = C0.to(OUT[out]).cuda()        # updated in place
    with G.Plan(0, lay) as p:
        p.set_kernel(kernel)
        p.run(A.cuda(), B.cuda(), C, bias.cuda(), relu, alpha=alpha, beta=beta, scale=scale.cuda())
        assert p.status() == 0
        assert p.last_kernel == kernel
    C_ref, _ = oracle.gemm_ex(A, B, alpha=alpha, beta=beta, C0=C0.to(OUT[out]).double().numpy(), scale=scale,
                              bias=bias, relu=relu, b_nk=(lay == "nk"))
    got = C.double().cpu().numpy()
    want = expect(C_ref, out)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[0]}: {got[tuple(bad[0])]} vs {want[tuple(bad[0])]}"


@pytest.mark.parametrize("kernel", [G.KERNEL_TC_PAIR, G.KERNEL_SKINNY])
def test_run_ex_float_tolerance_and_packed_c(kernel):
    M, N, K = (520, 300, 333) if kernel == G.KERNEL_TC_PAIR else (96, 300, 333)
    g = torch.Generator().manual_seed(5)
    A = torch.randn(M, K, generator=g).bfloat16()
    B = torch.randn(N, K, generator=g).bfloat16()
    C0 = torch.randn(M, N, generator=g)
    scale = (1 + 0.01 * torch.arange(N)).bfloat16()
    bias = torch.full((N,), 0.5).bfloat16()
    # C in a buffer with an odd pitch: the pack path writes through the workspace,
    # the previous values are read from C itself
    buf = torch.zeros(M, N + 3, device="cuda")
    C = buf[:, :N]
    C.copy_(C0)
    with G.Plan(0, "nk") as p:
        p.set_kernel(kernel)
        p.run(A.cuda(), B.cuda(), C, bias.cuda(), True, alpha=0.75, beta=0.25, scale=scale.cuda())
        assert p.status() == 0
    C_ref, S = oracle.gemm_ex(A, B, alpha=0.75, beta=0.25, C0=C0.numpy(), scale=scale, bias=bias, relu=True, b_nk=True)
    bound = 1e-3 * S + 1e-6 + 1e-6 * (np.abs(0.25 * C0.numpy()) + 0.5)
    err = np.abs(C.double().cpu().numpy() - C_ref)
    assert np.all(err <= bound), f"worst err/bound {(err / bound).max():.3f}"


def test_run_ex_k_zero_fill():
    M, N = 37, 41
    C0 = ints((M, N), 9, -30, 30).float().cuda()
    bias = ints((N,), 10, -5, 5).to(torch.bfloat16)
    C = C0.clone()
    with G.Plan(0, "kn") as p:
        A = torch.empty(M, 0, dtype=torch.bfloat16, device="cuda")
        B = torch.empty(0, N, dtype=torch.bfloat16, device="cuda")
        p.run(A, B, C, bias.cuda(), True, alpha=3.0, beta=2.0)
        assert p.status() == 0
        assert p.last_kernel == G.KERNEL_FILL
    want = np.maximum(bias.double().numpy()[None, :] + 2.0 * C0.double().cpu().numpy(), 0.0)
    assert np.array_equal(C.double().cpu().numpy(), want)


@pytest.mark.parametrize("implicit", [True, False])
def test_conv2d_scale_bias_relu_residual_exact(implicit):
    # the fused-convolution epilogue: per-channel scale and bias, ReLU, plus a residual (beta * y)
    Nb, H, W, Cout, R, pad = 2, 9, 9, 48, 3, 1
    C = 64 if implicit else 16                    # 16 channels: explicit im2col path
    x = int_bf16((Nb, H, W, C), 51)
    w = int_bf16((Cout, R, R, C), 52)
    scale = (2.0 ** ints((Cout,), 53, 0, 2)).to(torch.bfloat16)
    bias = ints((Cout,), 54, -20, 20).to(torch.bfloat16)
    res = ints((Nb * H * W, Cout), 55, -40, 40).float()
    y = res.clone().cuda()
    with G.Plan(0, "nk") as p:
        p.set_option(G.OPT_STREAM_K, 0)   # the workspace then holds only an im2col matrix
        p.conv2d(x.cuda(), w.cuda(), y, bias.cuda(), True, pad=pad, beta=1.0, scale=scale.cuda())
        assert p.status() == 0
        assert (p.workspace_bytes == 0) == implicit
    pos = [(n, oh, ow) for n in range(Nb) for oh in range(H) for ow in range(W)]
    conv = oracle.conv2d_at(x, w, pad, pos)
    want = oracle.epilogue_ex(conv, beta=1.0, C0=res.numpy(), scale=scale, bias=bias, relu=True)
    assert np.array_equal(y.double().cpu().numpy(), want)
