"""GPU parity tests of the warp-MMA small-M kernel (2 <= M <= 16, 16-bit or
fp8 operands, weight stored N x K; chosen automatically up to M = 8) through
the C ABI against the float64 oracle.

Integer inputs must match exactly (every partial sum is an integer below
2^24, exact in fp32 in any order); float inputs within 1e-3 * sum|a b| + 1e-6
(+ one output ulp for a 16-bit output).  Shapes cover one and two groups of 8
tokens, ragged K (tails inside a 16-byte piece, and k-slices that end inside a
32-k chunk), row counts that leave the last 16-row group partly empty, and N
below one group; the k-split choices 1, 2, 4 and 8 all occur.
"""
import numpy as np
import pytest
import torch

import oracle
from dnn_linear_layers_gb300 import gemm as G
from dnn_linear_layers_gb300.inputs import GemmCase, int_bf16

from parity import compare, oracle_full, run_case

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


def check(plan, case, kernel=G.KERNEL_WARP_MMA):
    A, B, bias, C = run_case(plan, case, kernel=kernel)
    assert plan.last_kernel == G.KERNEL_WARP_MMA
    C_ref, S = oracle_full(case, A, B, bias)
    return compare(case, C, C_ref, S)


@pytest.mark.parametrize("M", [2, 3, 5, 8, 9, 13, 16])
@pytest.mark.parametrize("N,K", [(1, 1), (7, 9), (16, 32), (513, 8), (1000, 1000), (300, 2049), (64, 4104),
                                 (2500, 264), (4096, 4096)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_warp_mma_integer_exact(plan, M, N, K, out):
    check(plan, GemmCase("wmma_int", M, N, K, b_nk=True, bias=True, relu=True, out=out, integer=True,
                         seed=M * 7 + N + K))


@pytest.mark.parametrize("M", [2, 8, 16])
@pytest.mark.parametrize("N,K", [(1000, 1000), (4096, 4096), (333, 5000), (14336, 4096)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_warp_mma_float_within_tolerance(plan, M, N, K, out):
    check(plan, GemmCase("wmma_f", M, N, K, b_nk=True, bias=True, out=out, b_std=K ** -0.5, seed=N + M))


@pytest.mark.parametrize("out", ["f32", "f16"])
@pytest.mark.parametrize("M", [4, 16])
def test_warp_mma_fp16(plan, M, out):
    check(plan, GemmCase("wmma_h", M, 520, 1000, b_nk=True, in_dtype="f16", out=out, integer=True, bias=True,
                         seed=4 + M))


@pytest.mark.parametrize("K", [1, 5, 8, 13, 263, 2047])
@pytest.mark.parametrize("M", [2, 16])
def test_warp_mma_reads_nothing_past_k(plan, M, K):
    """Rows whose pitch is 16-byte aligned but longer than K: the padding of
    both operands holds NaN, which would poison any sum that touched it."""
    N = 300
    ld = (K + 7) // 8 * 8 + 8
    A = int_bf16((M, K), K, lo=-3, hi=3)
    W = int_bf16((N, K), K + 1, lo=-3, hi=3)
    Ab = torch.full((M, ld), float("nan"), dtype=torch.bfloat16)
    Wb = torch.full((N, ld), float("nan"), dtype=torch.bfloat16)
    Ab[:, :K] = A
    Wb[:, :K] = W
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    plan.set_kernel(G.KERNEL_WARP_MMA)
    plan.run(Ab.cuda()[:, :K], Wb.cuda()[:, :K], C)
    assert plan.status() == 0 and plan.last_kernel == G.KERNEL_WARP_MMA
    assert np.array_equal(C.double().cpu().numpy(), oracle.gemm(A, W, b_nk=True))


@pytest.mark.parametrize("M,N,K", [(2, 257, 1001), (11, 100, 4095), (16, 64, 77)])
def test_warp_mma_misaligned_pitches_are_packed(plan, M, N, K):
    A = int_bf16((M, K + 1), M + K)
    W = int_bf16((N, K + 3), N + K)
    Cb = torch.full((M, N + 3), float("nan"), dtype=torch.float32, device="cuda")
    C = Cb[:, 1:N + 1]
    plan.set_kernel(G.KERNEL_WARP_MMA)
    plan.run(A.cuda()[:, 1:], W.cuda()[:, :K], C, relu=True)
    assert plan.status() == 0 and plan.last_kernel == G.KERNEL_WARP_MMA
    assert np.array_equal(C.double().cpu().numpy(), oracle.gemm(A[:, 1:], W[:, :K], relu=True, b_nk=True))
    assert torch.isnan(Cb[:, 0]).all() and torch.isnan(Cb[:, N + 1:]).all()


@pytest.mark.parametrize("M", [3, 16])
def test_warp_mma_extended_epilogue_exact(plan, M):
    """alpha, per-column scale, bias, beta * previous Y and ReLU (gemm_run_ex),
    exact on integers with power-of-two factors."""
    N, K = 700, 900
    A = int_bf16((M, K), 3)
    W = int_bf16((N, K), 4)
    scale = int_bf16((N,), 5, lo=-2, hi=2)
    bias = int_bf16((N,), 6, lo=-8, hi=8)
    C0 = int_bf16((M, N), 7, lo=-16, hi=16).float()
    C = C0.cuda()
    plan.set_kernel(G.KERNEL_WARP_MMA)
    plan.run(A.cuda(), W.cuda(), C, bias.cuda(), True, alpha=0.5, beta=2.0, scale=scale.cuda())
    assert plan.status() == 0 and plan.last_kernel == G.KERNEL_WARP_MMA
    ref, _ = oracle.gemm_ex(A, W, alpha=0.5, beta=2.0, C0=C0.double().numpy(), scale=scale, bias=bias, relu=True,
                            b_nk=True)
    assert np.array_equal(C.double().cpu().numpy(), ref)


@pytest.mark.parametrize("b_const", [False, True])
def test_warp_mma_chained_layers_see_previous_outputs(b_const):
    """Back-to-back layers on one stream, each reading the previous layer's
    output: with programmatic dependent launch and (b_const) the weight loads
    issued before the dependency wait, no kernel may read its input X before
    the producing kernel is done."""
    p = G.Plan(0, "nk", b_const=b_const)
    p.set_kernel(G.KERNEL_WARP_MMA)
    M, D = 16, 512
    Ws = [int_bf16((D, D), 60 + i, lo=-1, hi=1).cuda() for i in range(8)]
    x = int_bf16((M, D), 59, lo=-1, hi=1)
    h = x.cuda()
    outs = []
    for i, w in enumerate(Ws):
        y = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
        p.run(h, w, y, relu=True)
        h = torch.clamp(y, max=1.0) if i % 2 else y
        outs.append(h)
    assert p.status() == 0
    ref = x.double().numpy()
    for i, w in enumerate(Ws):
        ref = oracle.bf16_round(oracle.gemm(ref, w.cpu(), relu=True, b_nk=True))
        if i % 2:
            ref = np.minimum(ref, 1.0)
        assert np.array_equal(outs[i].double().cpu().numpy(), ref), f"layer {i}"
    p.close()


@pytest.mark.parametrize("M", [2, 4, 8])
def test_warp_mma_decode_layers_every_output(M):
    """The benchmark's decode layers, 4096 -> 14336 with bias, bf16 out, as
    dispatched (the warp-MMA kernel up to M = 8), every output."""
    N, K = 14336, 4096
    with G.Plan(0, "nk", b_const=True) as p:
        case = GemmCase("wmma_full", M, N, K, b_nk=True, bias=True, out="bf16", b_std=K ** -0.5, seed=77 + M)
        A, B, bias, C = run_case(p, case)
        assert p.last_kernel == G.KERNEL_WARP_MMA
        C_ref, S = oracle_full(case, A, B, bias)
        compare(case, C, C_ref, S)


def test_warp_mma_refuses_what_it_does_not_take(plan):
    x = torch.ones(17, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(32, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(17, 32, dtype=torch.float32, device="cuda")
    plan.set_kernel(G.KERNEL_WARP_MMA)
    with pytest.raises(G.GemmError) as e:
        plan.run(x, w, y)                                       # M = 17 > 16
    assert e.value.code == G.ERR_UNSUPPORTED
    with pytest.raises(G.GemmError) as e:                       # tf32 operands
        plan.run(x[:4].float(), w.float(), y[:4])
    assert e.value.code == G.ERR_UNSUPPORTED
    with G.Plan(0, "kn") as pk:                                  # K x N weight
        pk.set_kernel(G.KERNEL_WARP_MMA)
        with pytest.raises(G.GemmError) as e:
            pk.run(x[:4], torch.ones(64, 32, dtype=torch.bfloat16, device="cuda"), y[:4])
        assert e.value.code == G.ERR_UNSUPPORTED


def test_dispatch_warp_mma():
    """AUTO: M = 1 -> GEMV, 2 <= M <= 8 with a 16-bit or fp8 N x K weight ->
    warp-MMA, M = 9 or a K x N weight -> the tensor-core small-M kernel;
    GEMM_OPT_WARP_MMA_MAX_M moves the threshold (up to 16)."""
    with G.Plan(0, "nk") as p:
        assert p.get_option(G.OPT_WARP_MMA_MAX_M) == 8
        w = torch.ones(512, 256, dtype=torch.bfloat16, device="cuda")
        for M, want in [(1, G.KERNEL_GEMV), (2, G.KERNEL_WARP_MMA), (8, G.KERNEL_WARP_MMA),
                        (9, G.KERNEL_SKINNY), (16, G.KERNEL_SKINNY)]:
            A = torch.ones(M, 256, dtype=torch.bfloat16, device="cuda")
            C = torch.empty(M, 512, device="cuda")
            p.run(A, w, C)
            assert p.status() == 0 and p.last_kernel == want and torch.all(C == 256.0)
        A8 = torch.ones(4, 256, device="cuda").to(torch.float8_e4m3fn)
        C = torch.empty(4, 512, device="cuda")
        p.run(A8, w.to(torch.float8_e4m3fn), C)
        assert p.status() == 0 and p.last_kernel == G.KERNEL_WARP_MMA and torch.all(C == 256.0)
        p.set_option(G.OPT_WARP_MMA_MAX_M, 4)
        A = torch.ones(5, 256, dtype=torch.bfloat16, device="cuda")
        C = torch.empty(5, 512, device="cuda")
        p.run(A, w, C)
        assert p.status() == 0 and p.last_kernel == G.KERNEL_SKINNY
        p.set_option(G.OPT_WARP_MMA_MAX_M, 16)
        A = torch.ones(16, 256, dtype=torch.bfloat16, device="cuda")
        C = torch.empty(16, 512, device="cuda")
        p.run(A, w, C)
        assert p.status() == 0 and p.last_kernel == G.KERNEL_WARP_MMA and torch.all(C == 256.0)
        with pytest.raises(G.GemmError):
            p.set_option(G.OPT_WARP_MMA_MAX_M, 17)
    with G.Plan(0, "kn") as pk:
        A = torch.ones(4, 256, dtype=torch.bfloat16, device="cuda")
        C = torch.empty(4, 512, device="cuda")
        pk.run(A, torch.ones(256, 512, dtype=torch.bfloat16, device="cuda"), C)
        assert pk.status() == 0 and pk.last_kernel == G.KERNEL_SKINNY


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,N,K", [(2, 1000, 4096), (5, 300, 2000), (8, 129, 33), (16, 520, 1000), (3, 64, 4111),
                                   (8, 14336, 4096)])
def test_warp_mma_fp8_integer_exact(plan, fmt, out, M, N, K):
    """fp8 codes through m16n8k32: 16 k-values per 16-byte piece, ragged K
    (tails inside a piece), bf16 bias, exact on small integers."""
    f8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}[fmt]
    A = int_bf16((M, K), M + K).to(f8)
    W = int_bf16((N, K), N + K).to(f8)
    bias = int_bf16((N,), N, lo=-8, hi=8)
    C = torch.full((M, N), float("nan"), dtype=out, device="cuda")
    plan.set_kernel(G.KERNEL_WARP_MMA)
    plan.run(A.cuda(), W.cuda(), C, bias.cuda(), True)
    assert plan.status() == 0 and plan.last_kernel == G.KERNEL_WARP_MMA
    ref = oracle.gemm(A, W, bias=bias, relu=True, b_nk=True)
    want = oracle.bf16_round(ref) if out == torch.bfloat16 else ref
    assert np.array_equal(C.double().cpu().numpy(), want)


@pytest.mark.parametrize("M", [2, 16])
def test_warp_mma_fp8_float_with_scales(plan, M):
    N, K = 700, 1024
    g = torch.Generator().manual_seed(M)
    a_scale, b_scale = 0.5, 0.125
    A = (torch.randn(M, K, generator=g) / a_scale).to(torch.float8_e4m3fn)
    W = (torch.randn(N, K, generator=g) / b_scale).to(torch.float8_e4m3fn)
    C = torch.empty(M, N, device="cuda")
    plan.set_kernel(G.KERNEL_WARP_MMA)
    plan.run(A.cuda(), W.cuda(), C, alpha=a_scale * b_scale)
    assert plan.status() == 0 and plan.last_kernel == G.KERNEL_WARP_MMA
    C_ref, S = oracle.gemm_ex(A, W, alpha=a_scale * b_scale, b_nk=True)
    ok, worst, _ = oracle.check_close(C.double().cpu().numpy(), C_ref, S)
    assert ok, f"worst err/bound {worst:.3f}"


@pytest.mark.parametrize("K", [1, 15, 16, 17, 263, 2047])
def test_warp_mma_fp8_reads_nothing_past_k(plan, K):
    """fp8 rows with 16-byte aligned pitches longer than K, padded with NaN codes."""
    M, N = 5, 300
    ld = (K + 15) // 16 * 16 + 16
    A = int_bf16((M, K), K, lo=-3, hi=3).to(torch.float8_e4m3fn)
    W = int_bf16((N, K), K + 1, lo=-3, hi=3).to(torch.float8_e4m3fn)
    Ab = torch.full((M, ld), float("nan")).to(torch.float8_e4m3fn)
    Wb = torch.full((N, ld), float("nan")).to(torch.float8_e4m3fn)
    Ab[:, :K] = A
    Wb[:, :K] = W
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    plan.set_kernel(G.KERNEL_WARP_MMA)
    plan.run(Ab.cuda()[:, :K], Wb.cuda()[:, :K], C)
    assert plan.status() == 0 and plan.last_kernel == G.KERNEL_WARP_MMA
    assert np.array_equal(C.double().cpu().numpy(), oracle.gemm(A, W, b_nk=True))
