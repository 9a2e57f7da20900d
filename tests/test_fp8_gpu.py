"""FP8 (e4m3 / e5m2) GEMM on the tensor-core kernels (tcgen05 kind::f8f6f4)
against the oracle, which decodes the same bytes with its own e4m3 / e5m2
decoders and multiplies in float64.

Small integers (-4..4) are exact in both formats and every partial sum is an
integer below 2^24, so the fp32 output must equal the oracle exactly and a bf16
output its round-to-nearest-even; float inputs are checked against the
propagated tolerance, with the per-tensor scales passed as alpha.
"""
import numpy as np
import pytest
import torch

import oracle
from dnn_linear_layers_gb300 import gemm as G

pytestmark = pytest.mark.gpu

FMT = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
OUT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dnn_linear_layers_gb300 import build
    build.build()


def int_fp8(shape, seed, fmt):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-4, 5, shape, generator=g).to(FMT[fmt])


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("shape,kernel", [((300, 264, 260), G.KERNEL_TC_PAIR), ((129, 136, 128), G.KERNEL_TC_SINGLE),
                                          ((64, 200, 384), G.KERNEL_AUTO), ((513, 257, 1000), G.KERNEL_TC_PAIR)])
def test_fp8_exact_integers(fmt, out, shape, kernel):
    M, N, K = shape
    A = int_fp8((M, K), M + K, fmt)
    B = int_fp8((N, K), N + K + 1, fmt)
    bias = torch.randint(-8, 9, (N,), generator=torch.Generator().manual_seed(N)).to(torch.bfloat16)
    C = torch.full((M, N), float("nan"), dtype=OUT[out], device="cuda")
    with G.Plan(0, "nk") as p:
        p.set_kernel(kernel)
        p.run(A.cuda(), B.cuda(), C, bias.cuda(), True)
        assert p.status() == 0
        if kernel == G.KERNEL_AUTO and M <= 128:
            assert p.last_kernel == G.KERNEL_SKINNY          # small M: the weight-streaming kernel
        else:
            assert p.last_kernel in (G.KERNEL_TC_PAIR, G.KERNEL_TC_SINGLE)
    ref = oracle.gemm(A, B, bias=bias, relu=True, b_nk=True)
    want = oracle.bf16_round(ref) if out == "bf16" else ref
    got = C.double().cpu().numpy()
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[0]}: {got[tuple(bad[0])]} vs {want[tuple(bad[0])]}"


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_float_inputs_with_scales(fmt):
    M, N, K = 700, 520, 1024
    g = torch.Generator().manual_seed(3)
    a_scale, b_scale = 0.5, 0.125
    A = (torch.randn(M, K, generator=g) / a_scale).to(FMT[fmt])      # stored value = x / scale
    B = (torch.randn(N, K, generator=g) / b_scale).to(FMT[fmt])
    C = torch.empty(M, N, device="cuda")
    with G.Plan(0, "nk") as p:
        p.run(A.cuda(), B.cuda(), C, alpha=a_scale * b_scale)
        assert p.status() == 0
    C_ref, S = oracle.gemm_ex(A, B, alpha=a_scale * b_scale, b_nk=True)
    ok, worst, _ = oracle.check_close(C.double().cpu().numpy(), C_ref, S)
    assert ok, f"worst err/bound {worst:.3f}"


def test_fp8_misaligned_pitch_is_packed():
    M, N, K = 200, 136, 200
    A = int_fp8((M, K), 1, "e4m3")
    B = int_fp8((N, K), 2, "e4m3")
    abuf = torch.zeros(M, K + 5, dtype=torch.uint8, device="cuda")   # row pitch 205 bytes
    abuf[:, :K] = A.view(torch.uint8).cuda()
    Ad = abuf.view(torch.float8_e4m3fn)[:, :K]
    C = torch.empty(M, N, device="cuda")
    with G.Plan(0, "nk") as p:
        p.run(Ad, B.cuda(), C)
        assert p.status() == 0
        assert p.workspace_bytes > 0
    assert np.array_equal(C.double().cpu().numpy(), oracle.gemm(A, B, b_nk=True))


def test_fp8_convolution_is_refused():
    """fp8 operands run in every GEMM layout (see the layout tests), but the
    convolution entry points take 16-bit inputs only."""
    x = torch.zeros(1, 8, 8, 64, device="cuda").to(torch.float8_e4m3fn)
    w = torch.zeros(64, 3, 3, 64, device="cuda").to(torch.float8_e4m3fn)
    y = torch.zeros(64, 64, device="cuda")
    with G.Plan(0, "nk") as p:
        with pytest.raises(G.GemmError) as e:
            p.conv2d(x, w, y, pad=1)
        assert e.value.code == G.ERR_UNSUPPORTED


def test_fp8_4096_whole_matrix_exact_freivalds():
    M = N = K = 4096
    A = int_fp8((M, K), 11, "e4m3")
    B = int_fp8((N, K), 12, "e4m3")
    C = torch.empty(M, N, device="cuda")
    with G.Plan(0, "nk") as p:
        p.run(A.cuda(), B.cuda(), C)
        assert p.status() == 0
    Cc = C.cpu()
    rng = np.random.default_rng(13)
    for _ in range(2):
        r = rng.choice([-1, 1], size=N)
        assert oracle.freivalds_int(A, B, Cc, r, b_nk=True) == 0
    rows = np.array([0, 1, 127, 128, 255, 256, 2047, 4095])
    ref = oracle.gemm_rows(A, B, rows, b_nk=True)
    assert np.array_equal(Cc[torch.from_numpy(rows)].double().numpy(), ref)


# ---- small M: the weight-streaming kernel with fp8 weights and activations
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 128, 128), (16, 4096, 640), (100, 300, 1000), (128, 1000, 2048), (33, 136, 200)])
def test_fp8_small_m_exact_integers(fmt, out, shape):
    M, N, K = shape
    A = int_fp8((M, K), 7 * M + K, fmt)
    B = int_fp8((N, K), N + 3 * K, fmt)
    bias = torch.randint(-8, 9, (N,), generator=torch.Generator().manual_seed(N + 1)).to(torch.bfloat16)
    C = torch.full((M, N), float("nan"), dtype=OUT[out], device="cuda")
    with G.Plan(0, "nk", b_const=True) as p:
        p.set_kernel(G.KERNEL_SKINNY)
        p.run(A.cuda(), B.cuda(), C, bias.cuda(), True)
        assert p.status() == 0
        assert p.last_kernel == G.KERNEL_SKINNY
    ref = oracle.gemm(A, B, bias=bias, relu=True, b_nk=True)
    want = oracle.bf16_round(ref) if out == "bf16" else ref
    got = C.double().cpu().numpy()
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[0]}: {got[tuple(bad[0])]} vs {want[tuple(bad[0])]}"


def test_fp8_small_m_extended_epilogue_and_packing():
    M, N, K = 16, 520, 384
    A = int_fp8((M, K), 21, "e4m3")
    B = int_fp8((N, K), 22, "e4m3")
    g = torch.Generator().manual_seed(23)
    scale = torch.randint(-4, 5, (N,), generator=g).to(torch.bfloat16)
    bias = torch.randint(-4, 5, (N,), generator=g).to(torch.bfloat16)
    C0 = torch.randint(-4, 5, (M, N), generator=g).float()
    # activations with a row pitch of K + 3 bytes: packed first
    abuf = torch.zeros(M, K + 3, dtype=torch.uint8, device="cuda")
    abuf[:, :K] = A.view(torch.uint8).cuda()
    Ad = abuf.view(torch.float8_e4m3fn)[:, :K]
    C = C0.cuda().clone()
    with G.Plan(0, "nk") as p:
        p.run(Ad, B.cuda(), C, bias.cuda(), relu=True, alpha=0.5, beta=2.0, scale=scale.cuda())
        assert p.status() == 0
        assert p.last_kernel == G.KERNEL_SKINNY
    ref, _ = oracle.gemm_ex(A, B, alpha=0.5, beta=2.0, C0=C0, scale=scale, bias=bias, relu=True, b_nk=True)
    assert np.array_equal(C.double().cpu().numpy(), ref)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_small_m_float_inputs_with_scales(fmt):
    M, N, K = 64, 2048, 4096
    g = torch.Generator().manual_seed(31)
    a_scale, b_scale = 0.25, 0.0625
    A = (torch.randn(M, K, generator=g) / a_scale).to(FMT[fmt])
    B = (torch.randn(N, K, generator=g) / b_scale).to(FMT[fmt])
    C = torch.empty(M, N, device="cuda")
    with G.Plan(0, "nk") as p:
        p.run(A.cuda(), B.cuda(), C, alpha=a_scale * b_scale)
        assert p.status() == 0
        assert p.last_kernel == G.KERNEL_SKINNY
    C_ref, S = oracle.gemm_ex(A, B, alpha=a_scale * b_scale, b_nk=True)
    ok, worst, _ = oracle.check_close(C.double().cpu().numpy(), C_ref, S)
    assert ok, f"worst err/bound {worst:.3f}"
