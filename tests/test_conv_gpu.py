"""Convolution as explicit GEMM on the GPU: the im2col kernel against the
oracle's im2col (exact copy), and the im2col matrix times the weights against
the oracle's direct seven-loop convolution.

The full-size case is the 3 x 3, stride 1, pad 1 convolution of a batch of 32
56 x 56 x 256 NHWC activations (ReLU(N(0,1))) with 256 filters w[f][r][s][c]
~ N(0, 2/2304): M = 100352, K = 2304, N = 256.
"""
import numpy as np
import pytest
import torch

import oracle
from dnn_linear_layers_gb300 import gemm as G
from dnn_linear_layers_gb300.inputs import CONV, GemmCase, conv_tensors, int_bf16

from parity import compare

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


@pytest.mark.parametrize("shape", [(2, 9, 9, 16, 3, 3, 1, 1), (1, 7, 5, 3, 3, 3, 1, 1), (2, 8, 8, 8, 3, 3, 0, 2),
                                   (1, 6, 6, 24, 5, 5, 2, 1), (3, 4, 4, 8, 1, 1, 0, 1)])
def test_im2col_matches_oracle(plan, shape):
    Nb, H, W, C, R, S, pad, stride = shape
    x = int_bf16((Nb, H, W, C), sum(shape))
    cols = G.im2col(x.cuda(), R, S, pad, stride)
    torch.cuda.synchronize()
    if stride == 1:
        ref = oracle.im2col(x, R, S, pad)
    else:   # the oracle's im2col is stride 1; pick the strided rows of a stride-1 matrix
        full = oracle.im2col(x, R, S, pad)
        OH1 = H + 2 * pad - R + 1; OW1 = W + 2 * pad - S + 1
        OH = (H + 2 * pad - R) // stride + 1; OW = (W + 2 * pad - S) // stride + 1
        idx = [(n * OH1 + oh * stride) * OW1 + ow * stride for n in range(Nb) for oh in range(OH) for ow in range(OW)]
        ref = full[idx]
    assert np.array_equal(cols.double().cpu().numpy(), ref)


def test_small_conv_as_gemm_exact(plan):
    x = int_bf16((2, 9, 9, 16), 5)
    w = int_bf16((32, 3, 3, 16), 6)
    cols = G.im2col(x.cuda(), 3, 3, 1, 1)
    Y = torch.empty(cols.shape[0], 32, device="cuda")
    plan.run(cols, w.reshape(32, -1).cuda(), Y)
    assert plan.status() == 0
    pos = [(n, oh, ow) for n in range(2) for oh in range(9) for ow in range(9)]
    ref = oracle.conv2d_at(x, w, 1, pos)
    assert np.array_equal(Y.double().cpu().numpy(), ref)


def test_full_conv_config_sampled(plan):
    Nb, H, W, Cin, Cout = CONV["Nb"], CONV["H"], CONV["W"], CONV["Cin"], CONV["Cout"]
    x, w = conv_tensors()
    xd = x.cuda()
    cols = G.im2col(xd, 3, 3, 1, 1)                       # 100352 x 2304
    Wm = w.reshape(Cout, -1)
    Y = torch.empty(cols.shape[0], Cout, dtype=torch.bfloat16, device="cuda")
    plan.set_kernel(G.KERNEL_AUTO)
    plan.run(cols, Wm.cuda(), Y)
    assert plan.status() == 0
    rng = np.random.default_rng(4)
    # border and interior positions of several images
    pos = {(n, oh, ow) for n in (0, Nb - 1) for oh in (0, 1, H // 2, H - 1) for ow in (0, 1, W // 2, W - 1)}
    pos |= {(int(rng.integers(Nb)), int(rng.integers(H)), int(rng.integers(W))) for _ in range(48)}
    pos = sorted(pos)
    rows = np.array([(n * H + oh) * W + ow for n, oh, ow in pos])
    # the GPU im2col rows are the oracle's im2col rows, bit for bit
    A_rows = oracle.im2col_rows(x, 3, 3, 1, rows)
    assert np.array_equal(cols[torch.from_numpy(rows).cuda()].double().cpu().numpy(), A_rows)
    C_ref, S = oracle.gemm(A_rows, Wm, b_nk=True, with_mag=True)
    direct = oracle.conv2d_at(x, w, 1, pos)
    assert np.all(np.abs(direct - C_ref) <= 1e-12 * (S + 1))
    case = GemmCase("conv", len(rows), Cout, 9 * Cin, b_nk=True, out="bf16")
    compare(case, Y[torch.from_numpy(rows).cuda()].cpu(), C_ref, S)


# ---- implicit GEMM (gemm_conv2d): A tiles fetched from the NHWC activations
# through a TMA im2col tensor map, no im2col matrix in memory

IMPLICIT_SHAPES = [  # Nb, H, W, C, Cout, R(=S), pad
    (2, 9, 9, 64, 32, 3, 1),        # M = 162: one pair tile, ragged
    (1, 17, 13, 128, 200, 3, 1),    # two channel blocks per tap, ragged N
    (3, 8, 8, 64, 64, 1, 0),        # 1 x 1 filter: a plain GEMM over pixels
    (2, 12, 10, 64, 48, 5, 2),      # 5 x 5, pad 2
    (2, 11, 11, 64, 16, 3, 0),      # no padding: 9 x 9 outputs
    (4, 20, 20, 64, 256, 3, 1),     # M = 1600: several tiles, last one partial
]


def conv_out_hw(H, W, R, pad):
    return H + 2 * pad - R + 1, W + 2 * pad - R + 1


@pytest.mark.parametrize("shape", IMPLICIT_SHAPES)
def test_implicit_conv_exact_every_output(shape):
    Nb, H, W, C, Cout, R, pad = shape
    x = int_bf16((Nb, H, W, C), 11 + sum(shape))
    w = int_bf16((Cout, R, R, C), 12 + sum(shape))
    OH, OW = conv_out_hw(H, W, R, pad)
    with G.Plan(0, "kn") as p:   # the plan's B layout does not apply to convolutions
        p.set_option(G.OPT_STREAM_K, 0)   # no split-tile partials: the workspace stays empty
        y = torch.full((Nb * OH * OW, Cout), float("nan"), device="cuda")
        p.conv2d(x.cuda(), w.cuda(), y, pad=pad)
        assert p.status() == 0
        assert p.last_kernel == G.KERNEL_TC_PAIR
        assert p.workspace_bytes == 0, "implicit path must not build an im2col matrix"
    pos = [(n, oh, ow) for n in range(Nb) for oh in range(OH) for ow in range(OW)]
    ref = oracle.conv2d_at(x, w, pad, pos)
    assert np.array_equal(y.double().cpu().numpy(), ref)


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_implicit_conv_bitwise_equals_explicit_gemm(out):
    # same A tiles in the same order to the same MMAs: identical bits
    Nb, H, W, C, Cout = 3, 23, 19, 128, 96
    g = torch.Generator().manual_seed(7)
    x = torch.randn(Nb, H, W, C, generator=g).bfloat16().cuda()
    w = (torch.randn(Cout, 3, 3, C, generator=g) * (2 / (9 * C)) ** 0.5).bfloat16().cuda()
    b = (torch.randn(Cout, generator=g) * 0.02).bfloat16().cuda()
    od = torch.bfloat16 if out == "bf16" else torch.float32
    with G.Plan(0, "nk") as p:
        y_imp = torch.empty(Nb * H * W, Cout, dtype=od, device="cuda")
        p.conv2d(x, w, y_imp, bias=b, relu=True, pad=1)
        cols = G.im2col(x, 3, 3, 1, 1)
        y_exp = torch.empty_like(y_imp)
        p.run(cols, w.reshape(Cout, -1), y_exp, b, relu=True)
        assert p.status() == 0
    assert torch.equal(y_imp.view(torch.int16 if out == "bf16" else torch.int32),
                       y_exp.view(torch.int16 if out == "bf16" else torch.int32))


@pytest.mark.parametrize("shape", [(2, 9, 9, 16, 32, 3, 1),     # C not a multiple of 64
                                   (1, 5, 5, 64, 24, 3, 1),     # M = 25: small-M path
                                   (2, 9, 9, 64, 8, 1, 0)])     # 1 x 1, N = 8
def test_conv_fallback_paths_exact(shape):
    Nb, H, W, C, Cout, R, pad = shape
    x = int_bf16((Nb, H, W, C), 31 + sum(shape))
    w = int_bf16((Cout, R, R, C), 32 + sum(shape))
    OH, OW = conv_out_hw(H, W, R, pad)
    with G.Plan(0, "nk") as p:
        y = torch.full((Nb * OH * OW, Cout), float("nan"), device="cuda")
        p.conv2d(x.cuda(), w.cuda(), y, pad=pad)
        assert p.status() == 0
    pos = [(n, oh, ow) for n in range(Nb) for oh in range(OH) for ow in range(OW)]
    assert np.array_equal(y.double().cpu().numpy(), oracle.conv2d_at(x, w, pad, pos))


def test_full_conv_config_implicit_sampled(plan):
    Nb, H, W, Cin, Cout = CONV["Nb"], CONV["H"], CONV["W"], CONV["Cin"], CONV["Cout"]
    x, w = conv_tensors()
    xd, wd = x.cuda(), w.cuda()
    y = torch.empty(Nb * H * W, Cout, dtype=torch.bfloat16, device="cuda")
    plan.set_kernel(G.KERNEL_AUTO)
    plan.conv2d(xd, wd, y, pad=1)
    assert plan.status() == 0
    assert plan.last_kernel == G.KERNEL_TC_PAIR
    rng = np.random.default_rng(5)
    pos = {(n, oh, ow) for n in (0, Nb - 1) for oh in (0, 1, H // 2, H - 1) for ow in (0, 1, W // 2, W - 1)}
    pos |= {(int(rng.integers(Nb)), int(rng.integers(H)), int(rng.integers(W))) for _ in range(48)}
    pos = sorted(pos)
    rows = np.array([(n * H + oh) * W + ow for n, oh, ow in pos])
    A_rows = oracle.im2col_rows(x, 3, 3, 1, rows)
    C_ref, S = oracle.gemm(A_rows, w.reshape(Cout, -1), b_nk=True, with_mag=True)
    case = GemmCase("conv_implicit", len(rows), Cout, 9 * Cin, b_nk=True, out="bf16")
    compare(case, y[torch.from_numpy(rows).cuda()].cpu(), C_ref, S)
    # and the whole output equals the explicit path bit for bit
    cols = G.im2col(xd, 3, 3, 1, 1)
    y_exp = torch.empty_like(y)
    plan.run(cols, wd.reshape(Cout, -1), y_exp)
    assert plan.status() == 0
    assert torch.equal(y.view(torch.int16), y_exp.view(torch.int16))


# ---- convolution + epilogue + 2 x 2 max-pool in one kernel (gemm_conv2d_maxpool)

POOL_SHAPES = [  # Nb, H, W, C, Cout, R(=S), pad
    (2, 8, 8, 64, 32, 3, 1),        # a 64-column strip wider than the row
    (1, 64, 64, 64, 64, 3, 1),      # 64 x 64 images: one strip per output-row pair
    (3, 10, 72, 64, 96, 3, 1),      # second strip holds 8 columns
    (2, 12, 12, 128, 200, 1, 0),    # 1 x 1 filter, ragged N
    (1, 6, 130, 64, 48, 5, 2),      # 3 strips, odd number of CTA tiles
]


@pytest.mark.parametrize("shape", POOL_SHAPES)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_conv_maxpool_exact_every_output(shape, out):
    Nb, H, W, C, Cout, R, pad = shape
    x = int_bf16((Nb, H, W, C), 61 + sum(shape))
    w = int_bf16((Cout, R, R, C), 62 + sum(shape))
    g = torch.Generator().manual_seed(sum(shape))
    scale = (2.0 ** torch.randint(0, 3, (Cout,), generator=g)).to(torch.bfloat16)
    bias = torch.randint(-20, 21, (Cout,), generator=g).to(torch.bfloat16)
    OH, OW = conv_out_hw(H, W, R, pad)
    PH, PW = OH // 2, OW // 2
    od = torch.float32 if out == "f32" else torch.bfloat16
    y = torch.full((Nb * PH * PW, Cout), float("nan"), dtype=od, device="cuda")
    with G.Plan(0, "nk") as p:
        p.conv2d_maxpool(x.cuda(), w.cuda(), y, bias.cuda(), True, pad=pad, scale=scale.cuda())
        assert p.status() == 0
        assert p.last_kernel == G.KERNEL_TC_PAIR
        assert p.workspace_bytes == 0
    pos = [(n, ph, pw) for n in range(Nb) for ph in range(PH) for pw in range(PW)]
    ref = oracle.conv2d_maxpool_at(x, w, pad, pos, scale=scale, bias=bias, relu=True)
    want = oracle.bf16_round(ref) if out == "bf16" else ref
    got = y.double().cpu().numpy()
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[0]}: {got[tuple(bad[0])]} vs {want[tuple(bad[0])]}"


def test_conv_maxpool_refusals():
    x = torch.zeros(1, 9, 9, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(32, 3, 3, 64, dtype=torch.bfloat16, device="cuda")
    with G.Plan(0, "nk") as p:
        # odd output size: incomplete pooling windows
        y = torch.empty(16, 32, device="cuda")
        with pytest.raises(G.GemmError) as e:
            p.conv2d_maxpool(x, w, y, pad=1)
        assert e.value.code == G.ERR_INVALID_ARG
        # 16 channels: not the implicit-GEMM operand
        x16 = torch.zeros(1, 8, 8, 16, dtype=torch.bfloat16, device="cuda")
        w16 = torch.zeros(32, 3, 3, 16, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(G.GemmError) as e:
            p.conv2d_maxpool(x16, w16, torch.empty(16, 32, device="cuda"), pad=1)
        assert e.value.code == G.ERR_UNSUPPORTED
