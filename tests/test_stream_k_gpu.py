"""GPU parity of the stream-K split of the tensor-core kernels.

In a launch of at least one full wave of tiles, the tiles of the last, partial
wave of the persistent grid are split by k over the workers; each split
tile's contributors leave fp32 partials in the plan's workspace and the last
arrival of each 32-row slot adds them in contributor (k) order and applies the
epilogue.  Integer inputs keep every partial and every sum an exact integer
below 2^24, so results must equal the oracle exactly whatever the split; float
results must be within the usual bound and identical from run to run.
"""
import numpy as np
import pytest
import torch

import oracle
from dnn_linear_layers_gb300 import gemm as G
from dnn_linear_layers_gb300.inputs import GemmCase, int_bf16

from parity import compare, oracle_full, run_case

pytestmark = pytest.mark.gpu

# (M, N, K): tiles of 256 x 256 for pairs (128 x 256 for single CTAs) against
# 74-76 pairs (148-152 CTAs); with a minimum of 1 atom per worker (the option)
# every shape below splits its last wave
SHAPES = [
    (4096, 2048, 1024),    # 128 tiles: 1 wave + 52 split tiles, 16 atoms each
    (4096, 4096, 200),     # 256 tiles, 4 atoms, ragged K
    (3000, 5000, 2048),    # ragged edges, 240 tiles: 3 whole waves + 12 split tiles
    (4096, 4096, 520),     # 256 tiles, 9 atoms (odd: a one-atom last stage)
    (20000, 768, 333),     # 237 tiles, ragged K
    (9984, 2048, 4096),    # 312 tiles: 4 waves + 8 split tiles, long K: many contributors per tile
]


@pytest.fixture(scope="module")
def plans():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dnn_linear_layers_gb300 import build
    build.build()
    kn, nk = G.Plan(0, "kn"), G.Plan(0, "nk")
    yield {"kn": kn, "nk": nk}
    kn.close(); nk.close()


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("b_nk", [False, True])
@pytest.mark.parametrize("kernel", [G.KERNEL_TC_PAIR, G.KERNEL_TC_SINGLE])
def test_stream_k_integer_exact(plans, shape, b_nk, kernel):
    M, N, K = shape
    p = plans["nk" if b_nk else "kn"]
    p.set_option(G.OPT_STREAM_K, 1)
    case = GemmCase("sk_int", M, N, K, b_nk=b_nk, bias=True, relu=True, out="bf16", integer=True, seed=M + N + K)
    A, B, bias, C = run_case(p, case, kernel=kernel)
    assert p.last_kernel == kernel
    assert p.workspace_bytes > 0          # the split tiles' partials (no operand is packed here)
    C_ref, S = oracle_full(case, A, B, bias)
    compare(case, C, C_ref, S)


@pytest.mark.parametrize("shape", [(4096, 2048, 1024), (3000, 5000, 2048), (9984, 2048, 4096)])
def test_stream_k_float_deterministic_and_within_tolerance(plans, shape):
    """Float inputs: within the bound, bit-identical over repeated runs (the
    partials are added in k order whichever contributor arrives last), and
    within the bound of the unsplit result."""
    M, N, K = shape
    p = plans["kn"]
    p.set_option(G.OPT_STREAM_K, 1)
    case = GemmCase("sk_f", M, N, K, out="f32", seed=K)
    A, B, _ = case.tensors()
    Ad, Bd = A.cuda(), B.cuda()
    outs = []
    for _ in range(3):
        C = torch.empty(M, N, device="cuda")
        p.run(Ad, Bd, C)
        assert p.status() == 0
        outs.append(C.cpu())
    assert all(torch.equal(outs[0].view(torch.int32), o.view(torch.int32)) for o in outs[1:])
    C_ref, S = oracle.gemm(A, B, with_mag=True)
    compare(case, outs[0], C_ref, S)
    with G.Plan(0, "kn") as q:
        q.set_option(G.OPT_STREAM_K, 0)
        C0 = torch.empty(M, N, device="cuda")
        q.run(Ad, Bd, C0)
        assert q.status() == 0
    diff = np.abs(outs[0].double().numpy() - C0.double().cpu().numpy())
    assert np.all(diff <= 2 * oracle.tolerance(S))


@pytest.mark.parametrize("min_atoms", [0, 1, 2, 8, 64])
def test_stream_k_min_atoms_option(min_atoms):
    """Every split granularity (and none, the default) gives the exact result."""
    M, N, K = 4096, 2304, 1000
    with G.Plan(0, "nk") as p:
        p.set_option(G.OPT_STREAM_K, min_atoms)
        case = GemmCase("sk_opt", M, N, K, b_nk=True, bias=True, out="f32", integer=True, seed=min_atoms)
        A, B, bias, C = run_case(p, case)
        C_ref, S = oracle_full(case, A, B, bias)
        compare(case, C, C_ref, S)


def test_stream_k_extended_epilogue_exact():
    """alpha, per-column scale, bias, beta * previous C and ReLU applied by the
    last arrival of each split slot."""
    M, N, K = 4096, 2560, 2000
    A = int_bf16((M, K), 1)
    B = int_bf16((K, N), 2)
    scale = int_bf16((N,), 3, lo=-2, hi=2)
    bias = int_bf16((N,), 4, lo=-8, hi=8)
    C0 = int_bf16((M, N), 5, lo=-16, hi=16).float()
    C = C0.cuda()
    with G.Plan(0, "kn") as p:
        p.set_option(G.OPT_STREAM_K, 8)
        p.run(A.cuda(), B.cuda(), C, bias.cuda(), True, alpha=0.5, beta=-2.0, scale=scale.cuda())
        assert p.status() == 0 and p.workspace_bytes > 0
    ref, _ = oracle.gemm_ex(A, B, alpha=0.5, beta=-2.0, C0=C0.double().numpy(), scale=scale, bias=bias, relu=True)
    assert np.array_equal(C.double().cpu().numpy(), ref)


@pytest.mark.parametrize("fmt", ["e4m3", "tf32"])
def test_stream_k_other_operand_types_exact(fmt):
    M, N, K = 4096, 2560, 1536
    g = torch.Generator().manual_seed(9)
    dt = {"e4m3": torch.float8_e4m3fn, "tf32": torch.float32}[fmt]
    A = torch.randint(-4, 5, (M, K), generator=g).to(dt)
    B = torch.randint(-4, 5, (N, K), generator=g).to(dt)
    C = torch.empty(M, N, device="cuda")
    with G.Plan(0, "nk") as p:
        p.set_option(G.OPT_STREAM_K, 8)
        p.run(A.cuda(), B.cuda(), C)
        assert p.status() == 0 and p.workspace_bytes > 0
    assert np.array_equal(C.double().cpu().numpy(), oracle.gemm(A, B, b_nk=True))


def test_stream_k_timeout_then_clean_run():
    """A run aborted by the fault-injection hook may leave arrival counters
    behind; gemm_plan_status reports the timeout and clears them, so the next
    run is exact."""
    M, N, K = 4096, 2560, 2048
    A = int_bf16((M, K), 11)
    B = int_bf16((K, N), 12)
    ref = oracle.gemm(A, B)
    Ad, Bd = A.cuda(), B.cuda()
    with G.Plan(0, "kn") as p:
        p.set_option(G.OPT_STREAM_K, 8)
        p.set_timeout_ns(20_000_000)
        C = torch.empty(M, N, device="cuda")
        p.set_debug(1)
        p.run(Ad, Bd, C)
        assert p.status() == G.ERR_DEVICE_TIMEOUT
        p.set_debug(0)
        for _ in range(2):
            C = torch.empty(M, N, device="cuda")
            p.run(Ad, Bd, C)
            assert p.status() == 0
            assert np.array_equal(C.double().cpu().numpy(), ref)


def test_stream_k_implicit_conv_exact():
    """Implicit-GEMM convolution (A through the im2col tensor map) with split
    tiles: every output exact against the direct convolution."""
    Nb, H, W, C, Cout, R, pad = 8, 56, 56, 128, 256, 3, 1   # 98 tiles: 1 wave + 22 split tiles
    x = int_bf16((Nb, H, W, C), 21)
    w = int_bf16((Cout, R, R, C), 22)
    with G.Plan(0, "nk") as p:
        p.set_option(G.OPT_STREAM_K, 8)
        y = torch.full((Nb * H * W, Cout), float("nan"), device="cuda")
        p.conv2d(x.cuda(), w.cuda(), y, pad=pad)
        assert p.status() == 0 and p.last_kernel == G.KERNEL_TC_PAIR and p.workspace_bytes > 0
    pos = [(n, oh, ow) for n in range(Nb) for oh in range(H) for ow in range(W)]
    assert np.array_equal(y.double().cpu().numpy(), oracle.conv2d_at(x, w, pad, pos))
