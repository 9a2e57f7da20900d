"""GPU parity for a transposed A operand (plan flag GEMM_A_KM: A stored K x M,
the BLAS "transa" of the GEMM interface): the tensor-core kernels read A as an
MN-major operand.  The oracle gets the M x K matrix the stored K x M tensor
represents.  Integer cases are exact; float cases within 1e-3 * sum|a b| + 1e-6
(+ one output ulp for a 16-bit output), as in the other GEMM parity tests.
"""
import pytest
import torch

from dnn_linear_layers_gb300 import gemm as G
from dnn_linear_layers_gb300.inputs import GemmCase

from parity import alloc_with_guard, compare, guard_intact, oracle_full, out_dtype_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def plans():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dnn_linear_layers_gb300 import build
    build.build()
    ps = {lay: G.Plan(0, lay, a_layout="km") for lay in ("kn", "nk")}
    yield ps
    for p in ps.values():
        p.close()


def run_km(plans, case, kernel=G.KERNEL_AUTO, a_pitch=None, alpha=1.0, beta=0.0):
    """Run `case` with A handed over as its K x M transpose (row pitch a_pitch >= M)."""
    p = plans["nk" if case.b_nk else "kn"]
    A, B, bias = case.tensors()
    At = A.t().contiguous()
    if a_pitch is not None:
        full = torch.zeros(case.K, a_pitch, dtype=A.dtype)
        full[:, :case.M] = At
        Ad = full.cuda()[:, :case.M]          # the view keeps the pitch
        assert Ad.stride(0) == a_pitch
    else:
        Ad = At.cuda()
    Bd = B.cuda()
    biasd = bias.cuda() if bias is not None else None
    odt = out_dtype_of(case)
    buf, C, iv, bits = alloc_with_guard(case.M, case.N, odt)
    p.set_kernel(kernel)
    if alpha != 1.0 or beta != 0.0:
        p.run(Ad, Bd, C, biasd, relu=case.relu, alpha=alpha, beta=beta)
    else:
        p.run(Ad, Bd, C, biasd, relu=case.relu)
    assert p.status() == 0
    if kernel != G.KERNEL_AUTO:
        assert p.last_kernel == kernel
    else:
        assert p.last_kernel == G.KERNEL_TC_PAIR     # also for small M: the small-M kernel takes M x K A only
    assert guard_intact(buf, case.M, case.N, iv, bits)
    C_ref, S = oracle_full(case, A, B, bias)
    return compare(case, C.cpu(), C_ref, S)


@pytest.mark.parametrize("kernel", [G.KERNEL_TC_SINGLE, G.KERNEL_TC_PAIR])
@pytest.mark.parametrize("b_nk", [False, True])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_transposed_a_integer_exact_ragged(plans, kernel, b_nk, out):
    run_km(plans, GemmCase("km_int", 600, 700, 333, b_nk=b_nk, out=out, integer=True, seed=11), kernel)


@pytest.mark.parametrize("shape", [(1, 8, 8), (16, 300, 72), (128, 257, 130), (129, 64, 64), (513, 520, 1000)])
def test_transposed_a_shapes_integer_exact(plans, shape):
    M, N, K = shape
    run_km(plans, GemmCase("km_shape", M, N, K, b_nk=True, bias=True, relu=True, out="bf16", integer=True,
                           seed=M + N + K))


@pytest.mark.parametrize("kernel", [G.KERNEL_TC_SINGLE, G.KERNEL_TC_PAIR])
@pytest.mark.parametrize("b_nk", [False, True])
def test_transposed_a_float_within_tolerance(plans, kernel, b_nk):
    run_km(plans, GemmCase("km_float", 1000, 1100, 700, b_nk=b_nk, out="f32", seed=12), kernel)


@pytest.mark.parametrize("out", ["f32", "f16"])
def test_transposed_a_fp16(plans, out):
    run_km(plans, GemmCase("km_f16", 300, 400, 200, b_nk=False, out=out, in_dtype="f16", integer=True, seed=13))


def test_transposed_a_packed_pitch(plans):
    # a row pitch of M + 3 elements breaks the 16-byte rule: A is packed first
    run_km(plans, GemmCase("km_pack", 250, 260, 270, b_nk=True, out="f32", integer=True, seed=14), a_pitch=253)


def test_transposed_a_large_integer_exact(plans):
    run_km(plans, GemmCase("km_big", 2048, 2304, 512, b_nk=False, out="f32", integer=True, seed=15))


def test_transposed_a_refusals(plans):
    p = plans["nk"]
    A = torch.zeros(64, 32, dtype=torch.bfloat16, device="cuda")      # K x M
    B = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(32, 16, dtype=torch.float32, device="cuda")
    p.set_kernel(G.KERNEL_SKINNY)
    with pytest.raises(G.GemmError):
        p.run(A, B, C)
    p.set_kernel(G.KERNEL_AUTO)


@pytest.mark.parametrize("kernel", [G.KERNEL_TC_SINGLE, G.KERNEL_TC_PAIR])
def test_transposed_a_extended_epilogue_integer_exact(plans, kernel):
    # t = alpha * acc * scale + bias + beta * C_old, ReLU, with every step exact in
    # fp32 (alpha a power of two, integers well under 2^24)
    import oracle
    from dnn_linear_layers_gb300.inputs import int_bf16
    M, N, K = 300, 520, 64
    A = int_bf16((M, K), 60)
    B = int_bf16((N, K), 61)
    scale = int_bf16((N,), 62)
    bias = int_bf16((N,), 63)
    C0 = int_bf16((M, N), 64).float()
    p = plans["nk"]
    p.set_kernel(kernel)
    C = C0.cuda().clone()
    p.run(A.t().contiguous().cuda(), B.cuda(), C, bias.cuda(), relu=True, alpha=0.5, beta=2.0, scale=scale.cuda())
    assert p.status() == 0
    ref, _ = oracle.gemm_ex(A, B, alpha=0.5, beta=2.0, C0=C0, scale=scale, bias=bias, relu=True, b_nk=True)
    assert (C.double().cpu().numpy() == ref).all()
