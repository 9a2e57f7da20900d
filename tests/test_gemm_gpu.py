"""GPU parity tests: the CUDA path through the C ABI against the float64 oracle.

Sizes span several 256 x 256 tiles with ragged tails in M, N and K and stay
small enough for the oracle to finish in seconds.  Integer cases must match
exactly; float cases within 1e-3 * sum|a b| + 1e-6 (+ one output ulp for a
16-bit output).  Every run checks a NaN guard band around C.
"""
import numpy as np
import pytest
import torch

import oracle
from dnn_linear_layers_gb300 import gemm as G
from dnn_linear_layers_gb300.inputs import GemmCase, SMALL_F32, int_bf16

from parity import alloc_with_guard, compare, guard_intact, oracle_full, run_case

pytestmark = pytest.mark.gpu

KERNELS = {"single": G.KERNEL_TC_SINGLE, "pair": G.KERNEL_TC_PAIR, "skinny": G.KERNEL_SKINNY,
           "auto": G.KERNEL_AUTO}


@pytest.fixture(scope="module")
def plans():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dnn_linear_layers_gb300 import build
    build.build()
    kn = G.Plan(0, "kn")
    nk = G.Plan(0, "nk")
    yield {"kn": kn, "nk": nk}
    kn.close(); nk.close()


def plan_for(plans, case):
    return plans["nk" if case.b_nk else "kn"]


def check(plans, case, kernel=None):
    p = plan_for(plans, case)
    A, B, bias, C = run_case(p, case, kernel=KERNELS.get(kernel, kernel) if kernel else G.KERNEL_AUTO)
    if kernel and kernel != "auto":
        assert p.last_kernel == KERNELS.get(kernel, kernel)
    C_ref, S = oracle_full(case, A, B, bias)
    return compare(case, C, C_ref, S)


# ------------------------------------------------------------ first slice
@pytest.mark.parametrize("kernel", ["single", "pair"])
@pytest.mark.parametrize("b_nk", [False, True])
def test_one_tile_integer_exact(plans, kernel, b_nk):
    check(plans, GemmCase("one_tile", 256, 256, 64, b_nk=b_nk, out="f32", integer=True), kernel)


@pytest.mark.parametrize("kernel", ["single", "pair"])
def test_config_512_f32_out(plans, kernel):
    """M=N=K=512, N(0,1) bf16 inputs from seed 0, fp32 output, no epilogue."""
    check(plans, SMALL_F32, kernel)


@pytest.mark.parametrize("kernel", ["single", "pair"])
@pytest.mark.parametrize("b_nk", [False, True])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_integer_exact_ragged(plans, kernel, b_nk, out):
    check(plans, GemmCase("int_ragged", 600, 700, 333, b_nk=b_nk, out=out, integer=True, seed=3), kernel)


@pytest.mark.parametrize("kernel", ["single", "pair"])
@pytest.mark.parametrize("epi", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("b_nk", [False, True])
def test_epilogues_integer_exact(plans, kernel, epi, b_nk):
    bias, relu = epi
    check(plans, GemmCase("int_epi", 520, 530, 200, b_nk=b_nk, bias=bias, relu=relu, out="bf16",
                          integer=True, seed=5), kernel)


@pytest.mark.parametrize("kernel", ["single", "pair"])
@pytest.mark.parametrize("b_nk", [False, True])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_float_within_tolerance(plans, kernel, b_nk, out):
    check(plans, GemmCase("float_ragged", 700, 600, 1000, b_nk=b_nk, out=out, bias=True, relu=True,
                          seed=7), kernel)


@pytest.mark.parametrize("out", ["f32", "f16"])
@pytest.mark.parametrize("integer", [True, False])
def test_fp16_inputs(plans, out, integer):
    check(plans, GemmCase("fp16", 384, 520, 264, in_dtype="f16", out=out, integer=integer, bias=True, seed=9))


TAILS = [1, 7, 127, 129, 255, 257]


@pytest.mark.parametrize("kernel", ["auto", "single", "pair"])
@pytest.mark.parametrize("M", TAILS)
@pytest.mark.parametrize("N", [8, 129, 264])
@pytest.mark.parametrize("K", [8, 72, 264])
def test_tails_integer_exact(plans, M, N, K, kernel):
    check(plans, GemmCase("tails", M, N, K, out="f32", integer=True, seed=M + N + K), kernel)


@pytest.mark.parametrize("kernel", ["single", "pair"])
@pytest.mark.parametrize("b_nk", [False, True])
@pytest.mark.parametrize("shape", [(4096, 4096, 72), (2304, 4352, 40)])
def test_last_wave_split_into_halves_integer_exact(plans, kernel, b_nk, shape):
    """Shapes whose last persistent wave is partial, with stream-K off: its
    tiles run as two 128-column halves (whole tiles first, then halves); every
    output checked."""
    M, N, K = shape
    with G.Plan(0, "nk" if b_nk else "kn") as p:
        p.set_option(G.OPT_STREAM_K, 0)
        case = GemmCase("tail_split", M, N, K, b_nk=b_nk, bias=True, out="bf16", integer=True, seed=K)
        A, B, bias, C = run_case(p, case, kernel=KERNELS[kernel])
        assert p.workspace_bytes == 0
        C_ref, S = oracle_full(case, A, B, bias)
        compare(case, C, C_ref, S)


@pytest.mark.parametrize("option,value", [(G.OPT_GROUP_M, 1), (G.OPT_GROUP_M, 8), (G.OPT_GROUP_M, 16),
                                          (G.OPT_TAIL_SPLIT, 0),
                                          (G.OPT_K_SNAKE, 0), (G.OPT_PDL, 0), (G.OPT_L2_POLICY, 1),
                                          (G.OPT_L2_POLICY, 2), (G.OPT_SKINNY_SPLITS, 1),
                                          (G.OPT_SKINNY_STAGES, 2), (G.OPT_GEMV_MAX_M, 4), (G.OPT_STREAM_K, 0),
                                          (G.OPT_STREAM_K, 1), (G.OPT_WARP_MMA_MAX_M, 0),
                                          (G.OPT_WARP_MMA_MAX_M, 8)])
@pytest.mark.parametrize("shape", [(1300, 530, 200), (4096, 4096, 72), (16, 1000, 1000)])
def test_scheduling_options_change_no_result(plans, option, value, shape):
    """Every plan option only reschedules work: the results stay exact on
    integers (large shapes on the paired kernel, M = 16 on the small-M one)."""
    M, N, K = shape
    p = G.Plan(0, "nk")
    default = p.get_option(option)
    p.set_option(option, value)
    assert p.get_option(option) == value
    case = GemmCase("options", M, N, K, b_nk=True, bias=True, relu=True, out="bf16", integer=True, seed=M)
    A, B, bias, C = run_case(p, case)
    C_ref, S = oracle_full(case, A, B, bias)
    compare(case, C, C_ref, S)
    p.set_option(option, default)
    assert p.get_option(option) == default
    p.close()


def test_option_ranges_are_checked(plans):
    p = G.Plan(0)
    for option, bad in [(G.OPT_GROUP_M, -1), (G.OPT_GROUP_M, 1025), (G.OPT_TAIL_SPLIT, 2), (G.OPT_L2_POLICY, 3),
                        (G.OPT_SKINNY_SPLITS, 3), (G.OPT_SKINNY_STAGES, 1), (G.OPT_SKINNY_STAGES, 9),
                        (G.OPT_GEMV_MAX_M, 5), (G.OPT_STREAM_K, -1), (G.OPT_STREAM_K, 5000),
                        (G.OPT_WARP_MMA_MAX_M, -1), (G.OPT_WARP_MMA_MAX_M, 17), (0, 0), (8, 0),
                        (99, 0)]:
        before = p.get_option(option) if option in G.OPTIONS else None
        with pytest.raises(G.GemmError):
            p.set_option(option, bad)
        if before is not None:
            assert p.get_option(option) == before
    p.close()


# ------------------------------------------------------------ skinny-M path
@pytest.mark.parametrize("M", [1, 2, 15, 16, 17, 64, 100, 128])
@pytest.mark.parametrize("b_nk", [True, False])
def test_skinny_integer_exact(plans, M, b_nk):
    check(plans, GemmCase("skinny_int", M, 1000, 1000, b_nk=b_nk, bias=True, relu=True, out="bf16",
                          integer=True, seed=M), "skinny")


@pytest.mark.parametrize("M,N,K", [(1, 128, 4096), (3, 300, 520), (16, 4096, 64), (33, 700, 2000), (128, 257, 8)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_skinny_float_within_tolerance(plans, M, N, K, out):
    check(plans, GemmCase("skinny_f", M, N, K, b_nk=True, bias=True, out=out, b_std=K ** -0.5, seed=N), "skinny")


@pytest.mark.parametrize("out", ["f32", "f16"])
def test_skinny_fp16(plans, out):
    check(plans, GemmCase("skinny_h", 16, 520, 1000, b_nk=True, in_dtype="f16", out=out, integer=True,
                          bias=True, seed=4), "skinny")


@pytest.mark.parametrize("b_const", [False, True])
def test_skinny_chained_layers_see_previous_outputs(plans, b_const):
    """Back-to-back layers on one stream, each reading the previous layer's
    output: with programmatic dependent launch (and constant-weight prefetch)
    no kernel may read its input before the producing kernel is done.
    Integer data keeps every value exact (|y1| <= 128 fits bf16)."""
    p = G.Plan(0, "nk", b_const=b_const)
    p.set_kernel(G.KERNEL_SKINNY)
    M, D = 16, 128
    Ws = [int_bf16((D, D), 40 + i, lo=-1, hi=1) for i in range(6)]
    x = int_bf16((M, D), 39, lo=-1, hi=1)
    Wd = [w.cuda() for w in Ws]
    h = x.cuda()
    outs = []
    for i, w in enumerate(Wd):       # alternate a 0/1 clamp layer to keep values small
        y = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
        p.run(h, w, y, relu=True)
        h = torch.clamp(y, max=1.0) if i % 2 else y
        outs.append(h)
    assert p.status() == 0
    ref = x.double().numpy()
    for i, w in enumerate(Ws):
        ref = oracle.gemm(ref, w, relu=True, b_nk=True)
        ref = oracle.bf16_round(ref)
        if i % 2:
            ref = np.minimum(ref, 1.0)
        assert np.array_equal(outs[i].double().cpu().numpy(), ref), f"layer {i}"
    p.close()


def test_skinny_is_auto_choice_for_small_m(plans):
    """17 <= M <= 128: the tensor-core small-M kernel (M = 1 with an N x K
    weight takes the CUDA-core GEMV, 2 <= M <= 16 the warp-MMA kernel:
    tests/test_gemv_gpu.py, tests/test_warp_mma_gpu.py)."""
    p = plans["nk"]
    A = torch.ones(20, 256, dtype=torch.bfloat16, device="cuda")
    W = torch.ones(512, 256, dtype=torch.bfloat16, device="cuda")
    C = torch.empty(20, 512, device="cuda")
    p.set_kernel(G.KERNEL_AUTO)
    p.run(A, W, C)
    assert p.status() == 0 and p.last_kernel == G.KERNEL_SKINNY
    assert torch.all(C == 256.0)


@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (129, 77, 1000), (257, 1001, 99)])
@pytest.mark.parametrize("b_nk", [False, True])
def test_misaligned_strides_are_packed(plans, shape, b_nk):
    """Row lengths whose byte size is not a multiple of 16 go through the pack path."""
    M, N, K = shape
    check(plans, GemmCase("misaligned", M, N, K, b_nk=b_nk, out="bf16", integer=True, bias=True, seed=11))


def test_odd_1000_cube(plans):
    check(plans, GemmCase("odd1000", 1000, 1000, 1000, out="bf16", seed=1))


def test_k_zero_writes_epilogue(plans):
    p = plans["kn"]
    M, N = 37, 45
    bias = torch.linspace(-2, 2, N, dtype=torch.bfloat16, device="cuda")
    buf, C, iv, bits = alloc_with_guard(M, N, torch.float32)
    A = torch.empty((M, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((0, N), dtype=torch.bfloat16, device="cuda")
    p.run(A, B, C, bias, relu=True)
    assert p.status() == 0 and p.last_kernel == G.KERNEL_FILL
    assert guard_intact(buf, M, N, iv, bits)
    expect = torch.clamp(bias.float(), min=0).expand(M, N).cpu()
    assert torch.equal(C.cpu(), expect)


def test_empty_is_noop(plans):
    p = plans["kn"]
    before = p.launch_count
    C = torch.full((0, 5), 3.0, device="cuda")
    p.run(torch.empty((0, 4), dtype=torch.bfloat16, device="cuda"),
          torch.empty((4, 5), dtype=torch.bfloat16, device="cuda"), C)
    assert p.launch_count == before


def test_misaligned_bias_pointer(plans):
    p = plans["kn"]
    case = GemmCase("bias_off", 300, 264, 128, bias=True, out="f32", integer=True, seed=13)
    A, B, bias = case.tensors()
    big = torch.zeros(case.N + 1, dtype=torch.bfloat16)
    big[1:] = bias
    bias_dev = big.cuda()[1:]            # 2-byte offset: not 16-byte aligned
    C = torch.empty(case.M, case.N, device="cuda")
    p.run(A.cuda(), B.cuda(), C, bias_dev)
    assert p.status() == 0
    C_ref, S = oracle.gemm(A, B, bias=bias, with_mag=True)
    compare(case, C.cpu(), C_ref, S)


def test_non_default_stream(plans):
    p = plans["kn"]
    case = GemmCase("stream", 512, 512, 256, out="f32", integer=True, seed=17)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        A, B, bias, C = run_case(p, case, stream=s)
    C_ref, S = oracle_full(case, A, B, bias)
    compare(case, C, C_ref, S)


def test_deterministic_bits(plans):
    p = plans["kn"]
    case = GemmCase("det", 640, 768, 1024, out="f32", seed=19)
    A, B, _ = case.tensors()
    A, B = A.cuda(), B.cuda()
    outs = []
    for _ in range(5):
        C = torch.empty(case.M, case.N, device="cuda")
        p.run(A, B, C)
        outs.append(C.cpu())
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_packing_disabled_reports_alignment(plans):
    p = G.Plan(0, "kn")
    p.set_packing(False)
    A = torch.ones(8, 7, dtype=torch.bfloat16, device="cuda")
    B = torch.ones(7, 8, dtype=torch.bfloat16, device="cuda")
    C = torch.empty(8, 8, device="cuda")
    with pytest.raises(G.GemmError) as ei:
        p.run(A, B, C)
    assert ei.value.code == G.ERR_ALIGNMENT
    p.close()


@pytest.mark.parametrize("kernel", ["single", "pair"])
def test_bounded_wait_reports_timeout_and_context_survives(plans, kernel):
    """Fault injection on the host's request: the MMA warp withholds the first
    'accumulator ready' signal, the epilogue's bounded wait runs out, the run
    reports GEMM_ERR_DEVICE_TIMEOUT, and the next run on the same context is
    correct."""
    p = G.Plan(0, "kn")
    p.set_kernel(KERNELS[kernel])
    p.set_timeout_ns(20_000_000)          # 20 ms
    # one tile and one k-block; then several tiles per worker and a long K, so
    # the abort comes while issued copies are still in flight (the exit path
    # must let them land before shared memory is released)
    for M, K in ((256, 64), (4096, 2048)):
        p.set_debug(1)
        A = torch.ones(M, K, dtype=torch.bfloat16, device="cuda")
        B = torch.ones(K, M, dtype=torch.bfloat16, device="cuda")
        C = torch.zeros(M, M, device="cuda")
        p.run(A, B, C)
        assert p.status() == G.ERR_DEVICE_TIMEOUT
        p.set_debug(0)
        p.run(A, B, C)
        assert p.status() == 0
        assert torch.all(C == float(K))
    p.close()


@pytest.mark.parametrize("kernel", ["single", "pair"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("offs", [(0, 0, 1), (1, 3, 0), (5, 2, 3), (7, 7, 7)])
def test_unaligned_operands_and_direct_c_store(plans, kernel, out, offs):
    """A, B and C views starting 0..7 elements past a 16-byte boundary with odd
    pitches: A and B go through the realigning pack (interior 16-byte pieces by
    funnel shift, the first and last of each row byte by byte) in one launch,
    and C is written by the epilogue itself (any pitch, any alignment of its
    type); exact on integers, nothing outside C touched, beta * C read in place."""
    oa, ob, oc = offs
    M, N, K = 700, 523, 1037
    A = int_bf16((M, K), 71)
    B = int_bf16((K, N), 72)
    C0 = int_bf16((M, N), 73, lo=-8, hi=8).float()
    od = torch.float32 if out == "f32" else torch.bfloat16
    Ab = torch.zeros(M, K + 9, dtype=torch.bfloat16, device="cuda")
    Bb = torch.zeros(K, N + 9, dtype=torch.bfloat16, device="cuda")
    Ab[:, oa:oa + K] = A.cuda()
    Bb[:, ob:ob + N] = B.cuda()
    Cb = torch.full((M + 2, N + 9), float("nan"), dtype=od, device="cuda")
    Cv = Cb[1:M + 1, oc:oc + N]
    Cv.copy_(C0.to(od).cuda())
    p = G.Plan(0, "kn")
    p.set_kernel(KERNELS[kernel])
    p.run(Ab[:, oa:oa + K], Bb[:, ob:ob + N], Cv, relu=True, beta=2.0)
    assert p.status() == 0 and p.last_kernel == KERNELS[kernel]
    ref, _ = oracle.gemm_ex(A, B, beta=2.0, C0=C0.double().numpy(), relu=True)
    want = oracle.bf16_round(ref) if out == "bf16" else ref
    assert np.array_equal(Cv.double().cpu().numpy(), want)
    mask = torch.ones(M + 2, N + 9, dtype=torch.bool)
    mask[1:M + 1, oc:oc + N] = False
    assert torch.isnan(Cb.cpu()[mask].float()).all(), "write outside C"
    p.close()


@pytest.mark.parametrize("kernel", ["single", "pair"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("N", [513, 519, 520, 523, 527])
def test_right_edge_inside_a_16_byte_granule_is_not_overwritten(plans, kernel, out, N):
    """C with a 16-byte aligned base and pitch whose right edge (N x element
    size) is not a multiple of 16 bytes: the columns past N up to the next
    16-byte boundary belong to the caller and must keep their contents (a TMA
    store would write the whole granule, so the epilogue stores such a C
    itself)."""
    M, K = 300, 256
    od = torch.float32 if out == "f32" else torch.bfloat16
    per = 16 // (4 if out == "f32" else 2)
    ld = (N + per - 1) // per * per + per
    A = int_bf16((M, K), N)
    B = int_bf16((K, N), N + 1)
    Cb = torch.full((M + 2, ld), float("nan"), dtype=od, device="cuda")
    Cv = Cb[1:M + 1, :N]
    p = plans["kn"]
    p.set_kernel(KERNELS[kernel])
    p.run(A.cuda(), B.cuda(), Cv, relu=True)
    assert p.status() == 0
    ref = oracle.gemm(A, B, relu=True)
    want = oracle.bf16_round(ref) if out == "bf16" else ref
    assert np.array_equal(Cv.double().cpu().numpy(), want)
    mask = torch.ones(M + 2, ld, dtype=torch.bool)
    mask[1:M + 1, :N] = False
    assert torch.isnan(Cb.cpu()[mask].float()).all(), "write outside C"
