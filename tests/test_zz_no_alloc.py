"""gemm_run_noalloc: the entry point for callers that may not allocate device
memory (a process whose HBM is reserved up front by a pool or framework
allocator, or a latency-sensitive caller that cannot afford cudaMalloc's
device-wide synchronisation).  It packs misaligned operands into a fixed
scratch array that the library holds on each device instead of a plan
workspace.

Checked here through the C ABI: two calls in a row match the plan-based
gemm_run within the parity tolerance; small M (the single-CTA branch) and
K = 0 match the oracle exactly on integers; repeated calls change neither the
device's free memory nor torch's allocator; and a call whose packed operands
would not fit in the scratch is refused before anything runs.  Collected last so a
run that stops at the first failure has run every other test first; passes
alone in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from dnn_linear_layers_gb300 import gemm as G
from dnn_linear_layers_gb300.inputs import GemmCase

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dnn_linear_layers_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    return G.lib()


def _ld(t):
    return max(t.stride(0), t.shape[1], 1)


def run_noalloc(lib, A, B, C, bias, relu, b_nk, status=None):
    M, K = A.shape
    N = C.shape[1]
    epi = (G.EPI_BIAS if bias is not None else 0) | (G.EPI_RELU if relu else 0)
    return lib.gemm_run_noalloc(M, N, K, A.data_ptr(), _ld(A), B.data_ptr(), _ld(B),
                                bias.data_ptr() if bias is not None else None, C.data_ptr(), _ld(C),
                                epi, G.dtype_code(A.dtype, C.dtype), G.B_NK if b_nk else G.B_KN,
                                status.data_ptr() if status is not None else None,
                                torch.cuda.current_stream().cuda_stream)


def strided(t, extra_cols):
    """Copy of t inside a wider buffer: row pitch not a multiple of 16 bytes."""
    buf = torch.zeros(t.shape[0], t.shape[1] + extra_cols, dtype=t.dtype, device="cuda")
    buf[:, :t.shape[1]] = t.cuda()
    return buf[:, :t.shape[1]]


CASES = [
    # misaligned pitches on A, B and C: everything goes through the scratch
    (GemmCase("noalloc_kn", 700, 520, 333, bias=True, relu=True, out="bf16", seed=21), (1, 3, 1)),
    # Linear weight layout, fp32 out: A and W pitches misaligned, C aligned
    (GemmCase("noalloc_nk", 300, 1000, 1001, b_nk=True, bias=True, out="f32", seed=22), (1, 0, 0)),
]


def test_noalloc_matches_gemm_run_on_two_calls_in_a_row(lib):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for case, (pa, pb, pc) in CASES:
        A, B, bias = case.tensors()
        Ad = strided(A, pa) if pa else A.cuda()
        Bd = strided(B, pb) if pb else B.cuda()
        bd = bias.cuda() if bias is not None else None
        od = torch.float32 if case.out == "f32" else torch.bfloat16
        C_na = strided(torch.full((case.M, case.N), float("nan"), dtype=od), pc) if pc else \
            torch.full((case.M, case.N), float("nan"), dtype=od, device="cuda")
        rc = run_noalloc(lib, Ad, Bd, C_na, bd, case.relu, case.b_nk, status)
        assert rc == G.OK, G.strerror(rc)
        # the existing, plan-based entry point on the same operands
        with G.Plan(0, "nk" if case.b_nk else "kn") as p:
            C_run = torch.empty((case.M, case.N), dtype=od, device="cuda")
            p.run(Ad, Bd, C_run, bd, case.relu)
            assert p.status() == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        C_ref, S = oracle.gemm(A, B, bias=bias, relu=case.relu, b_nk=case.b_nk, with_mag=True)
        got = C_na.double().cpu().numpy()
        want = C_run.double().cpu().numpy()
        bound = oracle.tolerance(S, C_ref, out_bf16=(od == torch.bfloat16))
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got - want) <= bound), f"{case.name}: differs from gemm_run"
        ok, worst, _ = oracle.check_close(got, C_ref, S, out_bf16=(od == torch.bfloat16))
        assert ok, f"{case.name}: worst err/bound {worst:.3f}"


def test_noalloc_refuses_scratch_overflow_and_launches_nothing(lib):
    # A with a 4095-element pitch (8190 bytes) must be packed: 4100 x 4096 x 2 B > 32 MiB
    M, K, N = 4100, 4095, 64
    A = torch.ones(M, K, dtype=torch.bfloat16, device="cuda")
    B = torch.ones(K, N, dtype=torch.bfloat16, device="cuda")
    C = torch.full((M, N), 7.0, device="cuda")
    assert M * 4096 * 2 > 33554432 - 256
    rc = run_noalloc(lib, A, B, C, None, False, False)
    assert rc == G.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(C == 7.0)
    # the same product with an aligned pitch needs no scratch and runs
    A2 = torch.ones(M, 4096, dtype=torch.bfloat16, device="cuda")[:, :K]   # pitch 4096: aligned
    rc = run_noalloc(lib, A2, B, C, None, False, False)
    assert rc == G.OK
    torch.cuda.synchronize()
    assert torch.all(C == float(K))


SMALL_M = [
    # the single-CTA branch (M <= 128): misaligned A and B pitches, bias + ReLU
    (GemmCase("noalloc_m1", 1, 1000, 777, b_nk=True, bias=True, relu=True, out="bf16", integer=True, seed=31),
     (1, 3, 0)),
    (GemmCase("noalloc_m128", 128, 520, 333, bias=True, relu=True, out="f32", integer=True, seed=32), (1, 1, 1)),
]


@pytest.mark.parametrize("idx", range(len(SMALL_M)))
def test_noalloc_small_m_exact(lib, idx):
    case, (pa, pb, pc) = SMALL_M[idx]
    A, B, bias = case.tensors()
    Ad = strided(A, pa) if pa else A.cuda()
    Bd = strided(B, pb) if pb else B.cuda()
    od = torch.float32 if case.out == "f32" else torch.bfloat16
    C = strided(torch.full((case.M, case.N), float("nan"), dtype=od), pc) if pc else \
        torch.full((case.M, case.N), float("nan"), dtype=od, device="cuda")
    for _ in range(2):
        assert run_noalloc(lib, Ad, Bd, C, bias.cuda(), case.relu, case.b_nk) == G.OK
        torch.cuda.synchronize()
        ref = oracle.gemm(A, B, bias=bias, relu=case.relu, b_nk=case.b_nk)
        want = oracle.bf16_round(ref) if od == torch.bfloat16 else ref
        assert np.array_equal(C.double().cpu().numpy(), want), case.name


def test_noalloc_k0_misaligned_c(lib):
    """K = 0: C = epilogue(0) = ReLU(bias), written with any pitch."""
    M, N = 37, 50
    bias = torch.arange(-25, 25, dtype=torch.float32).to(torch.bfloat16).cuda()
    C = strided(torch.full((M, N), float("nan")), 3)
    A = torch.empty(M, 0, dtype=torch.bfloat16, device="cuda")
    B = torch.empty(0, N, dtype=torch.bfloat16, device="cuda")
    rc = lib.gemm_run_noalloc(M, N, 0, None, 0, None, 0, bias.data_ptr(), C.data_ptr(), _ld(C),
                              G.EPI_BIAS_RELU, G.BF16_F32OUT, G.B_KN, None, torch.cuda.current_stream().cuda_stream)
    assert rc == G.OK
    torch.cuda.synchronize()
    want = np.maximum(bias.double().cpu().numpy(), 0.0)[None, :].repeat(M, axis=0)
    assert np.array_equal(C.double().cpu().numpy(), want)
    del A, B


def test_noalloc_allocates_no_device_memory(lib):
    """Once a device is set up (first call: the scratch's address is looked up
    and the kernels used are loaded), further calls -- including ones that pack
    misaligned operands into the scratch -- change neither the device's free
    memory nor torch's allocator: nothing is allocated."""
    case, (pa, pb, pc) = CASES[0]
    A, B, bias = case.tensors()
    Ad, Bd, bd = strided(A, pa), strided(B, pb), bias.cuda()
    C = strided(torch.empty((case.M, case.N), dtype=torch.bfloat16), pc)
    A1, B1 = strided(A[:1], 1), strided(B.t().contiguous(), 3)      # M = 1, Linear weight layout
    C1 = torch.empty((1, case.N), dtype=torch.bfloat16, device="cuda")

    def calls():
        assert run_noalloc(lib, Ad, Bd, C, bd, True, False) == G.OK
        assert run_noalloc(lib, A1, B1, C1, bd, True, True) == G.OK
        torch.cuda.synchronize()

    calls()                                    # set-up and lazy kernel loading
    free0, alloc0 = torch.cuda.mem_get_info(0)[0], torch.cuda.memory_allocated(0)
    calls()
    calls()
    free1, alloc1 = torch.cuda.mem_get_info(0)[0], torch.cuda.memory_allocated(0)
    assert alloc1 == alloc0
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"


def test_noalloc_right_edge_inside_a_16_byte_granule(lib):
    """fp32 C with an aligned pitch and N = 523: nothing past column N is
    written (the epilogue stores such a C itself)."""
    M, N, K = 300, 523, 256
    A = torch.randint(-4, 5, (M, K), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    B = torch.randint(-4, 5, (K, N), generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    Cb = torch.full((M, 528), float("nan"), device="cuda")
    C = Cb[:, :N]
    assert run_noalloc(lib, A.cuda(), B.cuda(), C, None, False, False) == G.OK
    torch.cuda.synchronize()
    assert np.array_equal(C.double().cpu().numpy(), oracle.gemm(A, B))
    assert torch.isnan(Cb[:, N:]).all()
