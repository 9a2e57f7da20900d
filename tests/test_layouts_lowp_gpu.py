"""GPU parity of the fp8 (e4m3 / e5m2) and tf32 operand types in every
operand layout: B stored K x N or N x K, A stored M x K or K x M (plan flag
GEMM_A_KM).  The tensor-core kernels read an fp8 K x N B or K x M A as an
MN-major operand (boxes one 128-byte swizzle row wide, 128 columns); the
small-M kernel reads a K x N fp8 weight the same way.  A tf32 operand stored
MN-major is first transposed into the plan's workspace (the tensor cores take
tf32 K-major only).

Small integers (-4..4) are exact in all three formats and every partial sum is
an integer below 2^24, so an fp32 output must equal the oracle exactly and a
bf16 output its round-to-nearest-even.  Shapes span several tiles with ragged
M, N and K edges; the oracle gets the M x K and K x N (or N x K) matrices the
stored tensors represent.
"""
import numpy as np
import pytest
import torch

import oracle
from dnn_linear_layers_gb300 import gemm as G

from parity import alloc_with_guard, guard_intact

pytestmark = pytest.mark.gpu

FMT = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2, "tf32": torch.float32}
OUT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dnn_linear_layers_gb300 import build
    build.build()


def ints(shape, seed, fmt, lo=-4, hi=4):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g).to(FMT[fmt])


def run_layout(fmt, out, M, N, K, b_layout, a_layout, kernel, seed, bias=True, relu=True, opts=()):
    """Run one integer case through the C ABI; return (C on the host, expected)."""
    A = ints((M, K), seed, fmt)
    B = ints((N, K) if b_layout == "nk" else (K, N), seed + 1, fmt)
    bv = ints((N,), seed + 2, "e4m3", -8, 8).to(torch.bfloat16) if bias else None
    Ad = (A.t().contiguous() if a_layout == "km" else A).cuda()
    buf, C, iv, bits = alloc_with_guard(M, N, OUT[out])
    with G.Plan(0, b_layout, a_layout=a_layout) as p:
        for o, v in opts:
            p.set_option(o, v)
        p.set_kernel(kernel)
        p.run(Ad, B.cuda(), C, bv.cuda() if bv is not None else None, relu)
        assert p.status() == 0
        if kernel != G.KERNEL_AUTO:
            assert p.last_kernel == kernel
        last = p.last_kernel
    assert guard_intact(buf, M, N, iv, bits)
    ref = oracle.gemm(A, B, bias=bv, relu=relu, b_nk=b_layout == "nk")
    want = oracle.bf16_round(ref) if out == "bf16" else ref
    return C.double().cpu().numpy(), want, last


def assert_equal(got, want, what):
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first {bad[0]}: {got[tuple(bad[0])]} vs {want[tuple(bad[0])]}"


LAYOUTS = [("kn", "mk"), ("kn", "km"), ("nk", "km")]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "tf32"])
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("kernel", [G.KERNEL_TC_PAIR, G.KERNEL_TC_SINGLE])
@pytest.mark.parametrize("shape", [(300, 264, 260), (600, 700, 333), (129, 136, 128)])
def test_lowp_layouts_integer_exact(fmt, layout, kernel, shape):
    M, N, K = shape
    b_layout, a_layout = layout
    got, want, _ = run_layout(fmt, "f32", M, N, K, b_layout, a_layout, kernel, seed=M + N + K)
    assert_equal(got, want, f"{fmt} {layout} {shape}")


@pytest.mark.parametrize("fmt", ["e4m3", "tf32"])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_lowp_layouts_bf16_out(fmt, layout):
    b_layout, a_layout = layout
    got, want, _ = run_layout(fmt, "bf16", 513, 257, 1000, b_layout, a_layout, G.KERNEL_TC_PAIR, seed=5)
    assert_equal(got, want, f"{fmt} {layout}")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 128, 128), (16, 4096, 640), (33, 136, 200), (128, 1000, 2048)])
def test_fp8_small_m_kn_weight_exact(fmt, out, shape):
    """M <= 128 with a K x N fp8 weight: the small-M kernel (AUTO picks it)."""
    M, N, K = shape
    got, want, last = run_layout(fmt, out, M, N, K, "kn", "mk", G.KERNEL_AUTO, seed=7 * M + N)
    assert last == G.KERNEL_SKINNY
    assert_equal(got, want, f"{fmt} {shape}")


@pytest.mark.parametrize("fmt", ["e4m3", "tf32"])
def test_lowp_kn_last_wave(fmt):
    """4096 x 2560 K x N B: 160 pair tiles on 74-76 pairs.  A 16-bit B would
    split the last wave's tiles into N-halves; a K x N fp8 B runs whole tiles
    (a CTA's half of a half tile is narrower than one 128-byte box); a tf32 B,
    transposed to N x K first, takes the halves.  Exact either way."""
    got, want, _ = run_layout(fmt, "f32", 4096, 2560, 512, "kn", "mk", G.KERNEL_TC_PAIR, seed=17,
                              opts=((G.OPT_STREAM_K, 0),))
    assert_equal(got, want, fmt)


@pytest.mark.parametrize("fmt", ["e4m3", "tf32"])
def test_lowp_kn_stream_k_exact(fmt):
    got, want, _ = run_layout(fmt, "f32", 4096, 2560, 1536, "kn", "km", G.KERNEL_TC_PAIR, seed=19,
                              opts=((G.OPT_STREAM_K, 8),))
    assert_equal(got, want, fmt)


@pytest.mark.parametrize("fmt", ["e4m3", "tf32"])
@pytest.mark.parametrize("layout", [("kn", "mk"), ("nk", "km")])
def test_lowp_layouts_4096_whole_matrix_freivalds(fmt, layout):
    """4096 x 4096 x 2048: every output checked by two Freivalds products
    (exact integer arithmetic), eight rows checked element by element."""
    M = N = 4096
    K = 2048
    b_layout, a_layout = layout
    A = ints((M, K), 31, fmt)
    B = ints((N, K) if b_layout == "nk" else (K, N), 32, fmt)
    Ad = (A.t().contiguous() if a_layout == "km" else A).cuda()
    C = torch.empty(M, N, device="cuda")
    with G.Plan(0, b_layout, a_layout=a_layout) as p:
        p.run(Ad, B.cuda(), C)
        assert p.status() == 0
    Cc = C.cpu()
    rng = np.random.default_rng(33)
    for _ in range(2):
        r = rng.choice([-1, 1], size=N)
        assert oracle.freivalds_int(A, B, Cc, r, b_nk=b_layout == "nk") == 0
    rows = np.array([0, 1, 127, 128, 255, 256, 2047, 4095])
    ref = oracle.gemm_rows(A, B, rows, b_nk=b_layout == "nk")
    assert np.array_equal(Cc[torch.from_numpy(rows)].double().numpy(), ref)


def test_tf32_kn_float_within_tolerance():
    """Arbitrary fp32 inputs, K x N B and K x M A: within the tf32 bound
    (2^-9 + 2^-20 + K 2^-23) sum|a b| + 1e-6 of the float64 product."""
    M, N, K = 700, 520, 1024
    g = torch.Generator().manual_seed(41)
    A = torch.randn(M, K, generator=g)
    B = torch.randn(K, N, generator=g)
    C = torch.empty(M, N, device="cuda")
    with G.Plan(0, "kn", a_layout="km") as p:
        p.run(A.t().contiguous().cuda(), B.cuda(), C)
        assert p.status() == 0
    ref, S = oracle.gemm(A, B, with_mag=True)
    bound = (2.0 ** -9 + 2.0 ** -20 + K * 2.0 ** -23) * S + 1e-6
    assert np.all(np.abs(C.double().cpu().numpy() - ref) <= bound)


def test_fp8_kn_float_inputs_with_scales():
    M, N, K = 700, 520, 1024
    g = torch.Generator().manual_seed(43)
    a_scale, b_scale = 0.5, 0.125
    A = (torch.randn(M, K, generator=g) / a_scale).to(torch.float8_e4m3fn)
    B = (torch.randn(K, N, generator=g) / b_scale).to(torch.float8_e4m3fn)
    C = torch.empty(M, N, device="cuda")
    with G.Plan(0, "kn") as p:
        p.run(A.cuda(), B.cuda(), C, alpha=a_scale * b_scale)
        assert p.status() == 0
    C_ref, S = oracle.gemm_ex(A, B, alpha=a_scale * b_scale)
    ok, worst, _ = oracle.check_close(C.double().cpu().numpy(), C_ref, S)
    assert ok, f"worst err/bound {worst:.3f}"


@pytest.mark.parametrize("fmt", ["e4m3", "tf32"])
def test_lowp_kn_misaligned_pitch_is_packed(fmt):
    """A K x N B whose row pitch breaks the 16-byte rule is packed first."""
    M, N, K = 200, 136, 200
    A = ints((M, K), 51, fmt)
    B = ints((K, N), 52, fmt)
    es = 1 if fmt != "tf32" else 4
    extra = 5 if es == 1 else 1
    Bb = torch.zeros(K, N + extra, dtype=FMT[fmt])
    Bb[:, :N] = B
    Bd = Bb.cuda()[:, :N]
    assert (Bd.stride(0) * es) % 16 != 0
    C = torch.empty(M, N, device="cuda")
    with G.Plan(0, "kn") as p:
        p.run(A.cuda(), Bd, C)
        assert p.status() == 0 and p.workspace_bytes > 0
    assert np.array_equal(C.double().cpu().numpy(), oracle.gemm(A, B))


def test_tf32_mn_major_operands_use_the_workspace_even_without_packing():
    """Both operands transposed in one launch; aligned pitches, packing off."""
    M, N, K = 256, 512, 96
    A = ints((M, K), 61, "tf32")
    B = ints((K, N), 62, "tf32")
    C = torch.empty(M, N, device="cuda")
    with G.Plan(0, "kn", a_layout="km") as p:
        p.set_packing(False)
        p.run(A.t().contiguous().cuda(), B.cuda(), C)
        assert p.status() == 0
        assert p.workspace_bytes >= (M + N) * K * 4
    assert np.array_equal(C.double().cpu().numpy(), oracle.gemm(A, B))


def test_pointers_off_their_element_boundary_are_rejected():
    """A bf16 operand one byte off, an fp32 C two bytes off: GEMM_ERR_INVALID_ARG
    before anything runs."""
    import ctypes
    buf = torch.zeros(4 * 64 * 64 + 16, dtype=torch.uint8, device="cuda")
    ok = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(64, 64, device="cuda")
    L = G.lib()
    with G.Plan(0, "kn") as p:
        h = p._h
        stream = torch.cuda.current_stream().cuda_stream
        rc = L.gemm_run(h, 64, 64, 64, ctypes.c_void_p(buf.data_ptr() + 1), 64, ctypes.c_void_p(ok.data_ptr()), 64,
                        None, ctypes.c_void_p(C.data_ptr()), 64, G.EPI_NONE, G.BF16_F32OUT, ctypes.c_void_p(stream))
        assert rc == G.ERR_INVALID_ARG
        rc = L.gemm_run(h, 64, 64, 64, ctypes.c_void_p(ok.data_ptr()), 64, ctypes.c_void_p(ok.data_ptr()), 64,
                        None, ctypes.c_void_p(buf.data_ptr() + 2), 64, G.EPI_NONE, G.BF16_F32OUT,
                        ctypes.c_void_p(stream))
        assert rc == G.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(buf == 0)
