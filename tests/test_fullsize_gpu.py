"""Parity at the full workload sizes, in the launch configuration the benchmark
uses (automatic kernel choice), on outputs the oracle can compute one by one:

* whole sampled rows and columns (every tile boundary +-1, first, last and
  seeded random ones) against the float64 triple loop;
* Freivalds' check C r == A (B r) over the whole matrix: exact in int64 for
  integer inputs, against the propagated tolerance bound for float inputs.

The decode-like Linear layers (M <= 128) are small enough for the oracle to
compute every output.
"""
import numpy as np
import pytest
import torch

import oracle
from dnn_linear_layers_gb300 import gemm as G
from dnn_linear_layers_gb300.inputs import GemmCase, skinny_cases, transformer_cases, odd_cases

from parity import compare, out_dtype_of, sample_rows_cols

pytestmark = pytest.mark.gpu


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


def run_full(plans, case):
    p = plans["nk" if case.b_nk else "kn"]
    p.set_kernel(G.KERNEL_AUTO)
    A, B, bias = case.tensors()
    C = torch.empty((case.M, case.N), dtype=out_dtype_of(case), device="cuda")
    p.run(A.cuda(), B.cuda(), C, bias.cuda() if bias is not None else None, case.relu)
    assert p.status() == 0
    return A, B, bias, C.cpu()


def check_sampled(case, A, B, bias, C, n_random=24):
    rows, cols = sample_rows_cols(case.M, case.N, n_random=n_random, seed=case.seed)
    Cr, Sr = oracle.gemm_rows(A, B, rows, bias=bias, relu=case.relu, b_nk=case.b_nk, with_mag=True)
    compare(case, C[rows], Cr, Sr)
    Cc, Sc = oracle.gemm_cols(A, B, cols, bias=bias, relu=case.relu, b_nk=case.b_nk, with_mag=True)
    compare(case, C[:, cols], Cc, Sc)


def freivalds(case, A, B, bias, C, trials=2):
    rng = np.random.default_rng(case.seed + 99)
    for _ in range(trials):
        r = rng.choice([-1, 1], size=case.N)
        if case.integer:
            assert not case.relu
            bad = oracle.freivalds_int(A, B, C, r, b_nk=case.b_nk, bias=bias)
            assert bad == 0, f"{case.name}: {bad} rows fail Freivalds"
        elif not case.relu:
            ok, worst = oracle.freivalds_float(A, B, C, r.astype(float), b_nk=case.b_nk, bias=bias,
                                               out_bf16=case.out != "f32")
            assert ok, f"{case.name}: Freivalds ratio {worst:.3f}"


def test_square_8192_bf16(plans):
    case = GemmCase("square8192", 8192, 8192, 8192, out="bf16", seed=0)
    A, B, bias, C = run_full(plans, case)
    check_sampled(case, A, B, bias, C)
    freivalds(case, A, B, bias, C)


@pytest.mark.parametrize("n", [4096, 8192])
def test_square_nk_weight_layout(plans, n):
    """n^3 with B stored N x K (the Linear weight layout), as benchmarked:
    sampled tile-boundary rows and columns against the oracle, Freivalds on
    the whole matrix."""
    case = GemmCase(f"square{n}_nk", n, n, n, b_nk=True, out="bf16", seed=n + 7)
    A, B, bias, C = run_full(plans, case)
    check_sampled(case, A, B, bias, C, n_random=8)
    freivalds(case, A, B, bias, C, trials=1)


def test_square_8192_integer_exact_whole_matrix(plans):
    case = GemmCase("square8192_int", 8192, 8192, 8192, out="f32", integer=True, seed=1)
    A, B, bias, C = run_full(plans, case)
    freivalds(case, A, B, bias, C, trials=3)
    check_sampled(case, A, B, bias, C, n_random=8)


@pytest.mark.parametrize("n", [1024, 2048, 4096])
def test_square_sweep_integer_exact(plans, n):
    case = GemmCase(f"square{n}_int", n, n, n, out="bf16", integer=True, seed=n)
    A, B, bias, C = run_full(plans, case)
    check_sampled(case, A, B, bias, C, n_random=8)
    case32 = GemmCase(f"square{n}_int32", n, n, n, out="f32", integer=True, seed=n)
    A, B, bias, C = run_full(plans, case32)
    freivalds(case32, A, B, bias, C)


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_transformer_layers(plans, idx):
    case = transformer_cases()[idx]
    A, B, bias, C = run_full(plans, case)
    check_sampled(case, A, B, bias, C, n_random=16)
    freivalds(case, A, B, bias, C, trials=1)


@pytest.mark.parametrize("idx", range(6))
def test_decode_linear_layers_every_output(plans, idx):
    case = skinny_cases()[idx]
    A, B, bias, C = run_full(plans, case)
    C_ref, S = oracle.gemm(A, B, bias=bias, relu=case.relu, b_nk=True, with_mag=True)
    compare(case, C, C_ref, S)


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_odd_shapes(plans, idx):
    case = odd_cases()[idx]
    A, B, bias, C = run_full(plans, case)
    check_sampled(case, A, B, bias, C, n_random=16)
    freivalds(case, A, B, bias, C, trials=1)


@pytest.mark.parametrize("causal", [False, True])
def test_attention_full_size_sampled_heads(plans, causal):
    """The benchmark's attention workload (B 4, H 32, S 4096, D 128, bf16 in and
    out, seeded N(0, 1) inputs) in its launch configuration; eight seeded heads
    are checked against the float64 oracle, every output of each, with the
    bound of the attention parity tests (2 u max_j |V_jd| + 1e-5 plus one bf16
    ulp of the output, u = 2^-9)."""
    from dnn_linear_layers_gb300.inputs import normal_bf16
    B, H, S, D = 4, 32, 4096, 128
    q = normal_bf16((B, H, S, D), 0)
    k = normal_bf16((B, H, S, D), 1)
    v = normal_bf16((B, H, S, D), 2)
    o = torch.empty(B, H, S, D, dtype=torch.bfloat16, device="cuda")
    p = plans["nk"]
    p.attention(q.cuda(), k.cuda(), v.cuda(), o, causal=causal)
    assert p.status() == 0
    got = o.view(B * H, S, D).double().cpu().numpy()
    qf, kf, vf = (t.view(B * H, S, D) for t in (q, k, v))
    heads = np.random.default_rng(5 + causal).choice(B * H, size=8, replace=False)
    for hd in heads:
        ref = oracle.attention(qf[hd], kf[hd], vf[hd], causal=causal)
        vmax = np.abs(oracle._f64(vf[hd])).max(axis=0, keepdims=True)
        bound = 2 * 2.0 ** -9 * vmax + 1e-5 + oracle.ulp_bf16(ref)
        err = np.abs(got[hd] - ref)
        assert np.all(err <= bound), f"head {hd}: worst err/bound {(err / bound).max():.3f}"


# ---- benchmarked variants: the bench's own inputs at the bench's sizes ----

@pytest.mark.parametrize("n", [1024, 2048, 4096])
def test_square_sweep_float_sampled(plans, n):
    """The float square sweep as benchmarked (N(0,1) bf16, bf16 out)."""
    case = GemmCase(f"square{n}", n, n, n, out="bf16", seed=n + 1)
    A, B, bias, C = run_full(plans, case)
    check_sampled(case, A, B, bias, C, n_random=8)
    freivalds(case, A, B, bias, C, trials=1)


@pytest.mark.parametrize("M", [4])
@pytest.mark.parametrize("nk", [(14336, 4096), (4096, 4096)])
def test_decode_linear_layers_m4_every_output(plans, M, nk):
    N, K = nk
    case = GemmCase(f"linear_m{M}_{K}x{N}", M, N, K, b_nk=True, bias=True, b_std=K ** -0.5, seed=3)
    A, B, bias, C = run_full(plans, case)
    C_ref, S = oracle.gemm(A, B, bias=bias, relu=False, b_nk=True, with_mag=True)
    compare(case, C, C_ref, S)


FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def _fp8_run(A, B, bias, out=torch.bfloat16, relu=False):
    C = torch.empty(A.shape[0], B.shape[0], dtype=out, device="cuda")
    with G.Plan(0, "nk", b_const=True) as p:
        p.run(A.cuda(), B.cuda(), C, bias.cuda() if bias is not None else None, relu)
        assert p.status() == 0
    return C.cpu()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("M", [1, 4, 16, 128])
def test_decode_fp8_layers_every_output(fmt, M):
    """fp8 weights and activations at 4096 -> 14336 (the benchmark's inputs:
    N(0,1) drawn as bf16, then rounded to the format; bf16 bias N(0, 0.02^2)),
    every output within the tolerance; the oracle decodes the same codes."""
    from dnn_linear_layers_gb300.inputs import normal_bf16
    N, K = 14336, 4096
    A = normal_bf16((M, K), 0).to(FP8[fmt])
    B = normal_bf16((N, K), 1).to(FP8[fmt])
    bias = normal_bf16((N,), 2, 0.02)
    C = _fp8_run(A, B, bias)
    C_ref, S = oracle.gemm(A, B, bias=bias, b_nk=True, with_mag=True)
    ok, worst, _ = oracle.check_close(C.double().numpy(), C_ref, S, out_bf16=True)
    assert ok, f"worst err/bound {worst:.3f}"


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("M", [1, 16, 128])
def test_decode_fp8_layers_integer_exact(fmt, M):
    N, K = 14336, 4096
    g = torch.Generator().manual_seed(M)
    A = torch.randint(-4, 5, (M, K), generator=g).to(FP8[fmt])
    B = torch.randint(-4, 5, (N, K), generator=g).to(FP8[fmt])
    bias = torch.randint(-8, 9, (N,), generator=g).to(torch.bfloat16)
    C = _fp8_run(A, B, bias, out=torch.float32, relu=True)
    assert np.array_equal(C.double().numpy(), oracle.gemm(A, B, bias=bias, relu=True, b_nk=True))


def _int_operands(shape_a, shape_b, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    return (torch.randint(-4, 5, shape_a, generator=g).to(dtype), torch.randint(-4, 5, shape_b, generator=g).to(dtype))


def _sampled_exact(A, B, C, b_nk, n):
    rows, cols = sample_rows_cols(n, n, n_random=6, seed=n)
    assert np.array_equal(C[rows].double().numpy(), oracle.gemm_rows(A, B, rows, b_nk=b_nk))
    assert np.array_equal(C[:, cols].double().numpy(), oracle.gemm_cols(A, B, cols, b_nk=b_nk))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_square_8192_fp8(fmt):
    """8192^3 with fp8 operands (bf16 out) as benchmarked: integer inputs
    exact over the whole matrix (Freivalds in int64) and on sampled rows and
    columns; the bench's N(0,1) inputs within the tolerance on sampled rows."""
    from dnn_linear_layers_gb300.inputs import normal_bf16
    n = 8192
    A, B = _int_operands((n, n), (n, n), 21, FP8[fmt])
    C = _fp8_run(A, B, None, out=torch.float32)
    rng = np.random.default_rng(22)
    for _ in range(2):
        assert oracle.freivalds_int(A, B, C, rng.choice([-1, 1], size=n), b_nk=True) == 0
    _sampled_exact(A, B, C, True, n)
    A = normal_bf16((n, n), 0).to(FP8[fmt])
    B = normal_bf16((n, n), 1).to(FP8[fmt])
    C = _fp8_run(A, B, None)
    rows, _ = sample_rows_cols(n, n, n_random=8, seed=23)
    Cr, Sr = oracle.gemm_rows(A, B, rows, b_nk=True, with_mag=True)
    ok, worst, _ = oracle.check_close(C[rows].double().numpy(), Cr, Sr, out_bf16=True)
    assert ok, f"worst err/bound {worst:.3f}"


def test_square_8192_tf32():
    """8192^3 with fp32 operands multiplied as tf32 (bf16 out) as benchmarked:
    integer inputs exact (Freivalds and sampled rows / columns); N(0,1) fp32
    inputs on sampled rows within (2^-9 + 2^-20 + K 2^-23) S + 1e-6 plus one
    bf16 ulp (the tf32 bound, derived in tests/test_tf32_gpu.py)."""
    from dnn_linear_layers_gb300.inputs import normal_bf16
    n = 8192
    A, B = _int_operands((n, n), (n, n), 31, torch.float32)
    C = _fp8_run(A, B, None, out=torch.float32)
    rng = np.random.default_rng(32)
    for _ in range(2):
        assert oracle.freivalds_int(A, B, C, rng.choice([-1, 1], size=n), b_nk=True) == 0
    _sampled_exact(A, B, C, True, n)
    A = normal_bf16((n, n), 0, dtype=torch.float32)
    B = normal_bf16((n, n), 1, dtype=torch.float32)
    C = _fp8_run(A, B, None)
    rows, _ = sample_rows_cols(n, n, n_random=8, seed=33)
    Cr, Sr = oracle.gemm_rows(A, B, rows, b_nk=True, with_mag=True)
    bound = (2.0 ** -9 + 2.0 ** -20 + n * 2.0 ** -23) * Sr + 1e-6 + oracle.ulp_bf16(Cr)
    err = np.abs(C[rows].double().numpy() - Cr)
    assert np.all(err <= bound), f"worst err/bound {(err / bound).max():.3f}"


def test_square_8192_transposed_a():
    """8192^3 with A stored K x M (plan flag GEMM_A_KM), B K x N, bf16 out, as
    benchmarked: integer inputs exact over the whole matrix; the bench's N(0,1)
    inputs within the tolerance on sampled rows and columns."""
    from dnn_linear_layers_gb300.inputs import normal_bf16
    n = 8192
    for integer in (True, False):
        if integer:
            At, B = _int_operands((n, n), (n, n), 41, torch.bfloat16)
            od = torch.float32
        else:
            At, B = normal_bf16((n, n), 0), normal_bf16((n, n), 1)
            od = torch.bfloat16
        C = torch.empty(n, n, dtype=od, device="cuda")
        with G.Plan(0, "kn", a_layout="km") as p:
            p.run(At.cuda(), B.cuda(), C)
            assert p.status() == 0 and p.last_kernel == G.KERNEL_TC_PAIR
        C = C.cpu()
        A = At.t().contiguous()                 # the M x K operand the oracle reads
        if integer:
            rng = np.random.default_rng(42)
            assert oracle.freivalds_int(A, B, C, rng.choice([-1, 1], size=n)) == 0
            _sampled_exact(A, B, C, False, n)
        else:
            case = GemmCase("transa8192", n, n, n, out="bf16", seed=43)
            check_sampled(case, A, B, None, C, n_random=8)


def test_pooled_conv_full_size_every_output():
    """Convolution + bias + ReLU + 2 x 2 max-pool at 32 x 56 x 56 x 256 -> 256
    (the benchmark's configuration): integer inputs, every pooled output exact
    against the oracle's direct convolution; then the bench's inputs (ReLU(N(0,1))
    activations, N(0, 2/2304) weights, N(0, 0.02^2) bias) on sampled pooled
    positions within the tolerance."""
    from dnn_linear_layers_gb300.inputs import conv_tensors, int_bf16, normal_bf16
    Nb, H, W, C, Cout = 32, 56, 56, 256, 256
    PH, PW = H // 2, W // 2
    x = int_bf16((Nb, H, W, C), 71, lo=-2, hi=2)
    w = int_bf16((Cout, 3, 3, C), 72, lo=-2, hi=2)
    b = int_bf16((Cout,), 73, lo=-8, hi=8)
    y = torch.full((Nb * PH * PW, Cout), float("nan"), dtype=torch.float32, device="cuda")
    with G.Plan(0, "nk") as p:
        p.conv2d_maxpool(x.cuda(), w.cuda(), y, bias=b.cuda(), relu=True, pad=1)
        assert p.status() == 0 and p.last_kernel == G.KERNEL_TC_PAIR
    pos = [(n, ph, pw) for n in range(Nb) for ph in range(PH) for pw in range(PW)]
    ref = oracle.conv2d_maxpool_at(x, w, 1, pos, bias=b, relu=True)
    got = y.double().cpu().numpy()
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[0]}"
    x, w = conv_tensors()
    b = normal_bf16((Cout,), 2, 0.02)
    y = torch.empty(Nb * PH * PW, Cout, dtype=torch.bfloat16, device="cuda")
    with G.Plan(0, "nk") as p:
        p.conv2d_maxpool(x.cuda(), w.cuda(), y, bias=b.cuda(), relu=True, pad=1)
        assert p.status() == 0
    rng = np.random.default_rng(74)
    sel = sorted({(0, 0, 0), (Nb - 1, PH - 1, PW - 1)} |
                 {(int(rng.integers(Nb)), int(rng.integers(PH)), int(rng.integers(PW))) for _ in range(62)})
    ref = oracle.conv2d_maxpool_at(x, w, 1, sel, bias=b, relu=True)
    # the max of values each within its bound lies within the largest bound
    S = np.zeros_like(ref)
    xa, wa = x.double().abs(), w.double().abs()
    for dy in (0, 1):
        for dx in (0, 1):
            S = np.maximum(S, oracle.conv2d_at(xa, wa, 1, [(n, 2 * ph + dy, 2 * pw + dx) for n, ph, pw in sel]))
    rows = np.array([(n * PH + ph) * PW + pw for n, ph, pw in sel])
    ok, worst, _ = oracle.check_close(y[torch.from_numpy(rows).cuda()].double().cpu().numpy(), ref, S,
                                      out_bf16=True)
    assert ok, f"worst err/bound {worst:.3f}"


@pytest.mark.parametrize("causal", [False, True])
def test_attention_d64_full_size_sampled_heads(plans, causal):
    """The D = 64 attention workload (B 4, H 32, S 4096) on eight seeded heads,
    every output, with the attention bound (2 u max_j |V_jd| + 1e-5 plus one
    bf16 ulp, u = 2^-9)."""
    from dnn_linear_layers_gb300.inputs import normal_bf16
    B, H, S, D = 4, 32, 4096, 64
    q = normal_bf16((B, H, S, D), 0)
    k = normal_bf16((B, H, S, D), 1)
    v = normal_bf16((B, H, S, D), 2)
    o = torch.empty(B, H, S, D, dtype=torch.bfloat16, device="cuda")
    p = plans["nk"]
    p.attention(q.cuda(), k.cuda(), v.cuda(), o, causal=causal)
    assert p.status() == 0
    got = o.view(B * H, S, D).double().cpu().numpy()
    qf, kf, vf = (t.view(B * H, S, D) for t in (q, k, v))
    heads = np.random.default_rng(15 + causal).choice(B * H, size=8, replace=False)
    for hd in heads:
        ref = oracle.attention(qf[hd], kf[hd], vf[hd], causal=causal)
        vmax = np.abs(oracle._f64(vf[hd])).max(axis=0, keepdims=True)
        bound = 2 * 2.0 ** -9 * vmax + 1e-5 + oracle.ulp_bf16(ref)
        err = np.abs(got[hd] - ref)
        assert np.all(err <= bound), f"head {hd}: worst err/bound {(err / bound).max():.3f}"
