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
