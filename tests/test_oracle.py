"""Pins of the float64 oracle against what the pages and mathematics fix.

None of these compares the oracle with a retyped copy of itself: each check
is a printed value of the pages, a closed form, an invariant, a library
routine the definition reduces to on integers, or brute force on tiny inputs.
Chosen so that a dropped term, a wrong sign or index, or a transposed operand
fails at least one of them.
"""
import itertools
import json
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from dnn_linear_layers_gb300 import roofline
from dnn_linear_layers_gb300.inputs import int_bf16, normal_bf16

rng = np.random.default_rng(12345)


def rand_int(shape, lo=-4, hi=4):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float64)


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 9, 33), (64, 48, 130)])
def test_identity_and_permutation(M, N, K):
    A = rand_int((M, K)); B = rand_int((K, N))
    assert np.array_equal(oracle.gemm(A, np.eye(K)), A)
    assert np.array_equal(oracle.gemm(np.eye(M), A), A)
    assert np.array_equal(oracle.gemm(np.eye(K), B), B)
    # permutation matrices permute rows / columns exactly
    pr = rng.permutation(M); pc = rng.permutation(N)
    P = np.eye(M)[pr]; Q = np.eye(N)[:, pc]
    C = oracle.gemm(A, B)
    assert np.array_equal(oracle.gemm(P, C), C[pr])
    assert np.array_equal(oracle.gemm(C, Q), C[:, pc])


@pytest.mark.parametrize("M,N,K", [(5, 7, 3), (16, 3, 100), (2, 9, 257)])
def test_closed_form_rank_one_and_ramp(M, N, K):
    # A[i][k] = i+1, B[k][j] = j+1  =>  C[i][j] = K (i+1)(j+1)   (catches transposes, dropped k)
    A = np.repeat(np.arange(1, M + 1, dtype=np.float64)[:, None], K, axis=1)
    B = np.repeat(np.arange(1, N + 1, dtype=np.float64)[None, :], K, axis=0)
    C = oracle.gemm(A, B)
    assert np.array_equal(C, K * np.outer(np.arange(1, M + 1), np.arange(1, N + 1)))
    # A[i][k] = k, B[k][j] = (-1)^j  =>  C[i][j] = (-1)^j K(K-1)/2   (catches sign / k range)
    A2 = np.repeat(np.arange(K, dtype=np.float64)[None, :], M, axis=0)
    B2 = np.repeat(((-1.0) ** np.arange(N))[None, :], K, axis=0)
    C2 = oracle.gemm(A2, B2)
    assert np.array_equal(C2, np.repeat(((-1.0) ** np.arange(N))[None, :] * K * (K - 1) / 2, M, axis=0))
    # A[i][k] = k, B[k][j] = k  =>  sum k^2 = (K-1)K(2K-1)/6
    B3 = np.repeat(np.arange(K, dtype=np.float64)[:, None], N, axis=1)
    assert np.all(oracle.gemm(A2, B3) == (K - 1) * K * (2 * K - 1) / 6)


def test_matches_numpy_integer_matmul():
    """On integers the definition reduces to numpy's int64 matmul (a library routine)."""
    for (M, N, K) in [(1, 1, 1), (7, 5, 3), (33, 65, 129), (128, 130, 257)]:
        A = rng.integers(-4, 5, size=(M, K)); B = rng.integers(-4, 5, size=(K, N))
        C = oracle.gemm(A, B)
        assert np.array_equal(C, (A @ B).astype(np.float64))
        # the nk layout (W stored N x K) is the same product with B = W^T
        W = np.ascontiguousarray(B.T)
        assert np.array_equal(oracle.gemm(A, W, b_nk=True), C)


def test_brute_force_all_tiny_shapes():
    """Every shape up to 3x3x3 with entries in {-1, 0, 1}: exhaustive over A for
    fixed random B, and C compared with sums of explicit products built from
    itertools (each product enumerated once)."""
    for M, N, K in itertools.product((1, 2, 3), repeat=3):
        B = rng.integers(-2, 3, size=(K, N)).astype(np.float64)
        for trial in range(4):
            A = rng.integers(-2, 3, size=(M, K)).astype(np.float64)
            C = oracle.gemm(A, B)
            expect = np.zeros((M, N))
            for i, j, k in itertools.product(range(M), range(N), range(K)):
                expect[i, j] += A[i, k] * B[k, j]
            assert np.array_equal(C, expect)
            assert np.array_equal(oracle.gemm_py(A, B), expect)


def test_linearity_in_A_and_B():
    M, N, K = 19, 23, 41
    A1, A2 = rand_int((M, K)), rand_int((M, K))
    B1, B2 = rand_int((K, N)), rand_int((K, N))
    a, b = 3.0, -2.0
    assert np.array_equal(oracle.gemm(a * A1 + b * A2, B1), a * oracle.gemm(A1, B1) + b * oracle.gemm(A2, B1))
    assert np.array_equal(oracle.gemm(A1, a * B1 + b * B2), a * oracle.gemm(A1, B1) + b * oracle.gemm(A1, B2))


def test_transpose_identity():
    M, N, K = 13, 29, 37
    A = rand_int((M, K)); B = rand_int((K, N))
    C = oracle.gemm(A, B)
    assert np.array_equal(oracle.gemm(B.T, A.T), C.T)
    # nk layout with W = A: (B^T A^T) computed as B^T . W^T
    assert np.array_equal(oracle.gemm(np.ascontiguousarray(B.T), A, b_nk=True), C.T)


# ------------------------------------------------------------ pages' examples
def test_block_identity_8x8_from_pages(golden_dir):
    lines = [l.split("#")[0].strip() for l in (golden_dir / "block_identity_8x8.txt").read_text().splitlines()]
    lines = [l for l in lines if l]
    dims = {l.split()[0]: int(l.split()[1]) for l in lines if len(l.split()) == 2}
    T = dims["TILE"]
    A = rand_int((dims["M"], dims["K"])); B = rand_int((dims["K"], dims["N"]))
    C = oracle.gemm(A, B)

    def tile(X, name):
        r, c = int(name[1]), int(name[2])
        return X[r * T:(r + 1) * T, c * T:(c + 1) * T]

    n_checked = 0
    for l in lines:
        if "=" not in l:
            continue
        lhs, rhs = [s.strip() for s in l.split("=")]
        total = np.zeros((T, T))
        for term in rhs.split("+"):
            a_name, b_name = term.split()
            total = total + oracle.gemm(tile(A, a_name), tile(B, b_name))
        assert np.array_equal(tile(C, lhs), total), l
        n_checked += 1
    assert n_checked == 4


def _tiled_matmul_with_min_tails(A, B, tile):
    """The pages' tiled loop (i, j, k tiles clipped with min()), each tile product
    taken by the oracle on the sub-blocks."""
    M, K = A.shape; N = B.shape[1]
    C = np.zeros((M, N))
    for i in range(0, M, tile):
        ie = min(i + tile, M)
        for j in range(0, N, tile):
            je = min(j + tile, N)
            for k in range(0, K, tile):
                ke = min(k + tile, K)
                C[i:ie, j:je] += oracle.gemm(A[i:ie, k:ke], B[k:ke, j:je])
    return C


@pytest.mark.parametrize("M,N,K,tile", [(70, 33, 129, 64), (5, 64, 65, 4), (128, 128, 128, 64)])
def test_tiled_loop_with_ragged_tails_equals_definition(M, N, K, tile):
    A = rand_int((M, K)); B = rand_int((K, N))
    assert np.array_equal(_tiled_matmul_with_min_tails(A, B, tile), oracle.gemm(A, B))


# ------------------------------------------------------------- float bound
def test_float_result_within_rounding_bound_of_exact():
    """float64 oracle vs the exact rational result: |err| <= K * 2^-53 * sum|ab| (+ tiny)."""
    M, N, K = 4, 5, 300
    A = normal_bf16((M, K), 7).double().numpy(); B = normal_bf16((K, N), 8).double().numpy()
    C, S = oracle.gemm(A, B, with_mag=True)
    for i in range(M):
        for j in range(N):
            exact = sum((Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K)), Fraction(0))
            assert abs(Fraction(float(C[i, j])) - exact) <= Fraction(K * 2.0 ** -53) * Fraction(float(S[i, j])) * 2
            # S is the magnitude sum
    assert np.all(S >= np.abs(C) - 1e-12)


def test_magnitude_sum_closed_form():
    M, N, K = 3, 4, 10
    A = -np.ones((M, K)); B = np.ones((K, N)); B[::2] = -1
    C, S = oracle.gemm(A, B, with_mag=True)
    assert np.all(S == K)
    assert np.all(C == 0)   # five +1 and five -1 products


# ---------------------------------------------------------------- epilogue
def test_epilogue_special_cases():
    M, N, K = 9, 12, 31
    A = rand_int((M, K)); B = rand_int((K, N)); bias = rand_int((N,))
    C = oracle.gemm(A, B)
    assert np.array_equal(oracle.gemm(A, B, bias=np.zeros(N)), C)
    assert np.array_equal(oracle.gemm(A, B, bias=bias), C + bias[None, :])
    R = oracle.gemm(A, B, bias=bias, relu=True)
    assert np.all(R >= 0)
    pos = (C + bias) > 0
    assert np.array_equal(R[pos], (C + bias)[pos]) and np.all(R[~pos] == 0)
    assert np.array_equal(oracle.gemm(A, B, relu=True), np.maximum(C, 0))
    # K = 0: empty sum, output is the epilogue of 0
    Z = oracle.gemm(np.zeros((M, 0)), np.zeros((0, N)), bias=bias, relu=True)
    assert np.array_equal(Z, np.maximum(bias, 0)[None, :].repeat(M, 0))


def test_rows_and_cols_variants_agree_with_full():
    M, N, K = 40, 50, 77
    A = rand_int((M, K)); B = rand_int((K, N)); bias = rand_int((N,))
    C, S = oracle.gemm(A, B, bias=bias, relu=True, with_mag=True)
    rows = [0, 7, 39]; cols = [0, 31, 49]
    Cr, Sr = oracle.gemm_rows(A, B, rows, bias=bias, relu=True, with_mag=True)
    Cc, Sc = oracle.gemm_cols(A, B, cols, bias=bias, relu=True, with_mag=True)
    assert np.array_equal(Cr, C[rows]) and np.array_equal(Sr, S[rows])
    assert np.array_equal(Cc, C[:, cols]) and np.array_equal(Sc, S[:, cols])
    W = np.ascontiguousarray(B.T)
    assert np.array_equal(oracle.gemm_cols(A, W, cols, bias=bias, relu=True, b_nk=True), C[:, cols])
    assert np.array_equal(oracle.gemm_rows(A, W, rows, bias=bias, relu=True, b_nk=True), C[rows])


# -------------------------------------------------------------------- bf16
def test_bf16_round_matches_torch_on_fp32_values():
    """torch's fp32 -> bf16 cast is round-to-nearest-even: a library special case."""
    g = torch.Generator().manual_seed(3)
    x = torch.cat([torch.randn(20000, generator=g) * 10 ** torch.randint(-30, 30, (20000,), generator=g).float(),
                   torch.tensor([0.0, -0.0, 1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 - 2 ** -9, 3.0e38, 1e-40, -1e-42])])
    got = oracle.bf16_round(x.double().numpy())
    ref = x.to(torch.bfloat16).double().numpy()
    assert np.array_equal(got, ref)


def test_bf16_round_ties_and_ulp():
    assert oracle.bf16_round(np.array([1 + 2 ** -8]))[0] == 1.0            # tie -> even (down)
    assert oracle.bf16_round(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6  # tie -> even (up)
    assert oracle.bf16_round(np.array([257.0]))[0] == 256.0                 # integers above 256
    assert oracle.bf16_round(np.array([259.0]))[0] == 260.0
    assert oracle.ulp_bf16(np.array([1.0, 1.5, 256.0, 0.0]))[:3].tolist() == [2 ** -7, 2 ** -7, 2.0]
    assert oracle.ulp_bf16(np.array([0.0]))[0] == 2.0 ** -133


# --------------------------------------------------------------- Freivalds
def test_freivalds_detects_single_wrong_element():
    M, N, K = 64, 48, 96
    A = rand_int((M, K)); B = rand_int((K, N))
    C = oracle.gemm(A, B)
    r = rng.integers(-1, 2, size=N)
    r[r == 0] = 1
    assert oracle.freivalds_int(A, B, C, r) == 0
    bad = C.copy(); bad[5, 7] += 1
    assert oracle.freivalds_int(A, B, bad, r) == 1
    ok, worst = oracle.freivalds_float(A, B, C, r.astype(float))
    assert ok and worst < 1e-6
    bad2 = C.copy(); bad2[3, 3] += 500.0   # far above the propagated bound (~20 here)
    assert not oracle.freivalds_float(A, B, bad2, r.astype(float))[0]


def test_check_close_bound():
    C_ref = np.array([[1.0, 100.0]]); S = np.array([[1.0, 100.0]])
    assert oracle.check_close(C_ref + 1.0e-3 * S + 0.9e-6, C_ref, S)[0]
    assert not oracle.check_close(C_ref + 1.1e-3 * S + 1e-6, C_ref, S)[0]
    # one bf16 ulp allowed after a bf16 cast
    assert oracle.check_close(C_ref + 1e-3 * S + oracle.ulp_bf16(C_ref), C_ref, S, out_bf16=True)[0]


# ------------------------------------------------------------- convolution
def test_im2col_pins():
    # 1x1 "convolution" without padding is a reshape
    x = rand_int((2, 3, 4, 5))
    assert np.array_equal(oracle.im2col(x, 1, 1, 0), x.reshape(-1, 5))
    # all-ones input, 3x3, pad 1: row sums count the in-image neighbours x C
    ones = np.ones((1, 4, 5, 2))
    cnt = oracle.im2col(ones, 3, 3, 1).sum(1).reshape(4, 5)
    expect = np.full((4, 5), 9.0); expect[[0, -1], :] = 6; expect[:, [0, -1]] = 6
    expect[0, 0] = expect[0, -1] = expect[-1, 0] = expect[-1, -1] = 4
    assert np.array_equal(cnt, expect * 2)
    # centre tap of a 3x3 window is the pixel itself: column (1*3+1)*C + c
    x2 = rand_int((1, 4, 4, 3))
    M = oracle.im2col(x2, 3, 3, 1)
    assert np.array_equal(M[:, 4 * 3:5 * 3], x2.reshape(-1, 3))
    # rows variant
    assert np.array_equal(oracle.im2col_rows(x2, 3, 3, 1, [0, 5, 15]), M[[0, 5, 15]])


def test_conv_direct_equals_im2col_gemm_and_pins():
    x = rand_int((2, 6, 5, 4)); w = rand_int((3, 3, 3, 4))
    cols = oracle.im2col(x, 3, 3, 1)
    Y = oracle.gemm(cols, w.reshape(3, -1), b_nk=True)   # weights as W (Cout x RSC)
    pos = [(n, oh, ow) for n in range(2) for oh in range(6) for ow in range(5)]
    direct = oracle.conv2d_at(x, w, 1, pos)
    assert np.array_equal(direct, Y)
    # delta filter at the centre reproduces the input channel
    wd = np.zeros((4, 3, 3, 4)); wd[np.arange(4), 1, 1, np.arange(4)] = 1
    assert np.array_equal(oracle.conv2d_at(x, wd, 1, pos), x.reshape(-1, 4))
    # delta at (r, s) = (0, 0) shifts by (-1, -1) with zero fill
    ws = np.zeros((4, 3, 3, 4)); ws[np.arange(4), 0, 0, np.arange(4)] = 1
    out = oracle.conv2d_at(x, ws, 1, pos).reshape(2, 6, 5, 4)
    assert np.all(out[:, 0] == 0) and np.all(out[:, :, 0] == 0)
    assert np.array_equal(out[:, 1:, 1:], x[:, :-1, :-1])


# ------------------------------------------------------- printed numbers
def test_printed_numbers(golden_dir):
    g = json.loads((golden_dir / "printed_numbers.json").read_text())
    for c in g["matmul_intensity"]:
        _, _, ai = roofline.matmul_intensity(c["M"], c["K"], c["N"], c["dtype_bytes"])
        if "printed_rel_tol" in c:
            assert abs(ai - c["printed_ai"]) <= c["printed_rel_tol"] * c["printed_ai"]
        else:
            assert abs(ai - c["printed_ai"]) <= c["printed_abs_tol"]
    n = g["naive_ops_4096"]
    assert abs(n["n"] ** 3 - n["printed_macs"]) <= n["printed_rel_tol"] * n["printed_macs"]
    o = g["block_oi_fp32"]
    for b, v in zip(o["b"], o["printed"]):
        assert abs(roofline.block_oi(b) - v) <= o["abs_tol"]
    w = g["wave_quantisation"]
    for size, tiles in w["cases"]:
        assert roofline.tile_count(size, size, w["tile_m"], w["tile_n"]) == tiles
    c = g["im2col_cost"]
    OH = c["H"] + 2 * c["pad"] - c["R"] + 1; OW = c["W"] + 2 * c["pad"] - c["S"] + 1
    rows = c["Nb"] * OH * OW; kdim = c["R"] * c["S"] * c["C"]
    # the oracle's im2col of a small image with the same R, S, C has this column count
    assert oracle.im2col(np.zeros((1, 3, 3, c["C"])), c["R"], c["S"], c["pad"]).shape[1] == kdim
    assert abs(roofline.gemm_flops(rows, c["K"], kdim) / 1e9 - c["printed_gflop"]) <= c["printed_rel_tol"] * c["printed_gflop"]
    assert abs(rows * kdim * 4 / 1e6 - c["printed_matrix_mb"]) <= c["printed_rel_tol"] * c["printed_matrix_mb"]
    f = g["conv_fused_work"]
    fma = f["Nb"] * f["H"] * f["W"] * f["K"] * f["R"] * f["S"] * f["C"]
    assert abs(fma - f["printed_fma"]) <= f["printed_rel_tol"] * f["printed_fma"]
    assert abs(2 * fma / 1e9 - f["printed_gflop"]) <= f["printed_rel_tol"] * f["printed_gflop"]


def test_input_generators_are_seeded_and_exact():
    a = normal_bf16((4, 5), 1); b = normal_bf16((4, 5), 1)
    assert torch.equal(a, b) and a.dtype == torch.bfloat16
    i = int_bf16((100,), 2)
    assert i.float().abs().max() <= 4 and torch.equal(i.float(), i.float().round())


def test_extended_epilogue_exact_against_integer_closed_form():
    # integers and powers of two: every value below is exact in float64, so the
    # oracle must equal an independent int64 computation of the same formula
    rng = np.random.default_rng(41)
    M, N, K = 9, 13, 17
    A = rng.integers(-4, 5, size=(M, K)); B = rng.integers(-4, 5, size=(K, N))
    C0 = rng.integers(-50, 51, size=(M, N))
    e = rng.integers(0, 4, size=N)                 # scale = 2^e
    bias = rng.integers(-20, 21, size=N)
    P = A.astype(np.int64) @ B.astype(np.int64)
    want = 2 * P * (1 << e)[None, :] + bias[None, :] - 3 * C0     # alpha 2, beta -3
    got, S = oracle.gemm_ex(A, B, alpha=2.0, beta=-3.0, C0=C0, scale=(2.0 ** e), bias=bias)
    assert np.array_equal(got, want.astype(np.float64))
    # the magnitude sum scales with |alpha * scale|
    S_plain = np.abs(A)[:, :, None] * np.abs(B)[None, :, :]
    assert np.array_equal(S, 2.0 * (2.0 ** e)[None, :] * S_plain.sum(axis=1))
    # N x K weight layout gives the same result
    got_nk, _ = oracle.gemm_ex(A, B.T.copy(), alpha=2.0, beta=-3.0, C0=C0, scale=(2.0 ** e), bias=bias, b_nk=True)
    assert np.array_equal(got_nk, got)


def test_extended_epilogue_order_and_special_cases():
    A = np.array([[1.0, 2.0]]); B = np.array([[1.0], [1.0]])          # A.B = 3
    C0 = np.array([[10.0]])
    # relu comes last: 3 * 1 + (-5) + 1 * 10 = 8 > 0 although 3 - 5 < 0
    c, _ = oracle.gemm_ex(A, B, beta=1.0, C0=C0, bias=[-5.0], relu=True)
    assert c[0, 0] == 8.0
    # scale multiplies the product, not the bias: 3 * 4 + 1 = 13
    c, _ = oracle.gemm_ex(A, B, scale=[4.0], bias=[1.0])
    assert c[0, 0] == 13.0
    # beta only (zero product): beta * C0 + bias
    c, _ = oracle.gemm_ex(np.zeros((1, 2)), B, beta=0.5, C0=C0, bias=[1.0])
    assert c[0, 0] == 6.0
    # defaults reduce to the plain product with bias and ReLU
    rng = np.random.default_rng(3)
    A2 = rng.standard_normal((5, 7)); B2 = rng.standard_normal((7, 4)); b = rng.standard_normal(4)
    c1, _ = oracle.gemm_ex(A2, B2, bias=b, relu=True)
    assert np.array_equal(c1, oracle.gemm(A2, B2, bias=b, relu=True))


def test_fp8_decoders_pinned():
    # values fixed by the formats
    e4 = oracle.e4m3_to_f64
    assert e4([0x38])[0] == 1.0 and e4([0xB8])[0] == -1.0
    assert e4([0x7E])[0] == 448.0                      # largest finite: 1.75 * 2^8
    assert e4([0x01])[0] == 2.0 ** -9                  # smallest subnormal: 1/8 * 2^-6
    assert e4([0x08])[0] == 2.0 ** -6                  # smallest normal
    assert np.isnan(e4([0x7F])[0]) and np.isnan(e4([0xFF])[0])
    assert e4([0x00])[0] == 0.0 and np.signbit(e4([0x80])[0])
    e5 = oracle.e5m2_to_f64
    assert e5([0x3C])[0] == 1.0 and e5([0x7B])[0] == 57344.0
    assert e5([0x01])[0] == 2.0 ** -16 and e5([0x04])[0] == 2.0 ** -14
    assert e5([0x7C])[0] == np.inf and e5([0xFC])[0] == -np.inf and np.isnan(e5([0x7D])[0])
    # every code against torch's own float8 conversion (an independent implementation)
    codes = torch.arange(256, dtype=torch.uint8)
    for dt, dec in ((torch.float8_e4m3fn, e4), (torch.float8_e5m2, e5)):
        ref = codes.view(dt).to(torch.float64).numpy()
        got = dec(codes.numpy())
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], ref[~nan])


def test_fp8_small_integers_exact_and_gemm_on_decoded_values():
    # integers -4..4 are exact in both formats, so an fp8 GEMM of them is the
    # integer GEMM (numpy int64)
    rng = np.random.default_rng(8)
    A = rng.integers(-4, 5, size=(6, 40)); B = rng.integers(-4, 5, size=(9, 40))
    for dt in (torch.float8_e4m3fn, torch.float8_e5m2):
        At = torch.from_numpy(A).to(dt); Bt = torch.from_numpy(B).to(dt)
        assert np.array_equal(oracle._f64(At), A)
        C = oracle.gemm(At, Bt, b_nk=True)
        assert np.array_equal(C, (A @ B.T).astype(np.float64))


def test_conv_maxpool_closed_forms():
    # 1 x 1 identity filter: the convolution is x itself, so the fused result is
    # the 2 x 2 block maximum of x (numpy reshape / max), and with ReLU of it
    rng = np.random.default_rng(21)
    Nb, H, W, C = 2, 6, 8, 5
    x = rng.integers(-9, 10, size=(Nb, H, W, C)).astype(np.float64)
    w = np.eye(C).reshape(C, 1, 1, C)
    pos = [(n, ph, pw) for n in range(Nb) for ph in range(H // 2) for pw in range(W // 2)]
    got = oracle.conv2d_maxpool_at(x, w, 0, pos)
    want = x.reshape(Nb, H // 2, 2, W // 2, 2, C).max(axis=(2, 4)).reshape(-1, C)
    assert np.array_equal(got, want)
    got_relu = oracle.conv2d_maxpool_at(x, w, 0, pos, relu=True)
    assert np.array_equal(got_relu, np.maximum(want, 0.0))
    # a negative per-channel scale flips which element wins (max of -x is -min x)
    s = -np.ones(C)
    got_neg = oracle.conv2d_maxpool_at(x, w, 0, pos, scale=s)
    assert np.array_equal(got_neg, -x.reshape(Nb, H // 2, 2, W // 2, 2, C).min(axis=(2, 4)).reshape(-1, C))


def test_attention_closed_forms():
    rng = np.random.default_rng(31)
    Sq, Sk, D = 5, 7, 4
    Q = rng.standard_normal((Sq, D)); V = rng.standard_normal((Sk, D))
    # all scores equal: O is the mean of the visible value rows
    O = oracle.attention(Q, np.zeros((Sk, D)), V)
    assert np.allclose(O, np.broadcast_to(V.mean(axis=0), (Sq, D)), rtol=0, atol=1e-15)
    Oc = oracle.attention(Q, np.zeros((Sk, D)), V, causal=True)      # query i sees keys 0 .. i + 2
    for i in range(Sq):
        assert np.allclose(Oc[i], V[: i + Sk - Sq + 1].mean(axis=0), rtol=0, atol=1e-15)
    # two keys with scores 0 and ln 3: weights 1/4 and 3/4
    O2 = oracle.attention(np.array([[1.0]]), np.array([[0.0], [np.log(3.0)]]), np.array([[4.0], [8.0]]), scale=1.0)
    assert abs(O2[0, 0] - 7.0) < 1e-14
    # shifting every key by one vector shifts each query's scores by a constant
    K = rng.standard_normal((Sk, D))
    assert np.allclose(oracle.attention(Q, K + rng.standard_normal(D), V), oracle.attention(Q, K, V), atol=1e-12)
    # the default scale is 1 / sqrt(D): D = 4, q.k1 = 2 ln 3 gives the score ln 3, weights 1/4 and 3/4
    q = np.array([[2.0 * np.log(3.0), 0.0, 0.0, 0.0]])
    k = np.array([[0.0, 0.0, 0.0, 0.0], [1.0, 0.0, 0.0, 0.0]])
    assert abs(oracle.attention(q, k, np.array([[4.0], [8.0]]))[0, 0] - 7.0) < 1e-14
    # a query that sees no key gets zeros (causal, more queries than keys)
    Oz = oracle.attention(rng.standard_normal((6, D)), K[:3], V[:3], causal=True)
    assert np.array_equal(Oz[:3], np.zeros((3, D))) and np.all(Oz[3:] != 0)


def test_attention_matches_the_tiled_online_softmax_recurrence():
    """The oracle materialises the softmax; the FlashAttention recurrence of the
    pages (keys in tiles, a running row max m, a running sum l and the
    accumulator rescaled by e^(m_old - m_new) whenever m grows) reaches the same
    result without it.  Written out here with tiles of three keys, it must agree
    with the oracle to rounding, with and without the causal mask."""
    rng = np.random.default_rng(61)
    for Sq, Sk, D, causal in [(5, 7, 4, False), (6, 9, 3, True), (4, 4, 2, True), (8, 3, 5, True)]:
        Q = rng.standard_normal((Sq, D)); K = rng.standard_normal((Sk, D)); V = rng.standard_normal((Sk, D))
        s = 1.0 / np.sqrt(D)
        out = np.zeros((Sq, D))
        for i in range(Sq):
            m, l, acc = -np.inf, 0.0, np.zeros(D)
            for t0 in range(0, Sk, 3):
                keys = [j for j in range(t0, min(t0 + 3, Sk)) if not causal or j <= i + (Sk - Sq)]
                if not keys:
                    continue
                sc = np.array([s * float(Q[i] @ K[j]) for j in keys])
                m_new = max(m, float(sc.max()))
                f = np.exp(m - m_new) if np.isfinite(m) else 0.0
                p = np.exp(sc - m_new)
                l = l * f + float(p.sum())
                acc = acc * f + p @ V[keys]
                m = m_new
            out[i] = acc / l if l > 0 else 0.0
        assert np.allclose(oracle.attention(Q, K, V, causal=causal), out, rtol=0, atol=1e-13)

