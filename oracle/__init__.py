"""Float64 CPU oracle for the dense GEMM / Linear layer.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library (``dnn_linear_layers_gb300``) and neither imports the other.

Definitions followed (page titles and sections of the source pages):

* GEMM: ``C[i][j] = sum_k A[i][k] * B[k][j]`` -- youngju.dev "GEMM to
  FlashAttention", the ``naive_matmul`` listing (float64 accumulator).
* Linear layer ``output = W x input + b`` -- same page, header formula; with M
  tokens stored as rows this is ``Y = X W^T + b`` (W is out x in).
* ReLU ``max(0, x)`` after the bias -- CMU 15-418 "DNNs and ML accelerators"
  notes, section 2.1 (neuron ``f(sum x_i w_i + b)``).
* bf16 = 1 sign + 8 exponent + 7 mantissa bits, same exponent range as fp32 --
  same notes, section 2.7; rounding to nearest, ties to even (IEEE 754).
* im2col: each R x S x C neighbourhood flattened into one row -- same notes,
  section 2.3; direct convolution as the seven-loop nest, section 2.2.

The heavy loops are plain C (``oracle_gemm.c``) compiled with
``-ffp-contract=off`` and OpenMP over output rows.  ``gemm_py`` is a pure
Python twin for tiny sizes.  Parity pins for every function live in
``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "oracle_gemm.c"
_BUILD = _HERE / "_build"
_LIB = _BUILD / "liboracle.so"
_lib = None

_i64 = ctypes.c_int64
_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> Path:
    """Compile the C oracle with gcc (plain C, OpenMP, no FMA contraction)."""
    _BUILD.mkdir(exist_ok=True)
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _BUILD / f"liboracle.{os.getpid()}.so"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", str(_SRC), "-o", str(tmp), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_LIB))
        lib.oracle_gemm.argtypes = [_i64, _i64, _i64, _dp, _i64, _dp, _i64, ctypes.c_int,
                                    _dp, ctypes.c_int, _dp, _i64, _dp, _i64, ctypes.c_int]
        lib.oracle_gemm_rows.argtypes = [_i64, _i64, _dp, _i64, _dp, _i64, ctypes.c_int,
                                         _dp, ctypes.c_int, _ip, _i64, _dp, _dp, ctypes.c_int]
        lib.oracle_gemm_cols.argtypes = [_i64, _i64, _dp, _i64, _dp, _i64, ctypes.c_int,
                                         _dp, ctypes.c_int, _ip, _i64, _dp, _dp, ctypes.c_int]
        lib.oracle_conv2d_at.argtypes = [_i64] * 8 + [_dp, _dp, _ip, _i64, _dp]
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def e4m3_to_f64(codes) -> np.ndarray:
    """FP8 E4M3 bytes (the OCP "fn" variant: no infinities) to float64, from the
    format: bit 7 sign, bits 6..3 exponent with bias 7, bits 2..0 mantissa;
    exponent 0 encodes subnormals m/8 * 2^-6; S.1111.111 is NaN (so the largest
    finite value is 1.75 * 2^8 = 448)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    v = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    v = np.where((e == 15) & ((c & 7) == 7), np.nan, v)
    return sign * v


def e5m2_to_f64(codes) -> np.ndarray:
    """FP8 E5M2 bytes to float64, IEEE-754 style: bit 7 sign, bits 6..2 exponent
    with bias 15, bits 1..0 mantissa; exponent 0 encodes subnormals m/4 * 2^-14;
    exponent 31 is infinity (m = 0) or NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 2) & 0x1F
    m = (c & 3).astype(np.float64)
    v = np.where(e == 0, m / 4.0 * 2.0 ** -14, (1.0 + m / 4.0) * np.exp2(e - 15.0))
    v = np.where(e == 31, np.where((c & 3) == 0, np.inf, np.nan), v)
    return sign * v


def _f64(x) -> np.ndarray:
    """Widen to a C-contiguous float64 numpy array (exact for bf16/fp16/fp32/int;
    fp8 tensors are decoded from their bytes by e4m3_to_f64 / e5m2_to_f64)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu()
            if x.dtype == torch.float8_e4m3fn:
                return np.ascontiguousarray(e4m3_to_f64(x.view(torch.uint8).numpy()))
            if x.dtype == torch.float8_e5m2:
                return np.ascontiguousarray(e5m2_to_f64(x.view(torch.uint8).numpy()))
            x = x.to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(_dp)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def gemm(A, B, bias=None, relu: bool = False, b_nk: bool = False,
         with_mag: bool = False, threads: int = 0):
    """Full product in float64.

    A is M x K.  B is K x N, or N x K when ``b_nk`` (a Linear weight W).
    Returns C (M x N), and also S = sum_k |A_ik B_kj| when ``with_mag``.
    """
    A = _f64(A); B = _f64(B)
    M, K = A.shape
    N = B.shape[0] if b_nk else B.shape[1]
    assert (B.shape[1] if b_nk else B.shape[0]) == K, "inner dimensions differ"
    bias_a = None if bias is None else _f64(bias).reshape(-1)
    C = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64) if with_mag else None
    if M and N:
        _load().oracle_gemm(M, N, K, _ptr(A), K, _ptr(B), B.shape[1], int(b_nk),
                            _ptr(bias_a), int(relu), _ptr(C), N, _ptr(S), N, int(threads))
    return (C, S) if with_mag else C


def epilogue_ex(P, alpha=1.0, beta=0.0, C0=None, scale=None, bias=None, relu=False):
    """The extended epilogue written out on a float64 product P (M x N):
    t = alpha * P; t = t * scale[j]; t = t + bias[j]; t = t + beta * C0[i][j];
    t = max(0, t) -- each step only when its operand is given (the BLAS update
    C = alpha A.B + beta C of the youngju.dev "GEMM interface" listing, plus the
    per-channel scale / bias / ReLU of the CMU 15-418 notes' fused convolution,
    section 3.1)."""
    t = float(alpha) * np.asarray(P, dtype=np.float64)
    if scale is not None:
        t = t * _f64(scale).reshape(1, -1)
    if bias is not None:
        t = t + _f64(bias).reshape(1, -1)
    if beta != 0.0:
        t = t + float(beta) * _f64(C0)
    if relu:
        t = np.maximum(t, 0.0)
    return t


def gemm_ex(A, B, alpha=1.0, beta=0.0, C0=None, scale=None, bias=None, relu=False, b_nk=False, threads=0):
    """C = epilogue_ex(A.B) in float64, with the magnitude bound of each output:
    returns (C, S) where S = |alpha * scale_j| * sum_k |A_ik B_kj| (the part of
    the parity tolerance that scales with the products)."""
    P, S = gemm(A, B, b_nk=b_nk, with_mag=True, threads=threads)
    C = epilogue_ex(P, alpha, beta, C0, scale, bias, relu)
    f = abs(float(alpha)) * (np.abs(_f64(scale)).reshape(1, -1) if scale is not None else 1.0)
    return C, S * f


def gemm_rows(A, B, rows, bias=None, relu=False, b_nk=False, with_mag=False, threads=0):
    """Full rows ``rows`` of the product (len(rows) x N)."""
    A = _f64(A); B = _f64(B)
    M, K = A.shape
    N = B.shape[0] if b_nk else B.shape[1]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < M)
    bias_a = None if bias is None else _f64(bias).reshape(-1)
    C = np.zeros((rows.size, N)); S = np.zeros((rows.size, N)) if with_mag else None
    if rows.size and N:
        _load().oracle_gemm_rows(N, K, _ptr(A), K, _ptr(B), B.shape[1], int(b_nk),
                                 _ptr(bias_a), int(relu), rows.ctypes.data_as(_ip), rows.size,
                                 _ptr(C), _ptr(S), int(threads))
    return (C, S) if with_mag else C


def gemm_cols(A, B, cols, bias=None, relu=False, b_nk=False, with_mag=False, threads=0):
    """Full columns ``cols`` of the product (M x len(cols))."""
    A = _f64(A); B = _f64(B)
    M, K = A.shape
    N = B.shape[0] if b_nk else B.shape[1]
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    assert cols.size == 0 or (cols.min() >= 0 and cols.max() < N)
    bias_a = None if bias is None else _f64(bias).reshape(-1)
    C = np.zeros((M, cols.size)); S = np.zeros((M, cols.size)) if with_mag else None
    if cols.size and M:
        _load().oracle_gemm_cols(M, K, _ptr(A), K, _ptr(B), B.shape[1], int(b_nk),
                                 _ptr(bias_a), int(relu), cols.ctypes.data_as(_ip), cols.size,
                                 _ptr(C), _ptr(S), int(threads))
    return (C, S) if with_mag else C


def gemm_py(A, B, bias=None, relu=False):
    """Pure-Python triple loop (i, j, k), for tiny inputs only."""
    A = [[float(v) for v in row] for row in _f64(A)]
    B = [[float(v) for v in row] for row in _f64(B)]
    M, K, N = len(A), len(B), len(B[0]) if B else 0
    C = [[0.0] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            acc = 0.0
            for k in range(K):
                acc += A[i][k] * B[k][j]
            if bias is not None:
                acc += float(bias[j])
            if relu:
                acc = max(0.0, acc)
            C[i][j] = acc
    return np.array(C, dtype=np.float64).reshape(M, N)


# ---------------------------------------------------------------- bf16 ----
# bf16 has 8 significant bits (1 implicit + 7 stored), exponent range of fp32:
# normal numbers 2^-126 .. (2 - 2^-7) * 2^127, subnormal spacing 2^-133.
_BF16_MIN_EXP = -126
_BF16_SUB_ULP = 2.0 ** -133
_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    Written from the format definition: write |x| = m * 2^e with 1 <= m < 2,
    keep 8 significant bits (quantum 2^(e-7)), or the fixed subnormal quantum
    2^-133 below 2^-126, and round the scaled value half-to-even.  Values
    beyond the largest finite bf16 after rounding become +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    finite = np.isfinite(x)
    out[~finite] = x[~finite]
    xf = x[finite]
    ax = np.abs(xf)
    _, e2 = np.frexp(ax)             # ax = f * 2^e2, 0.5 <= f < 1  =>  exponent e = e2 - 1
    e = e2 - 1
    quantum = np.where(e < _BF16_MIN_EXP, _BF16_SUB_ULP, np.ldexp(1.0, e - 7))
    quantum = np.where(ax == 0.0, _BF16_SUB_ULP, quantum)
    q = np.rint(ax / quantum) * quantum   # ax/quantum is exact (power-of-two scale); rint is RNE
    q = np.where(q > _BF16_MAX, np.inf, q)
    out[finite] = np.copysign(q, xf)
    return out


def ulp_bf16(x) -> np.ndarray:
    """Spacing of bf16 numbers at |x|: 2^(floor(log2|x|) - 7), or 2^-133 at 0/subnormal."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, e2 = np.frexp(ax)
    e = e2 - 1
    u = np.where(e < _BF16_MIN_EXP, _BF16_SUB_ULP, np.ldexp(1.0, e - 7))
    return np.where(ax == 0.0, _BF16_SUB_ULP, u)


# ------------------------------------------------------------ tolerance ----
def tolerance(S, C_ref=None, out_bf16: bool = False) -> np.ndarray:
    """Per-element bound: 1e-3 * sum_k |A_ik B_kj| + 1e-6, plus one bf16 ulp
    of |C_ref| when the result went through a bf16 output cast."""
    t = 1e-3 * np.asarray(S, dtype=np.float64) + 1e-6
    if out_bf16:
        t = t + ulp_bf16(C_ref)
    return t


def check_close(C, C_ref, S, out_bf16: bool = False):
    """Return (ok, worst_ratio, index): worst |C - C_ref| / bound over all elements."""
    C = _f64(C); C_ref = np.asarray(C_ref, dtype=np.float64)
    bound = tolerance(S, C_ref, out_bf16)
    err = np.abs(C - C_ref)
    if err.size == 0:
        return True, 0.0, None
    ratio = err / bound
    idx = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
    worst = float(ratio[idx])
    return bool(np.all(err <= bound) and np.all(np.isfinite(C))), worst, idx


def exact_expected(C_ref, out_bf16: bool) -> np.ndarray:
    """Expected output for integer inputs: C_ref is an exact integer below 2^24,
    so the device's fp32 accumulator holds it exactly; a bf16 output is its
    single round-to-nearest-even."""
    return bf16_round(C_ref) if out_bf16 else np.asarray(C_ref, dtype=np.float64)


# ------------------------------------------------------------ Freivalds ----
def freivalds_int(A, B, C, r, b_nk=False, bias=None, relu=False):
    """Exact whole-matrix check for integer data (Freivalds 1977).

    Compares C r with A (B r) in int64, which holds every intermediate for the
    sizes used (|entries| <= 4, K <= 16384, N <= 16384).  Only valid without
    ReLU (ReLU is not linear); bias adds (sum_j bias_j r_j) to every row.
    Returns the number of rows that disagree.
    """
    assert not relu
    A = np.asarray(_f64(A)).astype(np.int64)
    B = np.asarray(_f64(B)).astype(np.int64)
    C = np.asarray(_f64(C)).astype(np.int64)
    r = np.asarray(r, dtype=np.int64)
    Br = (B @ r) if not b_nk else (B.T @ r)
    lhs = C @ r
    rhs = A @ Br
    if bias is not None:
        rhs = rhs + int(np.asarray(_f64(bias)).astype(np.int64) @ r)
    return int(np.count_nonzero(lhs != rhs))


def freivalds_float(A, B, C, r, b_nk=False, bias=None, out_bf16=False):
    """Whole-matrix check for float data against the propagated bound.

    |(C r)_i - (A (B r))_i| <= sum_j |r_j| tol_ij, where sum_j |r_j| * 1e-3 *
    sum_k |A_ik B_kj| = 1e-3 * (|A| (|B| |r|))_i.  For a bf16 output each
    element may also be off by one ulp of |C_ref|, bounded here by 2 ulp of
    |C| (C is within a factor 2 of C_ref at that point) plus the subnormal
    ulp.  Returns (ok, worst ratio).
    """
    A = _f64(A); B = _f64(B); C = _f64(C)
    r = np.asarray(r, dtype=np.float64)
    Bt = B.T if b_nk else B
    lhs = C @ r
    rhs = A @ (Bt @ r)
    if bias is not None:
        rhs = rhs + float(_f64(bias) @ r)
    bound = 1e-3 * (np.abs(A) @ (np.abs(Bt) @ np.abs(r))) + 1e-6 * np.abs(r).sum()
    if out_bf16:
        bound = bound + (2.0 * ulp_bf16(C) + _BF16_SUB_ULP) @ np.abs(r)
    # float64 evaluation of both sides adds rounding far below the bound
    bound = bound * (1.0 + 1e-9) + 1e-12
    ratio = np.abs(lhs - rhs) / bound
    return bool(np.all(ratio <= 1.0)), float(ratio.max(initial=0.0))


# ---------------------------------------------------------- convolution ----
def im2col(x, R: int, S: int, pad: int):
    """Explicit-GEMM matrix of a stride-1 convolution (definition written out).

    x is NHWC (Nb, H, W, C).  Row (n*OH + oh)*OW + ow holds the R x S x C
    neighbourhood of output (n, oh, ow), column (r*S + s)*C + c is
    x[n, oh+r-pad, ow+s-pad, c], zero outside the image.
    """
    x = _f64(x)
    Nb, H, W, C = x.shape
    OH, OW = H + 2 * pad - R + 1, W + 2 * pad - S + 1
    out = np.zeros((Nb * OH * OW, R * S * C))
    for n in range(Nb):
        for oh in range(OH):
            for ow in range(OW):
                row = (n * OH + oh) * OW + ow
                for r in range(R):
                    for s in range(S):
                        ih, iw = oh + r - pad, ow + s - pad
                        if 0 <= ih < H and 0 <= iw < W:
                            out[row, (r * S + s) * C:(r * S + s + 1) * C] = x[n, ih, iw, :]
    return out


def im2col_rows(x, R: int, S: int, pad: int, rows):
    """Selected rows of ``im2col`` without materialising the whole matrix."""
    x = _f64(x)
    Nb, H, W, C = x.shape
    OH, OW = H + 2 * pad - R + 1, W + 2 * pad - S + 1
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.size, R * S * C))
    for t, row in enumerate(rows):
        n, rem = divmod(int(row), OH * OW)
        oh, ow = divmod(rem, OW)
        for r in range(R):
            for s in range(S):
                ih, iw = oh + r - pad, ow + s - pad
                if 0 <= ih < H and 0 <= iw < W:
                    out[t, (r * S + s) * C:(r * S + s + 1) * C] = x[n, ih, iw, :]
    return out


def conv2d_at(x, w, pad: int, positions):
    """Direct convolution at output positions (n, oh, ow); x NHWC, w[f][r][s][c]."""
    x = _f64(x); w = _f64(w)
    Nb, H, W, Cin = x.shape
    Cout, R, S, Cin2 = w.shape
    assert Cin == Cin2
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64).reshape(-1, 3))
    out = np.zeros((pos.shape[0], Cout))
    if pos.shape[0]:
        _load().oracle_conv2d_at(Nb, H, W, Cin, Cout, R, S, pad, _ptr(x), _ptr(w),
                                 pos.ctypes.data_as(_ip), pos.shape[0], _ptr(out))
    return out


def conv2d_maxpool_at(x, w, pad: int, pooled_positions, alpha=1.0, scale=None, bias=None, relu=False):
    """Convolution, epilogue and 2 x 2 max-pool at pooled positions (n, ph, pw),
    the single-pass fused example of the CMU 15-418 notes, section 3.1: the
    maximum over dy, dx in {0, 1} of epilogue_ex(conv(x, w)[n, 2 ph + dy, 2 pw + dx])."""
    pos = np.asarray(pooled_positions, dtype=np.int64).reshape(-1, 3)
    outs = []
    for dy in (0, 1):
        for dx in (0, 1):
            full = [(int(n), int(2 * ph + dy), int(2 * pw + dx)) for n, ph, pw in pos]
            outs.append(epilogue_ex(conv2d_at(x, w, pad, full), alpha=alpha, scale=scale, bias=bias, relu=relu))
    return np.maximum(np.maximum(outs[0], outs[1]), np.maximum(outs[2], outs[3]))


def attention(Q, K, V, scale=None, causal=False):
    """Attention in float64 (CMU 15-418 notes, section 3.3: S = scale * Q K^T,
    each row's softmax, O = P V; the reference that example computes by
    materialising S).  Q [..., Sq, D], K and V [..., Sk, D].  causal: key j is
    visible to query i iff j <= i + (Sk - Sq); a row with no visible key gives
    zeros.  scale None means 1 / sqrt(D)."""
    Q = _f64(Q); K = _f64(K); V = _f64(V)
    Sq, D = Q.shape[-2], Q.shape[-1]
    Sk = K.shape[-2]
    s = (1.0 / np.sqrt(D)) if scale is None else float(scale)
    S = np.matmul(Q, np.swapaxes(K, -1, -2)) * s
    vis = np.ones((Sq, Sk), dtype=bool)
    if causal:
        vis = np.arange(Sk)[None, :] <= (np.arange(Sq)[:, None] + (Sk - Sq))
    S = np.where(vis, S, -np.inf)
    mx = np.max(S, axis=-1, keepdims=True)
    mx = np.where(np.isfinite(mx), mx, 0.0)
    E = np.where(vis, np.exp(S - mx), 0.0)
    den = E.sum(axis=-1, keepdims=True)
    P = np.where(den > 0, E / np.where(den > 0, den, 1.0), 0.0)
    return np.matmul(P, V)


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
