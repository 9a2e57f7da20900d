/*
 * Float64 reference for the dense matrix multiply and its Linear-layer form.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA path is
 * checked against.  It shares no code, header or constant with the CUDA
 * library and must never be linked into it.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg load it.
 *
 * What it computes (youngju.dev, "GEMM to FlashAttention", the `naive_matmul`
 * listing and the Linear-layer header `output = W x input + b`):
 *
 *     C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]          (ascending k)
 *     C[i][j] += bias[j]                                    (optional)
 *     C[i][j]  = max(0, C[i][j])                            (optional ReLU)
 *
 * The ReLU definition f(x) = max(0, x) applied after the bias follows the
 * neuron f(sum_i x_i w_i + b) of the CMU 15-418 "DNNs and ML accelerators"
 * notes, section 2.1.  All arithmetic is IEEE float64; the build uses
 * -ffp-contract=off so no multiply-add is fused.  The loop order is i-k-j:
 * for a fixed (i, j) the products are still added one by one in ascending k,
 * exactly as in the plain triple loop; only the order in which different
 * output elements progress is changed, which does not alter any element.
 *
 * B may be given K x N ("kn", B[k][j] at B[k*ldb + j]) or, for a Linear
 * weight W stored out x in, N x K ("nk", B(k, j) = W[j][k] at B[j*ldb + k]).
 *
 * Besides C the oracle can return S[i][j] = sum_k |A[i][k] * B[k][j]|, the
 * magnitude sum that the parity tolerance is scaled by.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static inline double b_at(const double* B, int64_t ldb, int b_nk, int64_t k, int64_t j) {
    return b_nk ? B[j * ldb + k] : B[k * ldb + j];
}

/* One output row i of the definition, written into crow[0..N-1] (and the
 * magnitude sums into srow when srow is not NULL). */
static void oracle_row(int64_t i, int64_t N, int64_t K,
                       const double* A, int64_t lda,
                       const double* B, int64_t ldb, int b_nk,
                       const double* bias, int relu,
                       double* crow, double* srow) {
    for (int64_t j = 0; j < N; ++j) {
        crow[j] = 0.0;
        if (srow) srow[j] = 0.0;
    }
    if (!b_nk) {
        /* i-k-j: stream row k of B; each crow[j] still sums in ascending k */
        for (int64_t k = 0; k < K; ++k) {
            const double a = A[i * lda + k];
            const double* brow = B + k * ldb;
            for (int64_t j = 0; j < N; ++j) {
                const double p = a * brow[j];
                crow[j] = crow[j] + p;
                if (srow) srow[j] = srow[j] + fabs(p);
            }
        }
    } else {
        /* i-j-k: row j of W is contiguous in k */
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0, mag = 0.0;
            const double* wrow = B + j * ldb;
            for (int64_t k = 0; k < K; ++k) {
                const double p = A[i * lda + k] * wrow[k];
                acc = acc + p;
                mag = mag + fabs(p);
            }
            crow[j] = acc;
            if (srow) srow[j] = mag;
        }
    }
    for (int64_t j = 0; j < N; ++j) {
        double y = crow[j];
        if (bias) y = y + bias[j];
        if (relu) y = (y > 0.0) ? y : 0.0;
        crow[j] = y;
    }
}

/* Full product: C (M x N, leading dimension ldc).  S may be NULL. */
void oracle_gemm(int64_t M, int64_t N, int64_t K,
                 const double* A, int64_t lda,
                 const double* B, int64_t ldb, int b_nk,
                 const double* bias, int relu,
                 double* C, int64_t ldc, double* S, int64_t lds,
                 int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < M; ++i)
        oracle_row(i, N, K, A, lda, B, ldb, b_nk, bias, relu,
                   C + i * ldc, S ? S + i * lds : NULL);
    (void)nthreads;
}

/* Selected full rows: out row r is row rows[r] of the product (nrows x N). */
void oracle_gemm_rows(int64_t N, int64_t K,
                      const double* A, int64_t lda,
                      const double* B, int64_t ldb, int b_nk,
                      const double* bias, int relu,
                      const int64_t* rows, int64_t nrows,
                      double* C, double* S, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < nrows; ++r)
        oracle_row(rows[r], N, K, A, lda, B, ldb, b_nk, bias, relu,
                   C + r * N, S ? S + r * N : NULL);
    (void)nthreads;
}

/* Selected full columns: out[i][c] is element (i, cols[c]) (M x ncols). */
void oracle_gemm_cols(int64_t M, int64_t K,
                      const double* A, int64_t lda,
                      const double* B, int64_t ldb, int b_nk,
                      const double* bias, int relu,
                      const int64_t* cols, int64_t ncols,
                      double* C, double* S, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t c = 0; c < ncols; ++c) {
            const int64_t j = cols[c];
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double p = A[i * lda + k] * b_at(B, ldb, b_nk, k, j);
                acc = acc + p;
                mag = mag + fabs(p);
            }
            if (bias) acc = acc + bias[j];
            if (relu) acc = (acc > 0.0) ? acc : 0.0;
            C[i * ncols + c] = acc;
            if (S) S[i * ncols + c] = mag;
        }
    }
    (void)nthreads;
}

/*
 * Direct 3x3-style convolution, the seven-loop nest of the CMU 15-418 notes,
 * section 2.2 (batch x output row x output column x output channel x input
 * channel x filter row x filter column), evaluated at selected output
 * positions.  Input x is NHWC (Nb x H x W x Cin), weights w[f][r][s][c]
 * (the layout of the fused-convolution example, section 3.1), stride 1 and
 * zero padding `pad`, output y[n][oh][ow][f] in NHWC.  pos holds npos
 * triples (n, oh, ow); out is npos x Cout.
 */
void oracle_conv2d_at(int64_t Nb, int64_t H, int64_t W, int64_t Cin,
                      int64_t Cout, int64_t R, int64_t S_, int64_t pad,
                      const double* x, const double* w,
                      const int64_t* pos, int64_t npos, double* out) {
    (void)Nb;
    const int64_t OH = H + 2 * pad - R + 1, OW = W + 2 * pad - S_ + 1;
    (void)OH; (void)OW;
    /* positions are independent: one thread per position, each sum in the
     * order of the loop nest below */
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t p = 0; p < npos; ++p) {
        const int64_t n = pos[3 * p], oh = pos[3 * p + 1], ow = pos[3 * p + 2];
        for (int64_t f = 0; f < Cout; ++f) {
            double acc = 0.0;
            for (int64_t c = 0; c < Cin; ++c)
                for (int64_t r = 0; r < R; ++r)
                    for (int64_t s = 0; s < S_; ++s) {
                        const int64_t ih = oh + r - pad, iw = ow + s - pad;
                        if (ih < 0 || ih >= H || iw < 0 || iw >= W) continue;
                        acc = acc + x[((n * H + ih) * W + iw) * Cin + c] *
                                        w[((f * R + r) * S_ + s) * Cin + c];
                    }
            out[p * Cout + f] = acc;
        }
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
