/*
 * gemm.h -- C ABI of the GB300 (sm_103a) GEMM / Linear-layer library.
 *
 * Operation (youngju.dev "GEMM to FlashAttention": the `naive_matmul` listing
 * C[i][j] = sum_k A[i][k] * B[k][j]; the Linear-layer header
 * output = W x input + b; CMU 15-418 "DNNs and ML accelerators" notes,
 * section 2.1: activation f(x) = max(0, x) applied after the bias):
 *
 *     C[i][j] = cast( relu?( sum_{k<K} A[i][k] * B(k, j)  (+ bias[j]) ) )
 *
 * Layout.  Every matrix is row-major with an explicit leading dimension given
 * in ELEMENTS (the lda/ldb/ldc of the BLAS GEMM interface, same page, "GEMM
 * interface").  A is M x K (A[i][k] at A + i*lda + k, lda >= K).  B is K x N
 * (B[k][j] at B + k*ldb + j, ldb >= N) by default; with the plan flag
 * GEMM_B_NK, B is a Linear weight W stored N x K, out x in (B(k, j) = W[j][k]
 * at B + j*ldb + k, ldb >= K) -- the "transb" of the BLAS interface.  C is
 * M x N (ldc >= N).  bias has N elements of the input type (bf16 for fp8 and
 * tf32 inputs).  With the plan flag GEMM_A_KM, A is stored K x M instead.
 *
 * Numerics.  A, B: bf16, fp16, fp8 (e4m3 / e5m2) or fp32 read as tf32 (see
 * gemm_dtype_t); products and sums in fp32 (the mixed-precision rule of the
 * same notes, section 2.7: low-precision storage, fp32 accumulation); the bias
 * is added in fp32 before the ReLU and the single final cast (round to
 * nearest even) to the output type.  gemm_run: alpha = 1 and beta = 0, C is
 * overwritten, never read; gemm_run_ex takes alpha, beta, a per-column scale.
 *
 * Memory.  A, B, bias and C are DEVICE pointers on the plan's device, owned by
 * the caller and never freed by the library.  The plan owns a small device
 * status block and, only when needed, a workspace: packed copies of operands
 * that break the 16-byte rule of the TMA copies (base address or leading
 * dimension x element size not a multiple of 16 bytes), K-major copies of tf32
 * operands stored MN-major, and the partial tiles of the optional stream-K
 * split.  The workspace is allocated on first need, grows, and is freed by
 * gemm_plan_destroy.
 *
 * Asynchrony.  gemm_run enqueues its kernels on `stream` (a cudaStream_t,
 * NULL = legacy default stream) and returns without waiting.  Only
 * gemm_plan_status synchronises.  A plan may be used by one stream at a time.
 *
 * Errors.  Every function returns 0 (GEMM_OK) or a negative GEMM_ERR_* code;
 * nothing is launched when argument validation fails.  No function exits the
 * process or throws.  Device-side waits are bounded: a wait that runs out of
 * time records GEMM_ERR_DEVICE_TIMEOUT in the plan's status word, which
 * gemm_plan_status reports (and clears).
 */
#ifndef GB300_GEMM_H
#define GB300_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gemm_plan* gemm_plan_t;

/* Epilogue applied to the fp32 accumulator before the output cast. */
typedef enum {
    GEMM_EPI_NONE = 0,       /* C = A.B                 */
    GEMM_EPI_BIAS = 1,       /* C = A.B + bias          */
    GEMM_EPI_RELU = 2,       /* C = max(0, A.B)         */
    GEMM_EPI_BIAS_RELU = 3   /* C = max(0, A.B + bias)  */
} gemm_epilogue_t;

/* Input type of A, B (and bias, scale) and output type of C.  The fp8 types
 * (OCP e4m3 / e5m2 bytes, both operands in one format; CMU 15-418 notes,
 * section 2.7: fewer bytes per operand, fp32 accumulation) take bf16 bias and
 * scale vectors, B stored either way and A either way (GEMM_A_KM), and run on
 * the small-M kernel for M <= 128 (A stored M x K), on the large-M kernels
 * otherwise; per-tensor scale factors go in gemm_run_ex's alpha.  The
 * tf32 types take fp32 A and B in memory, which
 * the tensor cores multiply at tf32 precision (8-bit exponent, 10-bit
 * mantissa; CMU 15-418 notes, section 2.7), with fp32 accumulation; like fp8
 * they take bf16 bias and scale vectors and every operand layout, and run on
 * the large-M kernels.  Neither type is taken by the convolution entry points
 * or by gemm_run_noalloc (GEMM_ERR_UNSUPPORTED). */
typedef enum {
    GEMM_BF16_F32OUT = 0,
    GEMM_BF16_BF16OUT = 1,
    GEMM_F16_F32OUT = 2,
    GEMM_F16_F16OUT = 3,
    GEMM_E4M3_F32OUT = 4,
    GEMM_E4M3_BF16OUT = 5,
    GEMM_E5M2_F32OUT = 6,
    GEMM_E5M2_BF16OUT = 7,
    GEMM_TF32_F32OUT = 8,
    GEMM_TF32_BF16OUT = 9
} gemm_dtype_t;

/* Plan flags. */
#define GEMM_B_KN 0u   /* B is K x N (default) */
#define GEMM_B_NK 1u   /* B is a Linear weight W, N x K */
/* B is constant while the plan's kernels may run (model weights): no earlier
 * work on the stream writes it.  Lets the small-M kernel start streaming B
 * while the previous kernel of the stream is still finishing; A, bias and C
 * are still touched only after that kernel is done. */
#define GEMM_B_CONST 2u
/* A is stored K x M (the transpose of the M x K operand, BLAS "transa"):
 * A(i, k) = A[k * lda + i], lda >= M.  Runs on the tensor-core kernels (also for
 * M <= 128), for every input type; not taken by gemm_run_noalloc. */
#define GEMM_A_KM 8u

/* Kernel selection (gemm_plan_set_kernel / gemm_plan_last_kernel). */
#define GEMM_KERNEL_AUTO 0
#define GEMM_KERNEL_TC_PAIR 1   /* tcgen05, 2-CTA clusters (cta_group::2), 256 x 256 tiles */
#define GEMM_KERNEL_TC_SINGLE 2 /* tcgen05, one CTA per tile (cta_group::1), 128 x 256 tiles */
#define GEMM_KERNEL_FILL 3      /* K == 0: epilogue of an empty sum */
#define GEMM_KERNEL_SKINNY 4    /* small-M Linear layer (weight streaming, tensor cores) */
#define GEMM_KERNEL_GEMV 5      /* M <= 4, B stored N x K: CUDA-core GEMV (weight streaming; auto for M = 1) */
/* 2 <= M <= 16, 16-bit or fp8 operands, B stored N x K: weight streaming with
 * warp-level tensor-core MMAs (mma.sync), no staging (auto for 2 <= M <= 8) */
#define GEMM_KERNEL_WARP_MMA 6

/* Return codes. */
#define GEMM_OK 0
#define GEMM_ERR_INVALID_ARG (-1)     /* null/negative/inconsistent argument   */
#define GEMM_ERR_ALIGNMENT (-2)       /* misaligned operand and packing disabled */
#define GEMM_ERR_UNSUPPORTED (-3)     /* dtype/epilogue/kernel not available   */
#define GEMM_ERR_CUDA (-4)            /* a CUDA call failed; see gemm_plan_last_cuda_error */
#define GEMM_ERR_DEVICE_TIMEOUT (-5)  /* a device-side wait ran out of time    */
#define GEMM_ERR_NO_MEMORY (-6)       /* workspace allocation failed           */

/* Extended epilogue (gemm_run_ex, gemm_conv2d), applied to the fp32
 * accumulator acc = sum_k A[i][k] B(k, j) in this order:
 *     t = alpha * acc;  t = t * scale[j]   (if scale);  t = t + bias[j] (if bias);
 *     t = t + beta * C_old[i][j]           (if beta != 0);  t = max(0, t) (if relu);
 *     C[i][j] = cast(t).
 * With scale = bias = NULL, relu = 0 this is the BLAS update C = alpha A.B +
 * beta C (youngju.dev "GEMM to FlashAttention", "GEMM interface"); scale, bias
 * and relu give the per-channel scale / bias / ReLU of a fused convolution
 * epilogue (CMU 15-418 notes, section 3.1).  C_old is C itself, read before it
 * is written (element by element, so C may be updated in place); scale and
 * bias hold N values of the input type (device memory). */
typedef struct {
    float alpha;          /* factor on A.B: 1 for the plain product           */
    float beta;           /* factor on the previous C: 0 = C is only written  */
    const void* scale;    /* NULL or N per-column factors                     */
    const void* bias;     /* NULL or N per-column addends                     */
    int relu;             /* nonzero: ReLU before the cast                    */
} gemm_epilogue_args_t;

/* Create a plan for `device` (a CUDA ordinal): the handle of the
 * create / use / destroy pattern of the cuBLAS example on youngju.dev "GEMM to
 * FlashAttention" (BLAS/cuBLAS interface listing), which gemm_run then takes
 * as its first argument.  flags: GEMM_B_KN or GEMM_B_NK, optionally
 * | GEMM_A_KM and | GEMM_B_CONST; any other bit is GEMM_ERR_INVALID_ARG.
 * Allocates the plan and its device status word; restores the caller's
 * current device before returning.  *plan is set only on success. */
int gemm_plan_create(gemm_plan_t* plan, int device, unsigned flags);

/* C = epilogue(A.B) (see above).  M, N, K >= 0; M == 0 or N == 0 is a no-op;
 * K == 0 writes epilogue(0).  `bias` may be NULL unless the epilogue adds it.
 * `epilogue` is a gemm_epilogue_t, `dtype` a gemm_dtype_t, `stream` a
 * cudaStream_t.  Every pointer must lie on a boundary of its element size
 * (else GEMM_ERR_INVALID_ARG); pitches and 16-byte alignment are free (the
 * plan packs what TMA cannot read).  tf32 operands stored MN-major (A with
 * GEMM_A_KM, B without GEMM_B_NK) are transposed into the plan's workspace
 * before the product, whatever gemm_plan_set_packing says.  Returns after
 * enqueueing the work. */
int gemm_run(gemm_plan_t plan, int64_t M, int64_t N, int64_t K,
             const void* A, int64_t lda, const void* B, int64_t ldb, const void* bias,
             void* C, int64_t ldc, int epilogue, int dtype, void* stream);

/* As gemm_run with the extended epilogue `epi` (not NULL; see
 * gemm_epilogue_args_t).  When epi->beta != 0 the previous contents of C are
 * read (C must be initialised).  Same returns as gemm_run. */
int gemm_run_ex(gemm_plan_t plan, int64_t M, int64_t N, int64_t K,
                const void* A, int64_t lda, const void* B, int64_t ldb,
                void* C, int64_t ldc, const gemm_epilogue_args_t* epi, int dtype, void* stream);

/* Synchronise the stream of the last gemm_run and report device-side errors:
 * GEMM_ERR_DEVICE_TIMEOUT if a bounded wait ran out since the last call (the
 * status word is then cleared), GEMM_ERR_CUDA if the stream reports an error.
 * The pages have no counterpart: it is this library's design, the host end of
 * the bounded device-side waits (a wait that runs out reports here instead of
 * hanging the GPU). */
int gemm_plan_status(gemm_plan_t plan);

/* Release the plan, its status word and its workspace (the destroy step of
 * the cuBLAS handle pattern, youngju.dev "GEMM to FlashAttention",
 * BLAS/cuBLAS interface listing).  Waits for the plan's last stream first.
 * NULL is accepted. */
int gemm_plan_destroy(gemm_plan_t plan);

/* Static description of a return code (never NULL; "unknown error" for a
 * code not listed above).  The pages have no counterpart: it is this
 * library's design, so that callers across the C ABI can print an error. */
const char* gemm_strerror(int code);

/* Explicit-GEMM (im2col) matrix of a convolution (CMU 15-418 "DNNs and ML
 * accelerators" notes, section 2.3: each R x S x C input neighbourhood becomes
 * one row; weights w[f][r][s][c] then form the N x K operand of gemm_run with
 * GEMM_B_NK).  x is NHWC (Nb x H x W x C, contiguous, device memory); out is
 * (Nb*OH*OW) x (R*S*C) row-major with row pitch ld_out >= R*S*C elements,
 * OH = (H + 2 pad - R) / stride + 1 (OW likewise):
 *     out[(n*OH + oh)*OW + ow][(r*S + s)*C + c] = x[n][oh*stride+r-pad][ow*stride+s-pad][c]
 * or 0 outside the image.  elem_bytes is the element size (2 for bf16/fp16).
 * Enqueued on `stream`; both buffers are caller-owned; returns GEMM_OK,
 * GEMM_ERR_INVALID_ARG or GEMM_ERR_CUDA. */
int gemm_im2col(const void* x, int64_t Nb, int64_t H, int64_t W, int64_t C, int R, int S, int pad, int stride,
                void* out, int64_t ld_out, int elem_bytes, void* stream);

/* Convolution as an implicit GEMM (CMU 15-418 "DNNs and ML accelerators"
 * notes, section 2.3: the im2col matrix need not be materialised; the GEMM's
 * operand tiles are gathered from the activations as they are needed).
 * Stride 1, zero padding `pad`:
 *     y[(n*OH + oh)*OW + ow][f] = epilogue( sum_{r<R, s<S, c<C}
 *         x[n][oh+r-pad][ow+s-pad][c] * w[f][r][s][c]  (+ bias[f]) )
 * with OH = H + 2 pad - R + 1, OW = W + 2 pad - S + 1 and x read as 0 outside
 * the image -- exactly gemm_run on gemm_im2col's matrix (M = Nb*OH*OW,
 * K = R*S*C) and the N x K weight matrix w (N = Cout).  x is NHWC
 * (Nb x H x W x C, contiguous), w is Cout x R x S x C (contiguous), y is
 * M x Cout row-major with row pitch ldy >= Cout; all are caller-owned device
 * memory; epi is NULL (plain convolution) or the extended epilogue of
 * gemm_run_ex (per-channel scale, bias, ReLU, beta * y); dtype as for gemm_run.
 * The plan's B-layout flag is ignored (w is always N x K).
 * When C is a multiple of 64, R == S, x is 16-byte aligned and M > 128, the
 * large-M kernel reads x through a TMA im2col tensor map (no extra memory);
 * otherwise the im2col matrix is built in the plan's workspace first (the
 * same result).  Returns as gemm_run. */
int gemm_conv2d(gemm_plan_t plan, int64_t Nb, int64_t H, int64_t W, int64_t C, int64_t Cout, int R, int S, int pad,
                const void* x, const void* w, void* y, int64_t ldy, const gemm_epilogue_args_t* epi, int dtype,
                void* stream);

/* Convolution fused with its epilogue and a 2 x 2 max-pool (stride 2), the
 * single-pass conv + scale/bias + ReLU + max-pool of CMU 15-418 "DNNs and ML
 * accelerators" notes, section 3.1 (example one):
 *     y[(n*PH + ph)*PW + pw][f] = max over dy, dx in {0, 1} of
 *         epilogue( conv(x, w)[n][2 ph + dy][2 pw + dx][f] )
 * with the convolution, OH and OW of gemm_conv2d, PH = OH / 2, PW = OW / 2,
 * and the epilogue of gemm_epilogue_args_t (alpha, scale, bias, relu; beta must
 * be 0; epi may be NULL).  OH and OW must be even (GEMM_ERR_INVALID_ARG).
 * Only the pooled values are written: y is (Nb*PH*PW) x Cout, row pitch ldy.
 * Runs on the large-M kernel with im2col loads, whose tiles are two output rows
 * x 64 columns, so every pooling window lies in one accumulator; it needs C a
 * multiple of 64, R == S, 16-bit inputs, x and y 16-byte aligned and
 * ldy x element size a multiple of 16 (else GEMM_ERR_UNSUPPORTED). */
int gemm_conv2d_maxpool(gemm_plan_t plan, int64_t Nb, int64_t H, int64_t W, int64_t C, int64_t Cout, int R, int S,
                        int pad, const void* x, const void* w, void* y, int64_t ldy,
                        const gemm_epilogue_args_t* epi, int dtype, void* stream);

/* Fused attention forward, per (batch, head):
 *     O = softmax(scale * Q K^T, each row over the visible keys) V
 * (the online-softmax / FlashAttention recurrence of CMU 15-418 "DNNs and ML
 * accelerators" notes, section 3.3, and youngju.dev "GEMM to FlashAttention":
 * the Sq x Sk scores are never written to memory).  Q and O are [B][H][Sq][D],
 * K and V [B][H][Sk][D], row-major and contiguous, 16-byte aligned device
 * memory (caller-owned); D is 64 or 128; dtype GEMM_BF16_* / GEMM_F16_*
 * (inputs, and fp32 or 16-bit O); scale <= 0 means 1 / sqrt(D).  causal != 0:
 * key j is visible to query i iff j <= i + (Sk - Sq); a query that sees no key
 * gets zeros.  Products and sums in fp32; the probabilities are rounded to the
 * input type before they multiply V.  B * H <= 65535.  Returns GEMM_OK,
 * GEMM_ERR_INVALID_ARG, GEMM_ERR_ALIGNMENT, GEMM_ERR_UNSUPPORTED or
 * GEMM_ERR_CUDA. */
int gemm_attention(gemm_plan_t plan, int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t D,
                   const void* Q, const void* K, const void* V, void* O, float scale, int causal, int dtype,
                   void* stream);

/* --- controls and introspection (benchmarks and tests) ------------------ */

/* Force a kernel (GEMM_KERNEL_*); GEMM_KERNEL_AUTO restores the dispatcher. */
int gemm_plan_set_kernel(gemm_plan_t plan, int kernel);

/* Kernel chosen by the last successful gemm_run (GEMM_KERNEL_*), or -1. */
int gemm_plan_last_kernel(gemm_plan_t plan);

/* Number of kernels this plan has launched since creation. */
int64_t gemm_plan_launch_count(gemm_plan_t plan);

/* cudaError_t of the last failing CUDA call made for this plan (0 if none). */
int gemm_plan_last_cuda_error(gemm_plan_t plan);

/* Bound, in nanoseconds, on any single device-side wait (default 1e9). */
int gemm_plan_set_timeout_ns(gemm_plan_t plan, uint64_t ns);

/* Allow (1, default) or forbid (0) packing of misaligned operands; when
 * forbidden, gemm_run returns GEMM_ERR_ALIGNMENT for them instead. */
int gemm_plan_set_packing(gemm_plan_t plan, int enabled);

/* Test hook: fault-injection flags.  Bit 0 makes the MMA warp skip the first
 * "accumulator ready" signal (gemm_attention: the first "PV product done"
 * signal) so a bounded wait runs out and the run reports
 * GEMM_ERR_DEVICE_TIMEOUT; the GPU context stays usable. */
int gemm_plan_set_debug(gemm_plan_t plan, unsigned flags);

/* Bytes of workspace the plan currently holds. */
int64_t gemm_plan_workspace_bytes(gemm_plan_t plan);

/* Tuning options of a plan, for benchmark sweeps and tests; the defaults are
 * the measured best and a caller never needs to change them.  No option
 * changes a result, only how the work is scheduled. */
/* tile-rows per rasterisation group, 1..1024, or 0 (default): 1 when one wave
 * of tiles spans three or more whole tile-rows, else 16 */
#define GEMM_OPT_GROUP_M 1
#define GEMM_OPT_TAIL_SPLIT 2      /* 0/1: run the last partial wave as half tiles (default 1) */
#define GEMM_OPT_K_SNAKE 3         /* 0/1: every other tile of a worker walks k backwards (default 1) */
#define GEMM_OPT_PDL 4             /* 0/1: programmatic dependent launch (default 1) */
#define GEMM_OPT_L2_POLICY 5       /* 0: A evict-last; 1: B evict-last; 2: both normal (default 0) */
#define GEMM_OPT_SKINNY_SPLITS 6   /* small-M kernel k-slices: 0 = automatic (default), 1, 2, 4, 8 */
#define GEMM_OPT_SKINNY_STAGES 7   /* small-M kernel ring depth: 0 = automatic (default), 2..8 */
#define GEMM_OPT_LOG 9             /* 0/1: one line per launch on stderr (default 0) */
#define GEMM_OPT_GEMV_MAX_M 10     /* M up to which the CUDA-core GEMV is chosen, 0..4 (default 1) */
#define GEMM_OPT_WARP_MMA_MAX_M 12 /* M up to which the warp-MMA kernel is chosen, 0..16 (default 8) */
/* Stream-K on the tensor-core kernels: in a launch of at least one full wave
 * of tiles, the tiles of the last, partial wave are split by k over the
 * workers so every worker carries the same work; the value is the fewest
 * k-atoms a worker takes (0: off, the last wave runs as N-halves; default
 * 0: on GB300 it measured equal or slower than the N-halves).  Split tiles
 * keep fp32 partials in the plan's workspace. */
#define GEMM_OPT_STREAM_K 11

/* Set / read a GEMM_OPT_* option.  GEMM_ERR_INVALID_ARG for a NULL plan, an
 * unknown option or a value outside the option's range (nothing changes). */
int gemm_plan_set_option(gemm_plan_t plan, int option, int64_t value);
int gemm_plan_get_option(gemm_plan_t plan, int option, int64_t* value);

/* Host-only argument check: the code gemm_run would return for these
 * arguments before touching the GPU (GEMM_OK if they are acceptable).
 * `flags` are the plan flags.  Needs no device and launches nothing. */
int gemm_validate(unsigned flags, int64_t M, int64_t N, int64_t K,
                  const void* A, int64_t lda, const void* B, int64_t ldb, const void* bias,
                  const void* C, int64_t ldc, int epilogue, int dtype);

/* --- entry point for callers that cannot allocate device memory --------- */

/* Size in bytes of the fixed device scratch that gemm_run_noalloc uses on
 * every GPU where the library is loaded (held until the process exits). */
#define GEMM_NOALLOC_SCRATCH_BYTES 33554432u   /* 32 MiB */

/* The pages have no counterpart to this function; it exists for callers that
 * may not allocate device memory: processes whose HBM is reserved up front by
 * a pool or framework allocator, and latency-sensitive callers that cannot
 * accept cudaMalloc/cudaFree (which may synchronise the whole device).
 *
 * Same operation, layouts and codes as gemm_run, on the CURRENT device, with
 * the plan flags passed directly (`flags`: GEMM_B_KN or GEMM_B_NK; any other
 * bit is GEMM_ERR_INVALID_ARG) and no plan.  It allocates nothing: A and B,
 * when they break the 16-byte TMA rule, are packed into a fixed scratch array
 * of GEMM_NOALLOC_SCRATCH_BYTES (minus 256 bytes for a status word) that the
 * library holds on each device; a call whose packed operands would not fit
 * returns GEMM_ERR_UNSUPPORTED and launches nothing.  C is written in place
 * whatever its alignment, and aligned A and B need no scratch at any size.
 *
 * `dev_status` (device memory, may be NULL): when given, device-side waits
 * that run out of time OR a non-zero bit into it (the caller clears it); when
 * NULL the scratch's own status word is cleared and used, and not reported.
 *
 * The first call on each device sets up that device (it looks up the
 * scratch's device address with cudaGetSymbolAddress and configures the
 * kernels); make that first call before any stream capture.  All calls on a
 * device share the scratch, which keeps the last call's contents: calls whose
 * GPU work overlaps (different streams or threads) race and must be ordered
 * by the caller.  Returns after enqueueing the work on `stream`. */
int gemm_run_noalloc(int64_t M, int64_t N, int64_t K,
                     const void* A, int64_t lda, const void* B, int64_t ldb, const void* bias,
                     void* C, int64_t ldc, int epilogue, int dtype, unsigned flags,
                     int* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_GEMM_H */
