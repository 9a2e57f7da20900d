// Very-small-M Linear layers that stream the weight without staging it:
//
//   Y[m][n] = epilogue( sum_k X[m][k] * W[n][k] ),   W stored N x K
//
// (a Linear weight, out x in).  Two kernels: the CUDA-core GEMV below (M <= 4,
// chosen for M = 1) and, further down, the warp-MMA kernel (2 <= M <= 16,
// chosen up to M = 8), which keeps the GEMV's loads and replaces its FMAs by
// warp-level tensor-core MMAs.
//
// GEMV.  With M <= 4 every weight byte feeds at most a
// few multiply-adds (arithmetic intensity about M FLOP per byte: youngju.dev
// "GEMM to FlashAttention", arithmetic-intensity listing, batch-1 case; CMU
// 15-418 notes, question 1 on GEMV), so the kernel is bound by streaming W
// from HBM and the tensor cores buy nothing.  The form follows the warp-level
// reduction of the CMU 15-418 notes, section 3.3 (example three): each warp
// owns output rows, its lanes stride the reduction dimension, and a butterfly
// of warp shuffles combines the lanes' partial sums.
//
// Design for sm_103a:
//   * every lane moves 16-byte pieces: lane l of a warp reads pieces
//     l, l + 32, l + 64, ... of a W row, so each warp-wide load covers 512
//     contiguous bytes (coalesced); W is read once, through the non-caching
//     path (ld.global.nc.L1::no_allocate), X through L1, where every warp of
//     the SM finds it;
//   * a warp works on R rows and U pieces per row at a time: R x U
//     independent 16-byte loads per lane are in flight before the first
//     multiply, and each X piece is reused for the R rows;
//   * the rows are split evenly over a grid sized to be resident at once
//     (contiguous row ranges of floor(N / warps) or one more per warp), so
//     every SM streams the same number of bytes;
//   * products and sums in fp32: 16-bit values widened exactly and multiplied
//     with the paired fp32 instruction (fma.rn.f32x2); fp8 codes converted
//     exactly to f16 pairs (cvt e4m3x2 / e5m2x2 -> f16x2) and multiplied into
//     fp32 by the mixed-precision fma.rn.f32.f16, which saves the f16 -> f32
//     widening (the fp8 layer is bound by instruction issue, not bytes: 0.70
//     -> 0.80 of HBM at 4096 -> 14336);
//   * a K tail that does not fill a 16-byte piece is read element by element
//     (nothing past K is touched);
//   * the epilogue (alpha, per-column scale, bias, beta * previous Y, ReLU,
//     the single cast) runs in the lane that holds the finished sum;
//   * programmatic dependent launch: the grid releases its dependents at once;
//     with constant weights (plan flag GEMM_B_CONST) each warp issues its first
//     W loads before waiting for the previous kernel of the stream, whose
//     output may be this layer's X.
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace gb300 {

namespace {

constexpr int kWarps = kGemvThreads / 32;

// W: streamed once, kept out of L1.  Volatile: issued in program order, so
// the prefetched loads stay ahead of the dependency wait.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// X: read by every warp of the SM, cached in L1.
__device__ __forceinline__ uint4 ld_keep16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// The elements k0 .. k0 + kPer - 1 of a row whose valid length is K (k0 < K
// < k0 + kPer), one element at a time, zeros past K.
template <int ES>
__device__ __forceinline__ uint4 ld_tail16(const char* row, int k0, int K) {
    union { uint4 u; uint8_t b[16]; uint16_t h[8]; } v;
    v.u = make_uint4(0u, 0u, 0u, 0u);
    constexpr int kPer = 16 / ES;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
        if (k0 + e < K) {
            if constexpr (ES == 2) v.h[e] = *reinterpret_cast<const uint16_t*>(row + (int64_t)(k0 + e) * 2);
            else v.b[e] = *reinterpret_cast<const uint8_t*>(row + (k0 + e));
        }
    }
    return v.u;
}

// ---- operand kinds: 16-byte piece -> pairs of fp32 values (exact) ----
// OP 0: bf16, 1: fp16, 2: e4m3, 3: e5m2.  kPairs pairs per piece.
template <int OP> struct Op;
template <> struct Op<0> {
    static constexpr int kEs = 2, kPairs = 4;
    static constexpr bool kMixed = false;
    static __device__ __forceinline__ uint64_t pair(const uint4& v, int j) {
        const uint32_t u = j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
        return f2_pack(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
    }
};
template <> struct Op<1> {
    static constexpr int kEs = 2, kPairs = 4;
    static constexpr bool kMixed = false;
    static __device__ __forceinline__ uint64_t pair(const uint4& v, int j) {
        const uint32_t u = j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
        __half2 h = *reinterpret_cast<const __half2*>(&u);
        const float2 f = __half22float2(h);
        return f2_pack(f.x, f.y);
    }
};
template <int E5M2> struct OpFp8 {
    static constexpr int kEs = 1, kPairs = 8;
    static constexpr bool kMixed = true;
    // codes 2j, 2j + 1 of the piece -> f16x2 (exact)
    static __device__ __forceinline__ uint32_t h2(const uint4& v, int j) {
        const uint32_t u = (j >> 1) == 0 ? v.x : (j >> 1) == 1 ? v.y : (j >> 1) == 2 ? v.z : v.w;
        const uint16_t c = (uint16_t)((j & 1) ? (u >> 16) : (u & 0xFFFFu));
        uint32_t r;
        if constexpr (E5M2) asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(r) : "h"(c));
        else asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(c));
        return r;
    }
};
template <> struct Op<2> : OpFp8<0> {};
template <> struct Op<3> : OpFp8<1> {};

// (lo, hi) += (a.lo * b.lo, a.hi * b.hi) for f16x2 a, b and an fp32 pair
__device__ __forceinline__ uint64_t f2_fma_h2(uint32_t a, uint32_t b, uint64_t c) {
    float lo, hi;
    f2_unpack(c, lo, hi);
    asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %1, ah, bh, %1;\n\t}"
        : "+f"(lo), "+f"(hi) : "r"(a), "r"(b));
    return f2_pack(lo, hi);
}

template <typename T> __device__ __forceinline__ float vec_f32(T v);
template <> __device__ __forceinline__ float vec_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <> __device__ __forceinline__ float vec_f32<__half>(__half v) { return __half2float(v); }
__device__ __forceinline__ float y_f32(float v) { return v; }
__device__ __forceinline__ float y_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float y_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float y_cvt(float v, float*) { return v; }
__device__ __forceinline__ __nv_bfloat16 y_cvt(float v, __nv_bfloat16*) { return __float2bfloat16_rn(v); }
__device__ __forceinline__ __half y_cvt(float v, __half*) { return __float2half_rn(v); }

// MT: tokens held (M <= MT); R rows x U pieces per lane in flight; OP operand
// kind; VecT type of bias / scale; OutT type of Y.
template <int MT, int R, int U, int OP, typename VecT, typename OutT>
__global__ void __launch_bounds__(kGemvThreads)
gemv_kernel(const GemvParams p) {
    using O = Op<OP>;
    constexpr int kPer = 16 / O::kEs;          // elements per 16-byte piece
    constexpr int kBlk = 32 * U * kPer;        // elements of a row per block of pieces
    const int warp = (int)(threadIdx.x >> 5), lane = (int)(threadIdx.x & 31u);
    const int64_t TW = (int64_t)gridDim.x * kWarps;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + warp;
    const int r_begin = (int)(gw * p.N / TW), r_end = (int)((gw + 1) * p.N / TW);
    const int M = p.M, K = p.K;
    const char* const W = static_cast<const char*>(p.W);
    const char* const X = static_cast<const char*>(p.X);

    grid_launch_dependents();
    bool waited = false;
    if (!p.w_prefetch || r_begin >= r_end) {
        grid_dependency_wait();
        waited = true;
    }

    for (int n0 = r_begin; n0 < r_end; n0 += R) {
        const int nr = min(R, r_end - n0);     // warp-uniform
        uint64_t acc[R][MT];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[r][m] = 0ull;
        for (int kb = 0; kb < K; kb += kBlk) {
            const bool full = kb + kBlk <= K;  // warp-uniform
            uint4 w[R][U];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const char* row = W + (int64_t)(n0 + r) * p.ldw * O::kEs;
#pragma unroll
                for (int i = 0; i < U; ++i) {
                    const int k = kb + (i * 32 + lane) * kPer;
                    if (r >= nr) w[r][i] = make_uint4(0u, 0u, 0u, 0u);
                    else if (full || k + kPer <= K) w[r][i] = ld_stream16(row + (int64_t)k * O::kEs);
                    else if (k < K) w[r][i] = ld_tail16<O::kEs>(row, k, K);
                    else w[r][i] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            if (!waited) {                     // W loads are in flight during the wait
                grid_dependency_wait();
                waited = true;
            }
            uint4 x[MT][U];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const char* row = X + (int64_t)m * p.ldx * O::kEs;
#pragma unroll
                for (int i = 0; i < U; ++i) {
                    const int k = kb + (i * 32 + lane) * kPer;
                    if (m >= M) x[m][i] = make_uint4(0u, 0u, 0u, 0u);
                    else if (full || k + kPer <= K) x[m][i] = ld_keep16(row + (int64_t)k * O::kEs);
                    else if (k < K) x[m][i] = ld_tail16<O::kEs>(row, k, K);
                    else x[m][i] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            if constexpr (O::kMixed) {
                // f16 pairs multiplied and added into fp32 by the mixed-precision
                // fma (exact products of the f16 values, one rounding each)
#pragma unroll
                for (int i = 0; i < U; ++i) {
#pragma unroll
                    for (int j = 0; j < O::kPairs; ++j) {
                        uint32_t xh[MT];
#pragma unroll
                        for (int m = 0; m < MT; ++m) xh[m] = O::h2(x[m][i], j);
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t wh = O::h2(w[r][i], j);
#pragma unroll
                            for (int m = 0; m < MT; ++m) acc[r][m] = f2_fma_h2(wh, xh[m], acc[r][m]);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < U; ++i) {
#pragma unroll
                    for (int j = 0; j < O::kPairs; ++j) {
                        uint64_t xp[MT];
#pragma unroll
                        for (int m = 0; m < MT; ++m) xp[m] = O::pair(x[m][i], j);
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint64_t wp = O::pair(w[r][i], j);
#pragma unroll
                            for (int m = 0; m < MT; ++m) acc[r][m] = f2_fma(wp, xp[m], acc[r][m]);
                        }
                    }
                }
            }
        }
        // butterfly: every lane ends with every (row, token) sum; lane
        // r * MT + m keeps sum (r, m) for the epilogue
        float mine = 0.0f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float lo, hi;
                f2_unpack(acc[r][m], lo, hi);
                float v = lo + hi;
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
                if (lane == r * MT + m) mine = v;
            }
        }
        const int r = lane / MT, m = lane - (lane / MT) * MT;
        if (lane < R * MT && r < nr && m < M) {
            const int n = n0 + r;
            float t = mine;
            if (p.epi & EPI_ALPHA) t *= p.ex.alpha;
            if (p.epi & EPI_SCALE) t *= vec_f32<VecT>(reinterpret_cast<const VecT*>(p.ex.scale)[n]);
            if (p.epi & EPI_BIAS) t += vec_f32<VecT>(reinterpret_cast<const VecT*>(p.bias)[n]);
            if (p.epi & EPI_BETA)
                t += p.ex.beta * y_f32(reinterpret_cast<const OutT*>(p.ex.c_old)[(int64_t)m * p.ex.ldc_old + n]);
            if (p.epi & EPI_RELU) t = fmaxf(t, 0.0f);
            reinterpret_cast<OutT*>(p.Y)[(int64_t)m * p.ldy + n] = y_cvt(t, (OutT*)nullptr);
        }
    }
}

// Pieces in flight per lane: MT = 1: 2 rows x 8 pieces; MT = 2: 2 x 4;
// MT = 4: 4 x 2 (each X piece serves four rows).
template <int MT> struct Shape;
template <> struct Shape<1> { static constexpr int R = 2, U = 8; };
template <> struct Shape<2> { static constexpr int R = 2, U = 4; };
template <> struct Shape<4> { static constexpr int R = 4, U = 2; };

// Kernel of (tokens held, operand type); nullptr if there is none.
using GemvFn = void (*)(const GemvParams);

template <int MT>
GemvFn kernel_for(int dtype) {
    constexpr int R = Shape<MT>::R, U = Shape<MT>::U;
    switch (dtype) {
        case DT_BF16_F32: return gemv_kernel<MT, R, U, 0, __nv_bfloat16, float>;
        case DT_BF16_BF16: return gemv_kernel<MT, R, U, 0, __nv_bfloat16, __nv_bfloat16>;
        case DT_F16_F32: return gemv_kernel<MT, R, U, 1, __half, float>;
        case DT_F16_F16: return gemv_kernel<MT, R, U, 1, __half, __half>;
        // fp8 codes; bf16 bias / scale
        case DT_E4M3_F32: return gemv_kernel<MT, R, U, 2, __nv_bfloat16, float>;
        case DT_E4M3_BF16: return gemv_kernel<MT, R, U, 2, __nv_bfloat16, __nv_bfloat16>;
        case DT_E5M2_F32: return gemv_kernel<MT, R, U, 3, __nv_bfloat16, float>;
        case DT_E5M2_BF16: return gemv_kernel<MT, R, U, 3, __nv_bfloat16, __nv_bfloat16>;
    }
    return nullptr;
}

GemvFn kernel_for(int mt, int dtype) {
    switch (mt) {
        case 1: return kernel_for<1>(dtype);
        case 2: return kernel_for<2>(dtype);
        case 4: return kernel_for<4>(dtype);
    }
    return nullptr;
}

// ---- 2 <= M <= 16: weight streaming with warp-level tensor-core MMAs ----
//
// With a few tokens every weight element still feeds only M multiply-adds, so
// the layer is bound by streaming W; beyond a couple of tokens the CUDA
// cores' FMA rate no longer keeps up with HBM, but one warp-level mma.sync
// m16n8k16 (16 weight rows x 8 tokens x 16 k) does 2048 of them.  The kernel
// keeps the GEMV's structure -- plain 16-byte loads straight into registers,
// no staging, no cluster, nothing to set up -- which is what a layer that
// streams for a few microseconds needs; the CTA-level tensor-core kernel
// spends ~6 us per launch on its pipeline fill, split-K reduction and set-up.
// Measured on GB300 at 4096 -> 14336: 0.90 of HBM for M = 2 and 4 (the
// tensor-core small-M kernel 0.78); with 9 to 16 tokens the second MMA per
// k-step makes it bound by the warp-level MMA rate (M = 16: 31 against 23
// us), so the dispatcher takes it up to M = 8.
//
// A warp owns 16 rows of W (rows g and g + 8 for lane group g = lane / 4) and
// a k-slice; lane q = lane % 4 of a group reads the 16-byte pieces at
// k = k0 + 8 q of its two rows and of tokens g and g + 8 of X.  A sum over k
// does not depend on the order of its terms, so these eight k-values of a
// lane are handed to two MMAs as their k-slots 2q, 2q + 1 (first two values)
// and 2q + 8, 2q + 9 (next two), and so on, identically for W and X: every
// slot of an MMA pairs W and X at the same k.  The warps of a CTA split K
// (KS ways) and add their fp32 tiles through shared memory in a fixed order.
__device__ __forceinline__ uint32_t u4_at(const uint4& v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// One warp-level MMA, 16 weight rows x 8 tokens: m16n8k16 for 16-bit
// operands (OPK 0 bf16, 1 fp16), m16n8k32 for fp8 codes (OPK 2 e4m3, 3 e5m2).
// Per lane, a0 / a2 hold row g and a1 / a3 row g + 8 at the lane's first and
// second k-slot group, b0 / b1 the same k-slot groups of token g.
template <int OPK>
__device__ __forceinline__ void mma_warp(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
#define GB300_MMA(SHAPE_TYPES)                                                                              \
    asm volatile("mma.sync.aligned." SHAPE_TYPES " {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};" \
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])                                            \
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1))
    if constexpr (OPK == 0) GB300_MMA("m16n8k16.row.col.f32.bf16.bf16.f32");
    else if constexpr (OPK == 1) GB300_MMA("m16n8k16.row.col.f32.f16.f16.f32");
    else if constexpr (OPK == 2) GB300_MMA("m16n8k32.row.col.f32.e4m3.e4m3.f32");
    else GB300_MMA("m16n8k32.row.col.f32.e5m2.e5m2.f32");
#undef GB300_MMA
}

// NH: groups of 8 tokens held (1: M <= 8, 2: M <= 16); U: chunks per lane in
// flight (a chunk is 4 pieces of 16 bytes across a lane group: 32 k of 16-bit
// or 64 k of fp8 values); KS: warps sharing a row group (k-slices), RG = 8 / KS
// row groups per CTA; OPK: operand kind as in mma_warp; VecT: type of the bias
// and scale vectors.
template <int NH, int U, int KS, int OPK, typename VecT, typename OutT>
__global__ void __launch_bounds__(kGemvThreads)
gemv_mma_kernel(const GemvParams p) {
    constexpr int RG = kWarps / KS;
    constexpr int ES = OPK >= 2 ? 1 : 2;       // bytes per element
    constexpr int kPer = 16 / ES;              // k-values per 16-byte piece
    constexpr int kChunk = 4 * kPer;           // k-values per chunk (a lane group's four pieces)
    __shared__ float red[kWarps][16 * 16];     // [warp][row * 16 + token]
    const int warp = (int)(threadIdx.x >> 5), lane = (int)(threadIdx.x & 31u);
    const int g = lane >> 2, q = lane & 3;
    const int rgl = warp / KS, ks = warp - (warp / KS) * KS;
    const int M = p.M, N = p.N, K = p.K;
    const int G = (N + 15) / 16;
    const int kc = ((K + KS - 1) / KS + kChunk - 1) / kChunk * kChunk;   // k per slice
    const int kb = ks * kc, ke = min(K, kb + kc);
    const char* const W = static_cast<const char*>(p.W);
    const char* const X = static_cast<const char*>(p.X);
    const int64_t ldw = p.ldw * ES, ldx = p.ldx * ES;
    // tokens g, g + 8 of X (zeros past M)
    const bool x0ok = g < M, x1ok = NH == 2 && g + 8 < M;
    const char* const x0row = X + (int64_t)g * ldx;
    const char* const x1row = X + (int64_t)(g + 8) * ldx;

    grid_launch_dependents();
    bool waited = false;
    if (!p.w_prefetch) {
        grid_dependency_wait();
        waited = true;
    }
    // one 16-byte piece of a row at element k, zeros where [k, k + kPer) leaves [kb, ke)
    auto piece = [&](const char* row, bool ok, int k, bool stream) -> uint4 {
        if (!ok || k >= ke) return make_uint4(0u, 0u, 0u, 0u);
        if (k + kPer <= ke) return stream ? ld_stream16(row + (int64_t)k * ES) : ld_keep16(row + (int64_t)k * ES);
        return ld_tail16<ES>(row, k, ke);
    };
    for (int blk = blockIdx.x; blk * RG < G; blk += gridDim.x) {
        const int grp = blk * RG + rgl;
        const int n0 = grp * 16;
        float acc[NH][4];
#pragma unroll
        for (int h = 0; h < NH; ++h) acc[h][0] = acc[h][1] = acc[h][2] = acc[h][3] = 0.0f;
        if (grp < G) {                          // warp-uniform
            const bool w0ok = n0 + g < N, w1ok = n0 + g + 8 < N;
            const char* const w0row = W + (int64_t)(n0 + g) * ldw;
            const char* const w1row = W + (int64_t)(n0 + g + 8) * ldw;
            for (int k0 = kb; k0 < ke; k0 += kChunk * U) {
                uint4 wa[U], wb[U], xa[U], xb[U];
#pragma unroll
                for (int i = 0; i < U; ++i) {
                    const int k = k0 + kChunk * i + kPer * q;
                    wa[i] = piece(w0row, w0ok, k, true);
                    wb[i] = piece(w1row, w1ok, k, true);
                }
                if (!waited) {                  // the first W loads are in flight during the wait
                    grid_dependency_wait();
                    waited = true;
                }
#pragma unroll
                for (int i = 0; i < U; ++i) {
                    const int k = k0 + kChunk * i + kPer * q;
                    xa[i] = piece(x0row, x0ok, k, false);
                    xb[i] = NH == 2 ? piece(x1row, x1ok, k, false) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int i = 0; i < U; ++i) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {   // words 2h, 2h + 1 of the lane's piece
                        const uint32_t a0 = u4_at(wa[i], 2 * h), a2 = u4_at(wa[i], 2 * h + 1);
                        const uint32_t a1 = u4_at(wb[i], 2 * h), a3 = u4_at(wb[i], 2 * h + 1);
                        mma_warp<OPK>(acc[0], a0, a1, a2, a3, u4_at(xa[i], 2 * h), u4_at(xa[i], 2 * h + 1));
                        if constexpr (NH == 2)
                            mma_warp<OPK>(acc[1], a0, a1, a2, a3, u4_at(xb[i], 2 * h), u4_at(xb[i], 2 * h + 1));
                    }
                }
            }
        }
        if (!waited) {                          // a CTA whose warps had no rows
            grid_dependency_wait();
            waited = true;
        }
        // fragment -> [row][token]: c0, c1 row g, tokens 2q, 2q + 1 (+ 8 h); c2, c3 row g + 8
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = 8 * h + 2 * q;
            const float* c = acc[h < NH ? h : 0];
            const bool live = h < NH;
            red[warp][g * 16 + t] = live ? c[0] : 0.0f;
            red[warp][g * 16 + t + 1] = live ? c[1] : 0.0f;
            red[warp][(g + 8) * 16 + t] = live ? c[2] : 0.0f;
            red[warp][(g + 8) * 16 + t + 1] = live ? c[3] : 0.0f;
        }
        __syncthreads();
        // thread i: output (row i % 16, token i / 16) of each row group of the CTA,
        // its k-slices added in slice order, then the epilogue
        const int row = (int)(threadIdx.x & 15u), tok = (int)(threadIdx.x >> 4);
        for (int r = 0; r < RG; ++r) {
            const int n = (blk * RG + r) * 16 + row;
            if (n < N && tok < M) {
                float t = 0.0f;
#pragma unroll
                for (int j = 0; j < KS; ++j) t += red[r * KS + j][row * 16 + tok];
                if (p.epi & EPI_ALPHA) t *= p.ex.alpha;
                if (p.epi & EPI_SCALE) t *= vec_f32<VecT>(reinterpret_cast<const VecT*>(p.ex.scale)[n]);
                if (p.epi & EPI_BIAS) t += vec_f32<VecT>(reinterpret_cast<const VecT*>(p.bias)[n]);
                if (p.epi & EPI_BETA)
                    t += p.ex.beta * y_f32(reinterpret_cast<const OutT*>(p.ex.c_old)[(int64_t)tok * p.ex.ldc_old + n]);
                if (p.epi & EPI_RELU) t = fmaxf(t, 0.0f);
                reinterpret_cast<OutT*>(p.Y)[(int64_t)tok * p.ldy + n] = y_cvt(t, (OutT*)nullptr);
            }
        }
        __syncthreads();
    }
}

template <int NH, int KS, int U>
GemvFn mma_kernel_for(int dtype) {
    switch (dtype) {
        case DT_BF16_F32: return gemv_mma_kernel<NH, U, KS, 0, __nv_bfloat16, float>;
        case DT_BF16_BF16: return gemv_mma_kernel<NH, U, KS, 0, __nv_bfloat16, __nv_bfloat16>;
        case DT_F16_F32: return gemv_mma_kernel<NH, U, KS, 1, __half, float>;
        case DT_F16_F16: return gemv_mma_kernel<NH, U, KS, 1, __half, __half>;
        // fp8 codes; bf16 bias / scale
        case DT_E4M3_F32: return gemv_mma_kernel<NH, U, KS, 2, __nv_bfloat16, float>;
        case DT_E4M3_BF16: return gemv_mma_kernel<NH, U, KS, 2, __nv_bfloat16, __nv_bfloat16>;
        case DT_E5M2_F32: return gemv_mma_kernel<NH, U, KS, 3, __nv_bfloat16, float>;
        case DT_E5M2_BF16: return gemv_mma_kernel<NH, U, KS, 3, __nv_bfloat16, __nv_bfloat16>;
    }
    return nullptr;
}

// u: chunks per lane in flight, 4, or 8 for one group of tokens and k split 8 ways
GemvFn mma_kernel_for(int nh, int ks, int dtype, int u = 4) {
#define GB300_KS(NHV) \
    switch (ks) { \
        case 1: return mma_kernel_for<NHV, 1, 4>(dtype); \
        case 2: return mma_kernel_for<NHV, 2, 4>(dtype); \
        case 4: return mma_kernel_for<NHV, 4, 4>(dtype); \
        case 8: return mma_kernel_for<NHV, 8, 4>(dtype); \
    }
    if (nh == 1 && ks == 8 && u == 8) return mma_kernel_for<1, 8, 8>(dtype);
    if (u != 4) return nullptr;
    if (nh == 1) { GB300_KS(1) } else if (nh == 2) { GB300_KS(2) }
#undef GB300_KS
    return nullptr;
}

// Co-resident CTAs per SM of the 8-chunk variant, per device and operand type
// (looked up once; 0 = not yet).
int g_wide_blocks[16][8];

}  // namespace

int gemv_tokens_held(int M) { return M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 0)); }

cudaError_t gemv_prepare(int M, int dtype, int* blocks_per_sm) {
    GemvFn fn = kernel_for(gemv_tokens_held(M), dtype);
    if (fn == nullptr) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, kGemvThreads, 0);
}

cudaError_t launch_gemv(int dtype, const GemvParams& p, int grid, cudaStream_t stream) {
    GemvFn fn = kernel_for(gemv_tokens_held(p.M), dtype);
    if (fn == nullptr || grid < 1) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

int gemv_mma_groups(int M) { return M <= 8 ? 1 : (M <= 16 ? 2 : 0); }

cudaError_t gemv_mma_prepare(int nh, int ks, int dtype, int* blocks_per_sm) {
    GemvFn fn = mma_kernel_for(nh, ks, dtype);
    if (fn == nullptr) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, kGemvThreads, 0);
}

cudaError_t launch_gemv_mma(int dtype, int ks, const GemvParams& p, int grid, cudaStream_t stream) {
    const int nh = gemv_mma_groups(p.M);
    GemvFn fn = mma_kernel_for(nh, ks, dtype);
    if (fn == nullptr || grid < 1) return cudaErrorInvalidValue;
    // A layer with no more 16-row groups than the grid has CTAs (every CTA one
    // group, k split over its 8 warps) runs in a single wave; if the variant
    // with 8 chunks in flight per lane (more registers, fewer CTAs per SM)
    // still fits that wave, it hides more load latency: 4096 -> 4096 at M = 4
    // 6.7 against 8.1 us.  Larger layers need several waves, where the 4-chunk
    // variant's extra CTAs per SM keep the waves balanced (4096 -> 14336: 19.3
    // against 24 us for the 8-chunk variant).
    if (nh == 1 && ks == kWarps && (int64_t)grid * 16 >= p.N && dtype >= 0 && dtype < 8) {
        int dev = 0, sms = 0;
        bool ok = cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 16 &&
                  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
        if (ok) {
            GemvFn wide = mma_kernel_for(1, kWarps, dtype, 8);
            int& bps = g_wide_blocks[dev][dtype];
            if (bps == 0 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, wide, kGemvThreads, 0) != cudaSuccess) {
                bps = -1;
                ok = false;
            }
            if (bps > 0 && grid <= sms * bps) fn = wide;
        }
        if (!ok) cudaGetLastError();   // a failed query only means the 4-chunk variant runs
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace gb300
