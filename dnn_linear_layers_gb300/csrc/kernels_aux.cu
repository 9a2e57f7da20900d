// Small memory-bound helper kernels of the GEMM path:
//
//  * fill_epilogue: the K == 0 case, where every output is the epilogue of an
//    empty sum (bias and/or ReLU of zero, then the cast);
//  * copy2d: strided 2-D copy used to pack operands whose base address or row
//    stride breaks the 16-byte rule of TMA into an aligned workspace, and to
//    copy a padded result back out.  Padding rows to an aligned length is the
//    "pad to a multiple of 16" advice of youngju.dev "GEMM to FlashAttention"
//    (PyTorch tips) and the tile/burst alignment remark of the devpress.csdn.net
//    notes, section 3.6;
//  * transpose2: tf32 operands stored MN-major, rewritten K-major into the
//    workspace before the GEMM;
//  * im2col: the explicit-GEMM form of a convolution, each R x S x C
//    neighbourhood flattened into one row (CMU 15-418 notes, section 2.3), used
//    to set up the convolution-as-GEMM workload.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace gb300 {

namespace {

template <typename InT, typename OutT>
__global__ void fill_epilogue_kernel(int64_t M, int64_t N, const InT* bias, uint32_t epi, float beta,
                                     const OutT* c_old, int64_t ldc_old, OutT* C, int64_t ldc) {
    const int64_t total = M * N;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = t / N, j = t - i * N;
        float v = 0.0f;   // alpha * (empty sum) * scale = 0
        if (epi & EPI_BIAS) v += static_cast<float>(bias[j]);
        if (epi & EPI_BETA) v += beta * static_cast<float>(c_old[i * ldc_old + j]);
        if (epi & EPI_RELU) v = fmaxf(v, 0.0f);
        C[i * ldc + j] = static_cast<OutT>(v);
    }
}

template <typename T>
__global__ void copy2d_kernel(const T* __restrict__ src, int64_t ld_src, T* __restrict__ dst, int64_t ld_dst,
                              int64_t rows, int64_t cols) {
    // one CTA per row chunk: threads stride along the row (coalesced on both sides)
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const T* s = src + r * ld_src;
        T* d = dst + r * ld_dst;
        for (int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; c < cols;
             c += (int64_t)gridDim.x * blockDim.x)
            d[c] = s[c];
    }
}

// Vectorised 2-D copy where one side is 16-byte aligned (the plan's packed
// workspace): each thread moves one 16-byte piece of a row.  Packing
// (dst_aligned) gathers the piece from the unaligned source element by element
// and writes it in one store, zero-filling the columns past `cols` up to the
// 16-byte boundary of the padded row; unpacking reads the aligned piece in one
// load and stores only the elements inside `cols`.
template <typename T>
__global__ void copy2d_vec_kernel(const T* __restrict__ src, int64_t ld_src, T* __restrict__ dst, int64_t ld_dst,
                                  int64_t rows, int64_t cols, int dst_aligned) {
    constexpr int V = 16 / sizeof(T);
    const int64_t chunks = (cols + V - 1) / V;
    const int64_t total = rows * chunks;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = t / chunks;
        const int64_t c0 = (t - r * chunks) * V;
        const T* s = src + r * ld_src + c0;
        T* d = dst + r * ld_dst + c0;
        if (dst_aligned) {
            union { uint4 u; T e[V]; } v;
#pragma unroll
            for (int j = 0; j < V; ++j) v.e[j] = (c0 + j < cols) ? s[j] : T(0);
            *reinterpret_cast<uint4*>(d) = v.u;
        } else {
            union { uint4 u; T e[V]; } v;
            v.u = *reinterpret_cast<const uint4*>(s);
#pragma unroll
            for (int j = 0; j < V; ++j)
                if (c0 + j < cols) d[j] = v.e[j];
        }
    }
}

// Packing of up to two operands in one launch (the GEMM's misaligned A and B):
// each thread builds one 16-byte piece of a destination row.  Row bytes
// [16 k, 16 k + 16) of the source start at any address; a piece whose aligned
// 16-byte words lie inside the row is assembled from those two words by a
// funnel shift (two 16-byte loads, one store), the row's first and last
// pieces byte by byte, so nothing outside the row is read.  Bytes past the
// row up to the piece boundary are written as zeros.
__global__ void pack2_kernel(PackJob j0, PackJob j1) {
    // block-stride over the rows of both jobs, threads over a row's pieces
    const int64_t rows = j0.rows + j1.rows;
    for (int64_t rr = blockIdx.x; rr < rows; rr += gridDim.x) {
        const bool first = rr < j0.rows;
        const PackJob& j = first ? j0 : j1;
        const int64_t r = first ? rr : rr - j0.rows;
        const uint8_t* row = j.src + r * j.ld_src_bytes;
        uint8_t* drow = j.dst + r * j.ld_dst_bytes;
        const uint32_t row_sh = (uint32_t)(reinterpret_cast<uintptr_t>(row) & 15u);   // same for every piece
        const uint4* abase = reinterpret_cast<const uint4*>(row - row_sh);
        for (int64_t k = threadIdx.x; k < j.chunks; k += blockDim.x) {
            const int64_t b0 = k * 16;
            uint4 out;
            if (k >= 1 && b0 - (int64_t)row_sh + 32 <= j.row_bytes) {
                const uint4 lo = __ldg(abase + k);
                const uint4 hi = row_sh ? __ldg(abase + k + 1) : lo;
                const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                const uint32_t q = row_sh >> 2, bits = (row_sh & 3u) * 8u;
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t a = q == 0 ? w[i] : q == 1 ? w[i + 1] : q == 2 ? w[i + 2] : w[i + 3];
                    const uint32_t b = q == 0 ? w[i + 1] : q == 1 ? w[i + 2] : q == 2 ? w[i + 3] : w[i + 4];
                    o[i] = __funnelshift_r(a, b, bits);
                }
                out = make_uint4(o[0], o[1], o[2], o[3]);
            } else {
                union { uint4 u; uint8_t b[16]; } v;
                v.u = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (b0 + e < j.row_bytes) v.b[e] = row[b0 + e];
                out = v.u;
            }
            *reinterpret_cast<uint4*>(drow + b0) = out;
        }
    }
}

// Transposition of up to two matrices of 32-bit elements in one launch (tf32
// operands stored MN-major, which the tensor cores read K-major only):
// blockIdx.y picks the job, blocks stride over its 64 x 64 tiles.  Thread
// (ty, tx) of a 16 x 16 block reads 16-byte pieces (4 columns) of rows ty,
// ty + 16, ty + 32, ty + 48 of the tile into shared memory (rows padded to 65
// words: at most two-way bank conflicts either way), then writes 16-byte
// pieces of the destination rows the same way.  Pieces at a ragged edge, or
// in a source whose rows are not 16-byte aligned, go element by element.  Bits
// are copied unchanged.
__global__ void __launch_bounds__(256) transpose2_kernel(TransJob j0, TransJob j1) {
    __shared__ uint32_t tile[64][65];
    const TransJob j = blockIdx.y ? j1 : j0;
    const int64_t tc = (j.cols + 63) / 64;
    const int64_t tiles = ((j.rows + 63) / 64) * tc;
    const int tx = (int)threadIdx.x & 15, ty = (int)threadIdx.x >> 4;
    const bool src_vec = ((reinterpret_cast<uintptr_t>(j.src) & 15u) == 0) && (j.ld_src & 3) == 0;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t r0 = (t / tc) * 64, c0 = (t - (t / tc) * tc) * 64;
        const int64_t c = c0 + 4 * tx;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rr = ty + 16 * i;
            const int64_t r = r0 + rr;
            uint32_t v[4] = {0u, 0u, 0u, 0u};
            if (r < j.rows) {
                const uint32_t* sp = j.src + r * j.ld_src + c;
                if (src_vec && c + 4 <= j.cols) {
                    const uint4 q = __ldg(reinterpret_cast<const uint4*>(sp));
                    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (c + e < j.cols) v[e] = __ldg(sp + e);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) tile[rr][4 * tx + e] = v[e];
        }
        __syncthreads();
        const int64_t r = r0 + 4 * tx;     // destination columns r .. r + 3
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int cc = ty + 16 * i;
            const int64_t dc = c0 + cc;        // destination row
            if (dc < j.cols) {
                uint32_t* dp = j.dst + dc * j.ld_dst + r;
                if (r + 4 <= j.rows) {
                    *reinterpret_cast<uint4*>(dp) =
                        make_uint4(tile[4 * tx][cc], tile[4 * tx + 1][cc], tile[4 * tx + 2][cc], tile[4 * tx + 3][cc]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (r + e < j.rows) dp[e] = tile[4 * tx + e][cc];
                }
            }
        }
        __syncthreads();
    }
}

// im2col for a stride-s, zero-padded R x S convolution on NHWC input: one warp
// per output row (n, oh, ow); the row is R*S segments of C contiguous input
// channels, each copied in 16-byte pieces (or zero-filled outside the image).
template <typename V>
__global__ void im2col_kernel(const uint8_t* __restrict__ x, int64_t Nb, int64_t H, int64_t W, int64_t C,
                              int R, int S, int pad, int stride, int64_t OH, int64_t OW,
                              uint8_t* __restrict__ out, int64_t ld_out_bytes, int elem_bytes) {
    const int64_t rows = Nb * OH * OW;
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t seg_bytes = C * elem_bytes;
    const int64_t vec_per_seg = seg_bytes / (int64_t)sizeof(V);
    for (int64_t row = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); row < rows; row += warps) {
        const int64_t n = row / (OH * OW);
        const int64_t rem = row - n * OH * OW;
        const int64_t oh = rem / OW, ow = rem - (rem / OW) * OW;
        uint8_t* orow = out + row * ld_out_bytes;
        for (int r = 0; r < R; ++r) {
            const int64_t ih = oh * stride + r - pad;
            for (int s = 0; s < S; ++s) {
                const int64_t iw = ow * stride + s - pad;
                V* dst = reinterpret_cast<V*>(orow + (int64_t)(r * S + s) * seg_bytes);
                if (ih < 0 || ih >= H || iw < 0 || iw >= W) {
                    V z;
                    memset(&z, 0, sizeof(V));
                    for (int64_t v = lane; v < vec_per_seg; v += 32) dst[v] = z;
                } else {
                    const V* src = reinterpret_cast<const V*>(x + ((n * H + ih) * W + iw) * seg_bytes);
                    for (int64_t v = lane; v < vec_per_seg; v += 32) dst[v] = src[v];
                }
            }
        }
    }
}

int blocks_for(int64_t work, int threads) {
    int64_t b = (work + threads - 1) / threads;
    if (b > 152 * 32) b = 152 * 32;
    if (b < 1) b = 1;
    return (int)b;
}

}  // namespace

cudaError_t launch_fill_epilogue(int dtype, int64_t M, int64_t N, const void* bias, uint32_t epi,
                                 const EpiArgs& ex, void* C, int64_t ldc, cudaStream_t stream) {
    const int threads = 256;
    const int blocks = blocks_for(M * N, threads);
    switch (dtype) {
        case DT_BF16_F32:
            fill_epilogue_kernel<__nv_bfloat16, float><<<blocks, threads, 0, stream>>>(
                M, N, (const __nv_bfloat16*)bias, epi, ex.beta, (const float*)ex.c_old, ex.ldc_old, (float*)C, ldc);
            break;
        case DT_BF16_BF16:
            fill_epilogue_kernel<__nv_bfloat16, __nv_bfloat16><<<blocks, threads, 0, stream>>>(
                M, N, (const __nv_bfloat16*)bias, epi, ex.beta, (const __nv_bfloat16*)ex.c_old, ex.ldc_old, (__nv_bfloat16*)C, ldc);
            break;
        case DT_F16_F32:
            fill_epilogue_kernel<__half, float><<<blocks, threads, 0, stream>>>(
                M, N, (const __half*)bias, epi, ex.beta, (const float*)ex.c_old, ex.ldc_old, (float*)C, ldc);
            break;
        case DT_E4M3_F32:
        case DT_E5M2_F32:
        case DT_TF32_F32:
            fill_epilogue_kernel<__nv_bfloat16, float><<<blocks, threads, 0, stream>>>(
                M, N, (const __nv_bfloat16*)bias, epi, ex.beta, (const float*)ex.c_old, ex.ldc_old, (float*)C, ldc);
            break;
        case DT_E4M3_BF16:
        case DT_E5M2_BF16:
        case DT_TF32_BF16:
            fill_epilogue_kernel<__nv_bfloat16, __nv_bfloat16><<<blocks, threads, 0, stream>>>(
                M, N, (const __nv_bfloat16*)bias, epi, ex.beta, (const __nv_bfloat16*)ex.c_old, ex.ldc_old,
                (__nv_bfloat16*)C, ldc);
            break;
        case DT_F16_F16:
            fill_epilogue_kernel<__half, __half><<<blocks, threads, 0, stream>>>(
                M, N, (const __half*)bias, epi, ex.beta, (const __half*)ex.c_old, ex.ldc_old, (__half*)C, ldc);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_copy2d(const void* src, int64_t ld_src, void* dst, int64_t ld_dst,
                          int64_t rows, int64_t cols, int elem_bytes, cudaStream_t stream) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t V = 16 / elem_bytes;
    const int64_t padded = (cols + V - 1) / V * V;
    const bool dst_vec = ((reinterpret_cast<uintptr_t>(dst) | (uintptr_t)(ld_dst * elem_bytes)) & 15u) == 0 &&
                         ld_dst >= padded;
    const bool src_vec = ((reinterpret_cast<uintptr_t>(src) | (uintptr_t)(ld_src * elem_bytes)) & 15u) == 0 &&
                         ld_src >= padded;
    if ((elem_bytes == 1 || elem_bytes == 2 || elem_bytes == 4) && (dst_vec || src_vec)) {
        int64_t blocks = (rows * (padded / V) + threads - 1) / threads;
        if (blocks > 152 * 32) blocks = 152 * 32;
        if (elem_bytes == 1)
            copy2d_vec_kernel<uint8_t><<<(int)blocks, threads, 0, stream>>>(
                (const uint8_t*)src, ld_src, (uint8_t*)dst, ld_dst, rows, cols, dst_vec ? 1 : 0);
        else if (elem_bytes == 2)
            copy2d_vec_kernel<uint16_t><<<(int)blocks, threads, 0, stream>>>(
                (const uint16_t*)src, ld_src, (uint16_t*)dst, ld_dst, rows, cols, dst_vec ? 1 : 0);
        else
            copy2d_vec_kernel<uint32_t><<<(int)blocks, threads, 0, stream>>>(
                (const uint32_t*)src, ld_src, (uint32_t*)dst, ld_dst, rows, cols, dst_vec ? 1 : 0);
        return cudaGetLastError();
    }
    int64_t bx = (cols + threads - 1) / threads;
    if (bx > 64) bx = 64;
    int64_t by = rows < 65535 ? rows : 65535;
    dim3 grid((unsigned)bx, (unsigned)by, 1);
    if (elem_bytes == 1)
        copy2d_kernel<uint8_t><<<grid, threads, 0, stream>>>((const uint8_t*)src, ld_src, (uint8_t*)dst,
                                                             ld_dst, rows, cols);
    else if (elem_bytes == 2)
        copy2d_kernel<uint16_t><<<grid, threads, 0, stream>>>((const uint16_t*)src, ld_src, (uint16_t*)dst,
                                                              ld_dst, rows, cols);
    else if (elem_bytes == 4)
        copy2d_kernel<uint32_t><<<grid, threads, 0, stream>>>((const uint32_t*)src, ld_src, (uint32_t*)dst,
                                                              ld_dst, rows, cols);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_pack2(const PackJob& j0, const PackJob& j1, cudaStream_t stream) {
    const int64_t rows = j0.rows + j1.rows;
    if (rows == 0) return cudaSuccess;
    const int64_t widest = j0.chunks > j1.chunks ? j0.chunks : j1.chunks;
    const int threads = widest >= 256 ? 256 : (int)((widest + 31) / 32 * 32);
    int64_t blocks = rows < 152 * 16 ? rows : 152 * 16;
    pack2_kernel<<<(int)blocks, threads, 0, stream>>>(j0, j1);
    return cudaGetLastError();
}

cudaError_t launch_transpose2(const TransJob& j0, const TransJob& j1, cudaStream_t stream) {
    auto tiles = [](const TransJob& j) { return ((j.rows + 63) / 64) * ((j.cols + 63) / 64); };
    const int64_t t0 = tiles(j0), t1 = tiles(j1);
    const int64_t most = t0 > t1 ? t0 : t1;
    if (most == 0) return cudaSuccess;
    // the destination is written in 16-byte pieces: it must be aligned that way
    if ((reinterpret_cast<uintptr_t>(j0.dst) & 15u) || (j0.ld_dst & 3) ||
        (t1 && ((reinterpret_cast<uintptr_t>(j1.dst) & 15u) || (j1.ld_dst & 3))))
        return cudaErrorInvalidValue;
    const int64_t blocks = most < 152 * 8 ? most : 152 * 8;   // one wave of 8 blocks per SM
    transpose2_kernel<<<dim3((unsigned)blocks, t1 ? 2u : 1u), 256, 0, stream>>>(j0, j1);
    return cudaGetLastError();
}

PackJob pack_job(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows, int64_t cols,
                 int elem_bytes) {
    PackJob j;
    j.src = static_cast<const uint8_t*>(src);
    j.ld_src_bytes = ld_src * elem_bytes;
    j.dst = static_cast<uint8_t*>(dst);
    j.ld_dst_bytes = ld_dst * elem_bytes;
    j.rows = rows;
    j.row_bytes = cols * elem_bytes;
    j.chunks = (j.row_bytes + 15) / 16;
    return j;
}

cudaError_t launch_im2col(const void* x, int64_t Nb, int64_t H, int64_t W, int64_t C, int R, int S, int pad,
                          int stride, void* out, int64_t ld_out, int elem_bytes, cudaStream_t stream) {
    const int64_t OH = (H + 2 * pad - R) / stride + 1, OW = (W + 2 * pad - S) / stride + 1;
    const int64_t rows = Nb * OH * OW;
    if (rows <= 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (rows + 7) / 8;
    if (blocks > 152 * 16) blocks = 152 * 16;
    const int64_t seg = C * elem_bytes;
    const uintptr_t al = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out) |
                         (uintptr_t)(ld_out * elem_bytes) | (uintptr_t)seg;
    if ((al & 15u) == 0)
        im2col_kernel<uint4><<<(int)blocks, threads, 0, stream>>>((const uint8_t*)x, Nb, H, W, C, R, S, pad, stride,
                                                                 OH, OW, (uint8_t*)out, ld_out * elem_bytes, elem_bytes);
    else if ((al & 1u) == 0)
        im2col_kernel<uint16_t><<<(int)blocks, threads, 0, stream>>>((const uint8_t*)x, Nb, H, W, C, R, S, pad,
                                                                    stride, OH, OW, (uint8_t*)out,
                                                                    ld_out * elem_bytes, elem_bytes);
    else
        im2col_kernel<uint8_t><<<(int)blocks, threads, 0, stream>>>((const uint8_t*)x, Nb, H, W, C, R, S, pad,
                                                                   stride, OH, OW, (uint8_t*)out,
                                                                   ld_out * elem_bytes, elem_bytes);
    return cudaGetLastError();
}

}  // namespace gb300
