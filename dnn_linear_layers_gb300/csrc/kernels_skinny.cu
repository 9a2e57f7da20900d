// Skinny-M Linear layer (decode-like): Y[M x N] = X[M x K] . W^T (+bias) (ReLU)
// for M <= 128, where the product is bound by streaming the weight W from HBM
// (arithmetic intensity about M FLOP per byte: youngju.dev "GEMM to
// FlashAttention", arithmetic-intensity listing, batch-1 case; CMU 15-418
// notes, question 1 on GEMV; BLAS level 2 is memory-bound).
//
// Design for sm_103a:
//   * roles swapped: the weight is the 128-row MMA operand (128 output
//     features per CTA) and the M tokens, padded to a multiple of 16, are the
//     MMA's N dimension, so the tensor core consumes W straight from a TMA ring
//     and the accumulator holds D^T[n][m] in TMEM (lane = feature, column = token);
//   * split-K across a thread-block cluster of S CTAs (one k-slice each), sized
//     so that every CTA of the grid is resident at once (one wave, equal work):
//     for a bandwidth-bound kernel this keeps every SM streaming W;
//   * the S partial tiles are reduced through distributed shared memory in a
//     fixed order (slice 0, 1, ..., S-1), so results are deterministic and no
//     global workspace is needed: each CTA pushes its partial rows to the CTA
//     that owns them (remote stores, no round trip), and each owner reduces,
//     applies bias / ReLU / cast and stores 128/S of the features, 8 adjacent
//     features (one 16-byte store) per thread and token.  (Measured on GB300:
//     faster than a feature-major layout with 16-byte scattered remote
//     stores, and than passing the partials through L2.)  The lane-wise
//     accumulate-then-combine is the warp-shuffle reduction idea of the CMU
//     15-418 notes, section 3.3, lifted to CTAs.
//   * W may be N x K (a Linear weight, K contiguous) or K x N (N contiguous);
//     the MMA reads either from 128-byte-swizzled shared memory;
//   * fp8 weights and activations (e4m3 / e5m2, N x K W): kind::f8f6f4 MMAs,
//     a k-block is still one 128-byte row per feature, now 128 elements, so the
//     ring and its descriptors are those of the 16-bit kernel with half the
//     weight bytes per output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace gb300 {

namespace {

constexpr int kThreads = 192;
constexpr int kMaxStages = 8;
constexpr int kWStage = 128 * 128;         // 128 features x one 128-byte k-block row, 16 KB
constexpr int kMiscBytes = 2048;          // barriers, then bias and scale staging

__device__ __forceinline__ void cluster_arrive_wait() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// store into the shared memory of a CTA of this cluster (address from mapa)
__device__ __forceinline__ void st_shared_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(addr), "f"(v) : "memory");
}

struct BoundedWait {
    uint64_t budget_ns;
    volatile int* abort;
    int* status;
    int bit;
    __device__ __forceinline__ bool operator()(uint32_t bar, uint32_t parity) const {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        uint32_t n = 0;
        while (true) {
            if (mbar_try_wait(bar, parity)) return true;
            if ((++n & 31u) == 0) {
                if (*abort) return false;
                if (globaltimer_ns() - t0 > budget_ns) {
                    atomicOr(status, bit);
                    *abort = 1;
                    return false;
                }
            }
        }
    }
};

template <typename T> __device__ __forceinline__ float to_float(T v);
template <> __device__ __forceinline__ float to_float<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <> __device__ __forceinline__ float to_float<__half>(__half v) { return __half2float(v); }
template <typename T> __device__ __forceinline__ T from_float(float v);
template <> __device__ __forceinline__ float from_float<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }
template <> __device__ __forceinline__ __half from_float<__half>(float v) { return __float2half_rn(v); }
__device__ __forceinline__ float out_float(float v) { return v; }
__device__ __forceinline__ float out_float(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float out_float(__half v) { return __half2float(v); }

// Grid: num_n_tiles * S CTAs, clusters of S along x.  CTA rank r of a cluster
// owns k-blocks [r*nkb/S, (r+1)*nkb/S) of feature tile blockIdx.x / S.  KIND 0:
// 16-bit operands (64 elements per k-block); KIND 1: fp8 (128 elements); InT is
// the type of the bias and scale vectors.
template <typename InT, typename OutT, int KIND>
__global__ void __launch_bounds__(kThreads, kSkinnyMaxCtasPerSm)
gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const SkinnyParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    const int mpad = p.mpad;                          // 16..128, multiple of 16
    const int kStages = p.stages;                     // 2..kMaxStages
    constexpr int kKb = KIND ? 128 : 64;              // elements per k-block
    const uint32_t x_stage = (uint32_t)mpad * 128u;   // mpad tokens x 64 k x 2 B
    const uint32_t off_x = kStages * kWStage;
    const uint32_t off_misc = off_x + kStages * x_stage;   // multiple of 1024
    const uint32_t misc = base + off_misc;
    auto bar_full = [&](int s) { return misc + 8u * s; };
    auto bar_empty = [&](int s) { return misc + 8u * (kMaxStages + s); };
    const uint32_t bar_acc = misc + 8u * (2 * kMaxStages);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + off_misc + 8 * (2 * kMaxStages + 1));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + off_misc + 8 * (2 * kMaxStages + 1) + 4);
    // receive buffer recv[slice][m][f] (fp32, S x mpad x 128/S x 4 B = mpad x
    // 512 B) reuses the front of the operand ring, which holds at least two
    // stages of 16 KB + mpad x 128 B, hence at least mpad x 512 B for mpad <= 128
    float* red = reinterpret_cast<float*>(base_ptr);
    const uint32_t red_addr = base;
    float* bias_s = reinterpret_cast<float*>(base_ptr + off_misc + 512);    // 128 floats: the tile's bias
    float* scale_s = reinterpret_cast<float*>(base_ptr + off_misc + 1024);  // 128 floats: its scale

    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    const int S = p.splits;
    const uint32_t rank = cluster_ctarank();
    const int tile = (int)(blockIdx.x) / S;
    const int f0 = tile * 128;                        // first feature of this tile
    const int nkb = p.num_k_blocks;
    const int kb_begin = (int)(((int64_t)rank * nkb) / S);
    const int kb_end = (int)(((int64_t)(rank + 1) * nkb) / S);

    if (threadIdx.x == 0) {
        // a stage is full once the producer's W and X bytes have landed
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_empty(s), 1);
        }
        mbar_init(bar_acc, 1);
        *abort_flag = 0;
        fence_mbarrier_init_cluster();
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(tmem_slot), p.tmem_cols);
        tmem_relinquish<1>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Everything above overlaps the previous kernel's tail; no global memory
    // (operands, bias, output) is touched before the stream's earlier work is
    // done -- except W, which the producer may start streaming first when the
    // caller declared it constant.
    const bool producer = warp == 0 && lane == 0;
    if (!producer) grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            const BoundedWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_PRODUCER};
            const uint64_t pol_w = l2_policy_evict_normal();   // streamed once
            const uint64_t pol_x = l2_policy_evict_last();     // read by every CTA
            auto load_w = [&](int s, int k0) {
                const uint32_t sw = base + s * kWStage;
                if (p.w_mn_major) {
                    // K x N weight: 128-byte boxes of kKb features x kKb k-rows
                    // (two for 16-bit operands, one for fp8), side by side
                    for (int c = 0; c < 128 / kKb; ++c)
                        tma_load_2d(sw + c * kKb * 128, &tmW, bar_full(s), f0 + c * kKb, k0, pol_w);
                } else {
                    tma_load_2d(sw, &tmW, bar_full(s), k0, f0, pol_w);
                }
            };
            // first ring of W before the dependency wait (constant weights only);
            // the ring's stages start empty, so no empty-barrier wait is needed
            const int nk = kb_end - kb_begin;
            const int pre = p.w_prefetch ? (nk < kStages ? nk : kStages) : 0;
            const uint32_t tx = kWStage + x_stage;
            for (int it = 0; it < pre; ++it) {
                mbar_arrive_expect_tx(bar_full(it), tx);
                load_w(it, (kb_begin + it) * kKb);
            }
            grid_dependency_wait();
            for (int it = 0; it < pre; ++it)
                tma_load_2d(base + off_x + it * x_stage, &tmX, bar_full(it), (kb_begin + it) * kKb, 0, pol_x);
            int issued = pre;
            for (int it = pre; it < nk; ++it) {
                const int s = it % kStages;
                const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                if (!w(bar_empty(s), ph ^ 1u)) break;
                mbar_arrive_expect_tx(bar_full(s), tx);
                const int k0 = (kb_begin + it) * kKb;
                load_w(s, k0);
                tma_load_2d(base + off_x + s * x_stage, &tmX, bar_full(s), k0, 0, pol_x);
                issued = it + 1;
            }
            // Copies already issued land before the ring is reused for the
            // reduction or released: wait (bounded) for the last phase of each
            // stage (immediately done in a run without abort).
            for (int it = issued - kStages < 0 ? 0 : issued - kStages; it < issued; ++it)
                if (!mbar_wait_bounded(bar_full(it % kStages), (uint32_t)(it / kStages) & 1u, p.timeout_ns))
                    atomicOr(p.status, ST_TIMEOUT_PRODUCER);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const BoundedWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_MMA};
            for (int kb = kb_begin, it = 0; kb < kb_end; ++kb, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                if (!w(bar_full(s), ph)) break;   // barrier wait orders the async-proxy bytes
                const uint32_t sw = base + s * kWStage;
                const uint32_t sx = base + off_x + s * x_stage;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    // MN-major: one MMA takes a quarter of the k-block, kKb / 4 k-rows
                    // of 128 bytes, and the feature boxes lie kKb * 128 bytes apart
                    const uint64_t adesc = p.w_mn_major ? smem_desc_sw128(sw + kk * kKb * 32, kKb * 128, 1024)
                                                        : smem_desc_sw128(sw + kk * 32, 16, 1024);
                    const uint64_t bdesc = smem_desc_sw128(sx + kk * 32, 16, 1024);
                    tc_mma<1, KIND>(tmem, adesc, bdesc, p.idesc, (it | kk) != 0 ? 1u : 0u);
                }
                tc_commit_1(bar_empty(s));
            }
            // signals the epilogue once every MMA above has completed
            tc_commit_1(bar_acc);
        }
    }

    // the epilogue warps, idle until the accumulator is ready, stage the
    // tile's bias in shared memory (a load issued now does not queue behind
    // the weight stream at the end)
    if (warp >= 2) {
        const int et = (int)threadIdx.x - 64;
        float bvl = 0.0f, svl = 1.0f;
        if ((p.epi & EPI_BIAS) && f0 + et < p.N) bvl = to_float<InT>(reinterpret_cast<const InT*>(p.bias)[f0 + et]);
        if ((p.epi & EPI_SCALE) && f0 + et < p.N)
            svl = to_float<InT>(reinterpret_cast<const InT*>(p.ex.scale)[f0 + et]);
        if (p.epi & EPI_ALPHA) svl *= p.ex.alpha;   // alpha * acc * scale: one factor per feature
        bias_s[et] = bvl;
        scale_s[et] = svl;
    }
    // ---- split-K reduction.  Every CTA of the cluster has finished its MMAs
    // once barrier (1) is passed, so all operand rings are free; each CTA then
    // pushes its partial tile, feature by feature, into the ring of the CTA
    // that owns the feature (128/S features per CTA) with remote stores, which
    // need no round trip (a warp writes 32 consecutive features of one token:
    // 128 contiguous bytes).  After barrier (2) each owner adds the S partials
    // from its own shared memory in slice order 0, 1, ..., S-1 (deterministic)
    // and applies bias / ReLU / cast, 8 consecutive features at a time.
    // Receive layout in the owner's ring: recv[slice][token][feature - first
    // owned feature], fp32.
    bool have_acc = true;
    if (warp >= 2) {
        const BoundedWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_EPILOGUE};
        const bool ready = w(bar_acc, 0);
        have_acc = __all_sync(0xffffffffu, ready);
    }
    tc_fence_before();
    __syncwarp();
    cluster_arrive_wait();   // (1) every ring of the cluster is idle
    const int per = 128 / S;                          // features owned by each CTA
    const int mcols = p.M < mpad ? p.M : mpad;        // token columns that matter
    if (warp >= 2) {
        tc_fence_after();
        const uint32_t q = warp & 3u;
        const int f = 32 * (int)q + (int)lane;        // feature row of the tile (TMEM lane)
        const uint32_t owner = (uint32_t)(f / per);
        const int fl = f - (int)owner * per;
        const uint32_t dst = mapa_shared(red_addr, owner) + (uint32_t)(((int)rank * mpad * per + fl) * 4);
        const bool zero = !have_acc || kb_end <= kb_begin;   // warp-uniform
        // 32 token columns per TMEM load (the allocation holds at least
        // round_up(mpad, 32) columns); columns past mcols are not sent
        for (int c = 0; c < mcols; c += 32) {
            uint32_t r[32];
            if (!zero) {
                tmem_ld_32x32b_x32(tmem + ((32u * q) << 16) + (uint32_t)c, r);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = 0u;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (c + j < mcols) st_shared_cluster_f32(dst + (uint32_t)((c + j) * per * 4), __uint_as_float(r[j]));
        }
    }
    tc_fence_before();
    __syncwarp();
    cluster_arrive_wait();   // (2) all partials delivered (release / acquire)
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<1>(tmem, p.tmem_cols);
    }
    {
        // work item = (token m, group of 8 owned features); 192 is a multiple
        // of the group count per token (2, 4, 8 or 16), so a thread keeps one
        // feature group and its bias for all its tokens
        const int groups = per / 8;
        const int t = (int)threadIdx.x;
        const int g = t % groups;
        const int mstep = kThreads / groups;
        const int fl = 8 * g;
        const int n = f0 + (int)rank * per + fl;      // first of the 8 features
        const bool relu = (p.epi & EPI_RELU) != 0;
        const bool full8 = n + 8 <= p.N;
        float bv[8], sv[8];   // staged by the epilogue warps; ordered by the cluster barriers
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            bv[e] = bias_s[(int)rank * per + fl + e];
            sv[e] = scale_s[(int)rank * per + fl + e];
        }
        const bool scaled = (p.epi & (EPI_SCALE | EPI_ALPHA)) != 0;
        const bool beta = (p.epi & EPI_BETA) != 0;
        const bool vec_c = full8 && p.ex.c_old_vec16;
        OutT* const Y = reinterpret_cast<OutT*>(p.Y);
        const bool vec = full8 && (reinterpret_cast<uintptr_t>(Y) % 16 == 0) &&
                         ((p.ldy * (int64_t)sizeof(OutT)) % 16 == 0);
        const int slice = mpad * per;                 // floats per slice
        for (int m = t / groups; m < mcols; m += mstep) {
            const float* src = red + m * per + fl;
            float4 a0 = *reinterpret_cast<const float4*>(src);
            float4 a1 = *reinterpret_cast<const float4*>(src + 4);
            for (int s = 1; s < S; ++s) {
                const float4 v0 = *reinterpret_cast<const float4*>(src + s * slice);
                const float4 v1 = *reinterpret_cast<const float4*>(src + s * slice + 4);
                a0.x += v0.x; a0.y += v0.y; a0.z += v0.z; a0.w += v0.w;
                a1.x += v1.x; a1.y += v1.y; a1.z += v1.z; a1.w += v1.w;
            }
            float o[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            float cv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) cv[e] = 0.0f;
            if (beta) {
                const OutT* crow = reinterpret_cast<const OutT*>(p.ex.c_old) + (int64_t)m * p.ex.ldc_old + n;
                if (vec_c) {
                    OutT c8[8];
                    if (sizeof(OutT) == 2) {
                        *reinterpret_cast<uint4*>(c8) = *reinterpret_cast<const uint4*>(crow);
                    } else {
                        reinterpret_cast<uint4*>(c8)[0] = reinterpret_cast<const uint4*>(crow)[0];
                        reinterpret_cast<uint4*>(c8)[1] = reinterpret_cast<const uint4*>(crow)[1];
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) cv[e] = out_float(c8[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (n + e < p.N) cv[e] = out_float(crow[e]);
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (scaled) o[e] *= sv[e];
                o[e] += bv[e];
                if (beta) o[e] += p.ex.beta * cv[e];
                if (relu) o[e] = fmaxf(o[e], 0.0f);
            }
            OutT* yrow = Y + (int64_t)m * p.ldy + n;
            if (vec) {
                OutT y8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y8[e] = from_float<OutT>(o[e]);
                if (sizeof(OutT) == 2) {
                    *reinterpret_cast<uint4*>(yrow) = *reinterpret_cast<const uint4*>(y8);
                } else {
                    reinterpret_cast<uint4*>(yrow)[0] = reinterpret_cast<const uint4*>(y8)[0];
                    reinterpret_cast<uint4*>(yrow)[1] = reinterpret_cast<const uint4*>(y8)[1];
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (n + e < p.N) yrow[e] = from_float<OutT>(o[e]);
            }
        }
    }
    // No barrier after the reduction: nothing reads or writes another CTA's
    // shared memory past barrier (2).
}

template <typename InT, typename OutT, int KIND = 0>
cudaError_t launch_skinny_impl(const CUtensorMap& tmW, const CUtensorMap& tmX, const SkinnyParams& p, int grid,
                               cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = skinny_smem_bytes(p.mpad, p.stages);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, gemm_skinny_kernel<InT, OutT, KIND>, tmW, tmX, p);
}

template <typename InT, typename OutT, int KIND = 0>
cudaError_t prepare_skinny_impl() {
    const int most = 227 * 1024;   // rings are sized on the host; this is the per-CTA ceiling
    auto fn = gemm_skinny_kernel<InT, OutT, KIND>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

}  // namespace

int skinny_smem_bytes(int mpad, int stages) {
    return stages * (kWStage + mpad * 128) + kMiscBytes + 1024 /*alignment*/;
}


cudaError_t skinny_prepare(int dtype) {
    switch (dtype) {
        case DT_BF16_F32: return prepare_skinny_impl<__nv_bfloat16, float>();
        case DT_BF16_BF16: return prepare_skinny_impl<__nv_bfloat16, __nv_bfloat16>();
        case DT_F16_F32: return prepare_skinny_impl<__half, float>();
        case DT_F16_F16: return prepare_skinny_impl<__half, __half>();
        // fp8 operands (the format is in the instruction descriptor); bf16 bias / scale
        case DT_E4M3_F32:
        case DT_E5M2_F32: return prepare_skinny_impl<__nv_bfloat16, float, 1>();
        case DT_E4M3_BF16:
        case DT_E5M2_BF16: return prepare_skinny_impl<__nv_bfloat16, __nv_bfloat16, 1>();
    }
    return cudaErrorInvalidValue;
}



cudaError_t launch_skinny(int dtype, const CUtensorMap& tmW, const CUtensorMap& tmX, const SkinnyParams& p,
                          int grid, cudaStream_t stream) {
    switch (dtype) {
        case DT_BF16_F32: return launch_skinny_impl<__nv_bfloat16, float>(tmW, tmX, p, grid, stream);
        case DT_BF16_BF16: return launch_skinny_impl<__nv_bfloat16, __nv_bfloat16>(tmW, tmX, p, grid, stream);
        case DT_F16_F32: return launch_skinny_impl<__half, float>(tmW, tmX, p, grid, stream);
        case DT_F16_F16: return launch_skinny_impl<__half, __half>(tmW, tmX, p, grid, stream);
        case DT_E4M3_F32:
        case DT_E5M2_F32: return launch_skinny_impl<__nv_bfloat16, float, 1>(tmW, tmX, p, grid, stream);
        case DT_E4M3_BF16:
        case DT_E5M2_BF16: return launch_skinny_impl<__nv_bfloat16, __nv_bfloat16, 1>(tmW, tmX, p, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gb300
