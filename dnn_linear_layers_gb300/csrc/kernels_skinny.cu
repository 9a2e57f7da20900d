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
//     global workspace is needed; each CTA of the cluster reduces, applies
//     bias / ReLU / cast and stores 128/S of the features.  The lane-wise
//     accumulate-then-combine is the warp-shuffle reduction idea of the CMU
//     15-418 notes, section 3.3, lifted to CTAs.
//   * W may be N x K (a Linear weight, K contiguous) or K x N (N contiguous);
//     the MMA reads either from 128-byte-swizzled shared memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace gb300 {

namespace {

constexpr int kThreads = 192;
constexpr int kStages = 6;
constexpr int kWStage = 128 * 64 * 2;      // 128 features x 64 k, 16 KB

__device__ __forceinline__ void cluster_arrive_wait() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr) : "memory");
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

// Grid: num_n_tiles * S CTAs, clusters of S along x.  CTA rank r of a cluster
// owns k-blocks [r*nkb/S, (r+1)*nkb/S) of feature tile blockIdx.x / S.
template <typename InT, typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const SkinnyParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    const int mpad = p.mpad;                          // 16..128, multiple of 16
    const uint32_t x_stage = (uint32_t)mpad * 128u;   // mpad tokens x 64 k x 2 B
    const uint32_t off_x = kStages * kWStage;
    const uint32_t off_misc = off_x + kStages * x_stage;   // multiple of 1024
    const uint32_t misc = base + off_misc;
    auto bar_full = [&](int s) { return misc + 8u * s; };
    auto bar_empty = [&](int s) { return misc + 8u * (kStages + s); };
    const uint32_t bar_acc = misc + 8u * (2 * kStages);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + off_misc + 8 * (2 * kStages + 1));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + off_misc + 8 * (2 * kStages + 1) + 4);
    // partial tile red[m][f] (fp32, token-major) reuses the front of the W ring
    float* red = reinterpret_cast<float*>(base_ptr);
    const uint32_t red_addr = base;

    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    const int S = p.splits;
    const uint32_t rank = cluster_ctarank();
    const int tile = (int)(blockIdx.x) / S;
    const int f0 = tile * 128;                        // first feature of this tile
    const int nkb = p.num_k_blocks;
    const int kb_begin = (int)(((int64_t)rank * nkb) / S);
    const int kb_end = (int)(((int64_t)(rank + 1) * nkb) / S);

    if (threadIdx.x == 0) {
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

    if (warp == 0) {
        if (lane == 0) {
            const BoundedWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_PRODUCER};
            const uint64_t pol_w = l2_policy_evict_normal();   // streamed once
            const uint64_t pol_x = l2_policy_evict_last();     // read by every CTA
            bool ok = true;
            for (int kb = kb_begin, it = 0; kb < kb_end; ++kb, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                if (!w(bar_empty(s), ph ^ 1u)) { ok = false; break; }
                mbar_arrive_expect_tx(bar_full(s), kWStage + x_stage);
                const uint32_t sw = base + s * kWStage;
                const int k0 = kb * 64;
                if (p.w_mn_major) {
                    tma_load_2d(sw, &tmW, bar_full(s), f0, k0, pol_w);
                    tma_load_2d(sw + 8192, &tmW, bar_full(s), f0 + 64, k0, pol_w);
                } else {
                    tma_load_2d(sw, &tmW, bar_full(s), k0, f0, pol_w);
                }
                tma_load_2d(base + off_x + s * x_stage, &tmX, bar_full(s), k0, 0, pol_x);
            }
            if (!ok) {
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 100000ull) { }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const BoundedWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_MMA};
            for (int kb = kb_begin, it = 0; kb < kb_end; ++kb, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                if (!w(bar_full(s), ph)) break;
                tc_fence_after();
                const uint32_t sw = base + s * kWStage;
                const uint32_t sx = base + off_x + s * x_stage;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t adesc = p.w_mn_major ? smem_desc_sw128(sw + kk * 2048, 8192, 1024)
                                                        : smem_desc_sw128(sw + kk * 32, 16, 1024);
                    const uint64_t bdesc = smem_desc_sw128(sx + kk * 32, 16, 1024);
                    tc_mma_f16<1>(tmem, adesc, bdesc, p.idesc, (it | kk) != 0 ? 1u : 0u);
                }
                tc_commit_1(bar_empty(s));
            }
            // signals the epilogue once every MMA above has completed
            tc_commit_1(bar_acc);
        }
    }

    // ---- partial tile: TMEM -> smem (all MMAs done, ring no longer in use)
    bool have_acc = true;
    if (warp >= 2) {
        const BoundedWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_EPILOGUE};
        const bool ready = w(bar_acc, 0);
        have_acc = __all_sync(0xffffffffu, ready);
        if (have_acc) {
            tc_fence_after();
            const uint32_t q = warp & 3u;
            const int f = 32 * (int)q + (int)lane;          // feature row within the tile
            const bool empty_slice = kb_end <= kb_begin;
            for (int c = 0; c < mpad; c += 16) {
                uint32_t r[16];
                tmem_ld_32x32b_x16(tmem + ((32u * q) << 16) + (uint32_t)c, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    red[(c + j) * 128 + f] = empty_slice ? 0.0f : __uint_as_float(r[j]);
            }
        }
    }
    tc_fence_before();
    __syncwarp();
    cluster_arrive_wait();   // every slice's partial tile is in its shared memory

    // ---- reduction over the cluster in slice order, epilogue, store
    {
        const int per = 128 / S;                    // features reduced by this CTA
        const int fr0 = (int)rank * per;
        const InT* bias = reinterpret_cast<const InT*>(p.bias);
        OutT* Y = reinterpret_cast<OutT*>(p.Y);
        const int total = per * p.M;
        for (int idx = threadIdx.x; idx < total; idx += kThreads) {
            const int m = idx / per;
            const int fl = fr0 + (idx - m * per);
            const int n = f0 + fl;
            const uint32_t off = (uint32_t)((m * 128 + fl) * 4);
            float acc = 0.0f;
            for (int s = 0; s < S; ++s) acc += ld_shared_cluster_f32(mapa_shared(red_addr + off, (uint32_t)s));
            if (n < p.N) {
                if (p.epi & EPI_BIAS) acc += to_float<InT>(bias[n]);
                if (p.epi & EPI_RELU) acc = fmaxf(acc, 0.0f);
                Y[(int64_t)m * p.ldy + n] = from_float<OutT>(acc);
            }
        }
    }
    (void)have_acc;
    __syncwarp();
    cluster_arrive_wait();   // no CTA leaves while a peer may still read its smem
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<1>(tmem, p.tmem_cols);
    }
}

template <typename InT, typename OutT>
cudaError_t launch_skinny_impl(const CUtensorMap& tmW, const CUtensorMap& tmX, const SkinnyParams& p, int grid,
                               cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = skinny_smem_bytes(p.mpad);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_skinny_kernel<InT, OutT>, tmW, tmX, p);
}

template <typename InT, typename OutT>
cudaError_t prepare_skinny_impl() {
    cudaError_t e = cudaFuncSetAttribute(gemm_skinny_kernel<InT, OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         skinny_smem_bytes(128));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gemm_skinny_kernel<InT, OutT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

}  // namespace

int skinny_smem_bytes(int mpad) {
    return kStages * kWStage + kStages * mpad * 128 + 1024 /*misc*/ + 1024 /*alignment*/;
}

cudaError_t skinny_prepare(int dtype) {
    switch (dtype) {
        case DT_BF16_F32: return prepare_skinny_impl<__nv_bfloat16, float>();
        case DT_BF16_BF16: return prepare_skinny_impl<__nv_bfloat16, __nv_bfloat16>();
        case DT_F16_F32: return prepare_skinny_impl<__half, float>();
        case DT_F16_F16: return prepare_skinny_impl<__half, __half>();
    }
    return cudaErrorInvalidValue;
}

cudaError_t skinny_blocks_per_sm(int mpad, int* out) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, gemm_skinny_kernel<__nv_bfloat16, __nv_bfloat16>,
                                                         kThreads, skinny_smem_bytes(mpad));
}

cudaError_t launch_skinny(int dtype, const CUtensorMap& tmW, const CUtensorMap& tmX, const SkinnyParams& p,
                          int grid, cudaStream_t stream) {
    switch (dtype) {
        case DT_BF16_F32: return launch_skinny_impl<__nv_bfloat16, float>(tmW, tmX, p, grid, stream);
        case DT_BF16_BF16: return launch_skinny_impl<__nv_bfloat16, __nv_bfloat16>(tmW, tmX, p, grid, stream);
        case DT_F16_F32: return launch_skinny_impl<__half, float>(tmW, tmX, p, grid, stream);
        case DT_F16_F16: return launch_skinny_impl<__half, __half>(tmW, tmX, p, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gb300
