// Fused attention forward: O = softmax(scale * Q K^T) V per (batch, head),
// never materialising the Sq x Sk score matrix -- the online-softmax
// recurrence of CMU 15-418 "DNNs and ML accelerators" notes, section 3.3
// (running max m, running sum l, accumulator rescaled by exp(m_old - m_new)
// whenever the max grows) and the FlashAttention tiling of youngju.dev "GEMM
// to FlashAttention" and the devpress.csdn.net notes, section 4 (Q, K, V in
// blocks that stay on chip).
//
// Design for sm_103a, one CTA per 128 queries of one head:
//   * warp 0: TMA producer -- Q once, K_j and V_j (128 keys each) into a
//     2-stage ring (3-D tensor maps: keys past Sk read as zero);
//   * warp 1: MMA issuer -- S_j = Q K_j^T into one of two TMEM score buffers
//     (so S_{j+1} is computed while the softmax works on S_j), then
//     O += P_j V_j into the TMEM accumulator once P_j is ready;
//   * warps 2..5: softmax, one thread per query row (TMEM lane), so row max
//     and row sum need no shuffles: pass 1 reads the row's 128 scores for the
//     max, pass 2 rereads them, writes P = 2^(s - m) as bf16 / fp16 into a
//     128-byte-swizzled shared-memory tile (the A operand of the PV product)
//     and adds up l; the accumulator row is rescaled in TMEM only when some
//     row of the warp raised its max.  At the end O / l is stored.
// Scores are taken in base 2 (scale * log2 e folded into one factor).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace gb300 {

namespace {

constexpr int kAttnThreads = 192;
constexpr int kBQ = 128;          // queries per CTA (TMEM lanes)
constexpr int kBKey = 128;        // keys per block
constexpr int kBox = 128 * 128;   // one 128-row x 128-byte swizzled box

template <int D>
struct AttnCfg {
    static constexpr int kQBytes = kBQ * D * 2;   // D / 64 boxes
    static constexpr int kKVBytes = kBKey * D * 2;
    static constexpr int kPBytes = kBQ * kBKey * 2;   // two boxes of 64 keys
    static constexpr int kStages = 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kOffP = kOffV + kStages * kKVBytes;
    static constexpr int kOffMisc = kOffP + kPBytes;
    static constexpr int kMiscBytes = 256;
    static constexpr int kSmem = kOffMisc + kMiscBytes + 1024;   // + alignment slack
    // barriers (8 bytes each) in the misc region
    static constexpr int kBarQ = 0, kBarK = 1, kBarV = 3, kBarKVEmpty = 5, kBarSFull = 7, kBarSFree = 9,
                         kBarP = 11, kBarO = 12, kBarDone = 13, kAbort = 14 * 8, kTmemPtr = kAbort + 4;
    static constexpr int kTmemS = 0;      // two score buffers: columns 0..127 and 128..255
    static constexpr int kTmemO = 256;    // accumulator: columns 256 .. 256 + D - 1
    static_assert(kTmemPtr + 4 <= kMiscBytes, "misc layout");
    static_assert(kSmem <= 232448, "shared memory budget");
};

struct AWait {
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

template <typename T> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
    const __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float cvt_out(float v, float*) { return v; }
__device__ __forceinline__ __nv_bfloat16 cvt_out(float v, __nv_bfloat16*) { return __float2bfloat16_rn(v); }
__device__ __forceinline__ __half cvt_out(float v, __half*) { return __float2half_rn(v); }

__device__ __forceinline__ void st_shared_v4u(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// number of 128-key blocks query block q0 .. q0 + 127 looks at
__device__ __forceinline__ int key_blocks(const AttnParams& p, int q0) {
    const int all = (p.Sk + kBKey - 1) / kBKey;
    if (!p.causal) return all;
    const int i_last = min(q0 + kBQ - 1, p.Sq - 1);
    const int j_last = i_last + (p.Sk - p.Sq);   // last visible key of the block's last query
    if (j_last < 0) return 0;
    return min(all, j_last / kBKey + 1);
}

template <int D, typename InT, typename OutT>
__global__ void __launch_bounds__(kAttnThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using Cfg = AttnCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);
    const uint32_t misc = base + Cfg::kOffMisc;
    auto bar = [&](int i) { return misc + 8u * (uint32_t)i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + Cfg::kOffMisc + Cfg::kAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + Cfg::kOffMisc + Cfg::kTmemPtr);

    const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
    const int bh = (int)blockIdx.y;
    const int q0 = (int)blockIdx.x * kBQ;
    const int nkb = key_blocks(p, q0);

    if (threadIdx.x == 0) {
        mbar_init(bar(Cfg::kBarQ), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(Cfg::kBarK + s), 1);
            mbar_init(bar(Cfg::kBarV + s), 1);
            mbar_init(bar(Cfg::kBarKVEmpty + s), 1);
            mbar_init(bar(Cfg::kBarSFull + s), 1);
            mbar_init(bar(Cfg::kBarSFree + s), 4);   // the four softmax warps
        }
        mbar_init(bar(Cfg::kBarP), 4);
        mbar_init(bar(Cfg::kBarO), 1);
        mbar_init(bar(Cfg::kBarDone), 1);
        *abort_flag = 0;
        fence_mbarrier_init_cluster();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(tmem_slot), 512);
        tmem_relinquish<1>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0 && nkb > 0) {
            const AWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_PRODUCER};
            const uint64_t pol_q = l2_policy_evict_normal();
            const uint64_t pol_kv = l2_policy_evict_last();   // read by every query block of the head
            mbar_arrive_expect_tx(bar(Cfg::kBarQ), Cfg::kQBytes);
#pragma unroll
            for (int b = 0; b < D / 64; ++b)
                tma_load_3d(base + Cfg::kOffQ + b * kBox, &tmQ, bar(Cfg::kBarQ), 64 * b, q0, bh, pol_q);
            for (int j = 0; j < nkb; ++j) {
                const int s = j & 1;
                if (!w(bar(Cfg::kBarKVEmpty + s), (((uint32_t)j >> 1) & 1u) ^ 1u)) break;
                mbar_arrive_expect_tx(bar(Cfg::kBarK + s), Cfg::kKVBytes);
#pragma unroll
                for (int b = 0; b < D / 64; ++b)
                    tma_load_3d(base + Cfg::kOffK + s * Cfg::kKVBytes + b * kBox, &tmK, bar(Cfg::kBarK + s), 64 * b,
                                j * kBKey, bh, pol_kv);
                mbar_arrive_expect_tx(bar(Cfg::kBarV + s), Cfg::kKVBytes);
#pragma unroll
                for (int b = 0; b < D / 64; ++b)
                    tma_load_3d(base + Cfg::kOffV + s * Cfg::kKVBytes + b * kBox, &tmV, bar(Cfg::kBarV + s), 64 * b,
                                j * kBKey, bh, pol_kv);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && nkb > 0) {
            const AWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_MMA};
            bool ok = w(bar(Cfg::kBarQ), 0);
            const uint32_t tS = tmem + Cfg::kTmemS, tO = tmem + Cfg::kTmemO;
            for (int j = 0; j <= nkb && ok; ++j) {
                if (j < nkb) {   // S_j = Q K_j^T
                    const int sb = j & 1, s = j & 1;
                    ok = w(bar(Cfg::kBarSFree + sb), (((uint32_t)j >> 1) & 1u) ^ 1u) &&
                         w(bar(Cfg::kBarK + s), ((uint32_t)j >> 1) & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kq = base + Cfg::kOffQ, kk0 = base + Cfg::kOffK + s * Cfg::kKVBytes;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (uint32_t)((kk >> 2) * kBox + (kk & 3) * 32);
                        tc_mma<1>(tS + (uint32_t)sb * 128u, smem_desc_sw128(kq + off, 16, 1024),
                                  smem_desc_sw128(kk0 + off, 16, 1024), p.idesc_s, kk ? 1u : 0u);
                    }
                    tc_commit_1(bar(Cfg::kBarSFull + sb));
                }
                if (j >= 1) {    // O += P_{j-1} V_{j-1}
                    const int jp = j - 1, s = jp & 1;
                    ok = w(bar(Cfg::kBarP), (uint32_t)jp & 1u) && w(bar(Cfg::kBarV + s), ((uint32_t)jp >> 1) & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t pp = base + Cfg::kOffP, vv = base + Cfg::kOffV + s * Cfg::kKVBytes;
#pragma unroll
                    for (int kk = 0; kk < kBKey / 16; ++kk) {
                        const uint32_t aoff = (uint32_t)((kk >> 2) * kBox + (kk & 3) * 32);
                        // V is K x N = keys x D with D contiguous: MN-major, 64-column
                        // chunks one box apart, 16 key rows per step
                        tc_mma<1>(tO, smem_desc_sw128(pp + aoff, 16, 1024),
                                  smem_desc_sw128(vv + (uint32_t)kk * 2048u, kBox, 1024), p.idesc_o,
                                  (jp | kk) ? 1u : 0u);
                    }
                    tc_commit_1(bar(Cfg::kBarO));
                    tc_commit_1(bar(Cfg::kBarKVEmpty + s));
                }
            }
            // every MMA issued has finished before TMEM is released
            tc_commit_1(bar(Cfg::kBarDone));
            const AWait wd{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_MMA};
            wd(bar(Cfg::kBarDone), 0);
        }
    } else {
        // ---- softmax warps: thread = query row r (TMEM lane 32 q + lane)
        const AWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_EPILOGUE};
        const uint32_t q = warp & 3u;
        const int r = 32 * (int)q + (int)lane;
        const int i = q0 + r;                              // query index
        const int lim = p.causal ? i + (p.Sk - p.Sq) : p.Sk - 1;   // last visible key
        const uint32_t lrow = (32u * q) << 16;             // TMEM lane offset of this warp
        const uint32_t prow = base + Cfg::kOffP + (uint32_t)r * 128u;
        float m = -INFINITY, l = 0.0f;
        bool ok = true;
        for (int j = 0; j < nkb && ok; ++j) {
            const int sb = j & 1;
            ok = __all_sync(0xffffffffu, w(bar(Cfg::kBarSFull + sb), ((uint32_t)j >> 1) & 1u));
            if (!ok) break;
            tc_fence_after();
            const uint32_t tS = tmem + lrow + Cfg::kTmemS + (uint32_t)sb * 128u;
            const int k0 = j * kBKey;
            // pass 1: row max of the visible scores (base 2)
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tS + (uint32_t)c * 32u, v);
                tmem_ld_wait();
#pragma unroll
                for (int t = 0; t < 32; ++t)
                    if (k0 + 32 * c + t <= lim) mx = fmaxf(mx, __uint_as_float(v[t]) * p.scale_log2);
            }
            const float m_new = fmaxf(m, mx);
            const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;      // nothing visible yet
            const float alpha = (m == -INFINITY) ? 0.0f : exp2f(m - m_use);
            // P_j goes where P_{j-1} was, and O is rescaled: PV_{j-1} must be done
            if (j >= 1) {
                ok = __all_sync(0xffffffffu, w(bar(Cfg::kBarO), (uint32_t)(j - 1) & 1u));
                if (!ok) break;
                tc_fence_after();
            }
            // pass 2: P = 2^(s - m), row sum, P as 16-bit into the swizzled A tile
            float sum = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tS + (uint32_t)c * 32u, v);
                tmem_ld_wait();
                float e[32];
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const bool vis = k0 + 32 * c + t <= lim;
                    e[t] = vis ? exp2f(__uint_as_float(v[t]) * p.scale_log2 - m_use) : 0.0f;
                    sum += e[t];
                }
                // keys 32 c .. 32 c + 31: box c / 2, 16-byte pieces 4 (c & 1) .. + 3
                const uint32_t box = prow + (uint32_t)(c >> 1) * (uint32_t)kBox;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint32_t piece = (uint32_t)(4 * (c & 1) + t) ^ ((uint32_t)r & 7u);
                    st_shared_v4u(box + (piece << 4), pack2<InT>(e[8 * t], e[8 * t + 1]),
                                  pack2<InT>(e[8 * t + 2], e[8 * t + 3]), pack2<InT>(e[8 * t + 4], e[8 * t + 5]),
                                  pack2<InT>(e[8 * t + 6], e[8 * t + 7]));
                }
            }
            l = l * alpha + sum;
            // the score buffer is free for S_{j+2}
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_local(bar(Cfg::kBarSFree + sb));
            // rescale the accumulator row when the max of some row of the warp grew
            if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.0f)) {
                const uint32_t tO = tmem + lrow + Cfg::kTmemO;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tO + (uint32_t)c * 32u, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * alpha);
                    tmem_st_32x32b_x32(tO + (uint32_t)c * 32u, v);
                }
                tmem_st_wait();
            }
            m = m_new;
            // P_j (generic-proxy stores) and the rescaled O are ready for the MMA
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_local(bar(Cfg::kBarP));
        }
        // ---- O / l, stored by row.  The TMEM loads are warp-collective: the
        // whole warp loads (conditions below are warp-uniform); only the stores
        // depend on the row being a real query.
        if (ok && nkb > 0) {
            ok = __all_sync(0xffffffffu, w(bar(Cfg::kBarO), (uint32_t)(nkb - 1) & 1u));
            if (ok) tc_fence_after();
        }
        const bool store = i < p.Sq;
        OutT* orow = reinterpret_cast<OutT*>(p.O) + ((int64_t)bh * p.Sq + (store ? i : 0)) * D;
        const float inv = (ok && l > 0.0f) ? 1.0f / l : 0.0f;
        const uint32_t tO = tmem + lrow + Cfg::kTmemO;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            if (ok && nkb > 0) {
                tmem_ld_32x32b_x32(tO + (uint32_t)c * 32u, v);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int t = 0; t < 32; ++t) v[t] = 0u;
            }
            if (store) {
                OutT o[32];
#pragma unroll
                for (int t = 0; t < 32; ++t) o[t] = cvt_out(__uint_as_float(v[t]) * inv, (OutT*)nullptr);
                constexpr int kVec = 32 * (int)sizeof(OutT) / 16;
#pragma unroll
                for (int t = 0; t < kVec; ++t)
                    reinterpret_cast<uint4*>(orow + 32 * c)[t] = reinterpret_cast<const uint4*>(o)[t];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<1>(tmem, 512);
    }
}

template <int D, typename InT, typename OutT>
cudaError_t launch_impl(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnParams& p,
                        cudaStream_t stream) {
    dim3 grid((unsigned)((p.Sq + kBQ - 1) / kBQ), (unsigned)p.BH, 1);
    attn_fwd_kernel<D, InT, OutT><<<grid, kAttnThreads, AttnCfg<D>::kSmem, stream>>>(tmQ, tmK, tmV, p);
    return cudaGetLastError();
}

template <int D, typename InT, typename OutT>
cudaError_t prepare_impl() {
    return cudaFuncSetAttribute(attn_fwd_kernel<D, InT, OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                AttnCfg<D>::kSmem);
}

template <int D>
cudaError_t launch_d(int dtype, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                     const AttnParams& p, cudaStream_t stream) {
    switch (dtype) {
        case DT_BF16_F32: return launch_impl<D, __nv_bfloat16, float>(tmQ, tmK, tmV, p, stream);
        case DT_BF16_BF16: return launch_impl<D, __nv_bfloat16, __nv_bfloat16>(tmQ, tmK, tmV, p, stream);
        case DT_F16_F32: return launch_impl<D, __half, float>(tmQ, tmK, tmV, p, stream);
        case DT_F16_F16: return launch_impl<D, __half, __half>(tmQ, tmK, tmV, p, stream);
    }
    return cudaErrorInvalidValue;
}

template <int D>
cudaError_t prepare_d(int dtype) {
    switch (dtype) {
        case DT_BF16_F32: return prepare_impl<D, __nv_bfloat16, float>();
        case DT_BF16_BF16: return prepare_impl<D, __nv_bfloat16, __nv_bfloat16>();
        case DT_F16_F32: return prepare_impl<D, __half, float>();
        case DT_F16_F16: return prepare_impl<D, __half, __half>();
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t attention_prepare(int dtype) {
    cudaError_t e = prepare_d<64>(dtype);
    return e != cudaSuccess ? e : prepare_d<128>(dtype);
}

cudaError_t launch_attention(int dtype, int D, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                             const CUtensorMap& tmV, const AttnParams& p, cudaStream_t stream) {
    if (D == 64) return launch_d<64>(dtype, tmQ, tmK, tmV, p, stream);
    if (D == 128) return launch_d<128>(dtype, tmQ, tmK, tmV, p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gb300
