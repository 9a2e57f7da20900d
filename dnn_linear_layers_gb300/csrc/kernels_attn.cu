// Fused attention forward: O = softmax(scale * Q K^T) V per (batch, head),
// never materialising the Sq x Sk score matrix -- the online-softmax
// recurrence of CMU 15-418 "DNNs and ML accelerators" notes, section 3.3
// (running max m, running sum l, accumulator rescaled by exp(m_old - m_new)
// whenever the max grows) and the FlashAttention tiling of youngju.dev "GEMM
// to FlashAttention" and the devpress.csdn.net notes, section 4 (Q, K, V in
// blocks that stay on chip).
//
// Design for sm_103a, one CTA per 128 queries of one head:
//   * warp 0: TMA producer -- Q once, K_j and V_j (128 keys each) into
//     2-stage rings (3-D tensor maps: keys past Sk read as zero).  K runs one
//     block ahead of V (a K slot frees when its score product is done, a V
//     slot only when its PV product is), so the next K block is on chip before
//     the tensor core wants it;
//   * warps 1 and 2: MMA issuers -- warp 1 S_j = Q K_j^T into one of two TMEM
//     score buffers (S_{j+1} is computed while the softmax works on S_j), warp
//     2 O += P_j V_j into the TMEM accumulator once P_j is ready.  An MMA
//     instruction is accepted only as the tensor pipe drains, so one thread
//     issuing both products would leave the pipe idle while it waited for the
//     other's operands; two threads keep it fed from whichever is ready;
//   * warps 3..10: softmax in two groups of four warps that take the key blocks
//     in turn (group 0 the even ones, group 1 the odd ones), one thread per
//     query row (TMEM lane) in each, so the two warps that share an SM
//     sub-partition work on different blocks and hide each other's latency.
//     A row's reference max passes from group to group once per block through
//     shared memory behind a (bounded) mbarrier; each group keeps a partial
//     row sum until the end.  Each thread reads its 128 scores from TMEM once
//     (the score buffer is handed back at once), P = 2^(s - m) is written
//     as bf16 / fp16 into one of two 128-byte-swizzled shared-memory tiles
//     (the A operand of the PV product; two, so P_j is written while P_{j-1} V
//     runs).  The reference max m of a row moves only when the block max
//     exceeds it by more than 8 (a factor 2^8): O = sum_j 2^(s_j - m) v_j /
//     sum_j 2^(s_j - m) holds for any m, so a stale m changes nothing but the
//     rounding, and the accumulator row is rescaled in TMEM only then.
// Scores are taken in base 2 (scale * log2 e folded into one factor).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace gb300 {

namespace {

constexpr int kAttnThreads = 352;
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
    static constexpr int kOffP = kOffV + kStages * kKVBytes;   // two P tiles
    static constexpr int kOffMisc = kOffP + 2 * kPBytes;
    static constexpr int kOffXch = 256;   // in misc: float hand-off [2 groups][128 rows], sums [2][128]
    static constexpr int kMiscBytes = kOffXch + 2 * 2 * kBQ * 4;
    // the tiles want 1024-byte alignment; a window starting at a multiple of
    // 256 bytes fits (the kernel checks, and stops with a status bit if not)
    static constexpr int kSlack = 768;
    static constexpr int kSmem = kOffMisc + kMiscBytes + kSlack;
    // barriers (8 bytes each) in the misc region; pairs are indexed by buffer
    static constexpr int kBarQ = 0, kBarK = 1, kBarV = 3, kBarKEmpty = 5, kBarVEmpty = 7, kBarSFull = 9,
                         kBarSFree = 11, kBarPFull = 13, kBarODone = 15, kBarDone = 17,
                         kBarHand = 18,  // [4 lane quarters][2 groups]: a group published its max
                         kBarFin = 26,   // [4 lane quarters]: both groups wrote their row sums
                         kAbort = 30 * 8, kTmemPtr = kAbort + 4;
    static constexpr int kTmemS = 0;      // two score buffers: columns 0..127 and 128..255
    static constexpr int kTmemO = 256;    // accumulator: columns 256 .. 256 + D - 1
    static_assert(kTmemPtr + 4 <= kOffXch, "misc layout");
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

// 2^x on the special-function unit (ex2.approx: relative error about 2^-22,
// subnormal results flushed to zero, 2^-inf = +0)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Pairs of fp32 values in one 64-bit register, for the paired fp32
// instructions of sm_100-class SMs (one instruction does two lanes of work).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// max of three (one instruction on sm_100-class SMs)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
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
    if (base - raw > (uint32_t)Cfg::kSlack) {   // same for every thread: nothing started yet
        if (threadIdx.x == 0) atomicOr(p.status, ST_SMEM_LAYOUT);
        return;
    }
    const int bh = (int)blockIdx.y;
    const int q0 = (int)blockIdx.x * kBQ;
    const int nkb = key_blocks(p, q0);

    if (threadIdx.x == 0) {
        mbar_init(bar(Cfg::kBarQ), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(Cfg::kBarK + s), 1);
            mbar_init(bar(Cfg::kBarV + s), 1);
            mbar_init(bar(Cfg::kBarKEmpty + s), 1);
            mbar_init(bar(Cfg::kBarVEmpty + s), 1);
            mbar_init(bar(Cfg::kBarSFull + s), 1);
            mbar_init(bar(Cfg::kBarSFree + s), 4);   // the four warps of the group that owns buffer s
            mbar_init(bar(Cfg::kBarPFull + s), 4);
            mbar_init(bar(Cfg::kBarODone + s), 1);
        }
        for (int x = 0; x < 8; ++x) mbar_init(bar(Cfg::kBarHand + x), 32);   // one warp
        for (int x = 0; x < 4; ++x) mbar_init(bar(Cfg::kBarFin + x), 64);    // both groups' warps of a quarter
        mbar_init(bar(Cfg::kBarDone), 2);   // the two MMA issuers
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
            // block j of K or V: one 128-key box per 64 columns
            auto load_kv = [&](const CUtensorMap* map, int off, int barid, int j) {
                const int s = j & 1;
                mbar_arrive_expect_tx(bar(barid + s), Cfg::kKVBytes);
#pragma unroll
                for (int b = 0; b < D / 64; ++b)
                    tma_load_3d(base + off + s * Cfg::kKVBytes + b * kBox, map, bar(barid + s), 64 * b, j * kBKey, bh,
                                pol_kv);
            };
            // order K_0, K_1, V_0, K_2, V_1, ...: slot j & 1 of K frees when S_{j-2}
            // is done, that of V when P_{j-2} V_{j-2} is
            if (w(bar(Cfg::kBarKEmpty), 1u)) {
                load_kv(&tmK, Cfg::kOffK, Cfg::kBarK, 0);
                for (int j = 0; j < nkb; ++j) {
                    if (j + 1 < nkb) {
                        const int jn = j + 1;
                        if (!w(bar(Cfg::kBarKEmpty + (jn & 1)), (((uint32_t)jn >> 1) & 1u) ^ 1u)) break;
                        load_kv(&tmK, Cfg::kOffK, Cfg::kBarK, jn);
                    }
                    if (!w(bar(Cfg::kBarVEmpty + (j & 1)), (((uint32_t)j >> 1) & 1u) ^ 1u)) break;
                    load_kv(&tmV, Cfg::kOffV, Cfg::kBarV, j);
                }
            }
        }
    } else if (warp == 1) {
        // ---- S issuer: S_j = Q K_j^T into score buffer j & 1
        if (lane == 0 && nkb > 0) {
            const AWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_MMA};
            bool ok = w(bar(Cfg::kBarQ), 0);
            const uint32_t tS = tmem + Cfg::kTmemS;
            for (int j = 0; j < nkb && ok; ++j) {
                const int s = j & 1;
                ok = w(bar(Cfg::kBarSFree + s), (((uint32_t)j >> 1) & 1u) ^ 1u) &&
                     w(bar(Cfg::kBarK + s), ((uint32_t)j >> 1) & 1u);
                if (!ok) break;
                tc_fence_after();
                const uint32_t kq = base + Cfg::kOffQ, kk0 = base + Cfg::kOffK + s * Cfg::kKVBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (uint32_t)((kk >> 2) * kBox + (kk & 3) * 32);
                    tc_mma<1>(tS + (uint32_t)s * 128u, smem_desc_sw128(kq + off, 16, 1024),
                              smem_desc_sw128(kk0 + off, 16, 1024), p.idesc_s, kk ? 1u : 0u);
                }
                tc_commit_1(bar(Cfg::kBarSFull + s));
                tc_commit_1(bar(Cfg::kBarKEmpty + s));
            }
            tc_commit_1(bar(Cfg::kBarDone));
            // every MMA of both issuers has finished before TMEM is released
            const AWait wd{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_MMA};
            wd(bar(Cfg::kBarDone), 0);
        }
    } else if (warp == 2) {
        // ---- PV issuer: O += P_j V_j once the softmax has written P_j
        if (lane == 0 && nkb > 0) {
            const AWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_MMA};
            bool ok = true;
            const uint32_t tO = tmem + Cfg::kTmemO;
            for (int j = 0; j < nkb && ok; ++j) {
                const int s = j & 1;
                ok = w(bar(Cfg::kBarPFull + s), ((uint32_t)j >> 1) & 1u) &&
                     w(bar(Cfg::kBarV + s), ((uint32_t)j >> 1) & 1u);
                if (!ok) break;
                tc_fence_after();
                const uint32_t pp = base + Cfg::kOffP + s * Cfg::kPBytes, vv = base + Cfg::kOffV + s * Cfg::kKVBytes;
#pragma unroll
                for (int kk = 0; kk < kBKey / 16; ++kk) {
                    const uint32_t aoff = (uint32_t)((kk >> 2) * kBox + (kk & 3) * 32);
                    // V is K x N = keys x D with D contiguous: MN-major, 64-column
                    // chunks one box apart, 16 key rows per step
                    tc_mma<1>(tO, smem_desc_sw128(pp + aoff, 16, 1024),
                              smem_desc_sw128(vv + (uint32_t)kk * 2048u, kBox, 1024), p.idesc_o,
                              (j | kk) ? 1u : 0u);
                }
                tc_commit_1(bar(Cfg::kBarODone + s));
                tc_commit_1(bar(Cfg::kBarVEmpty + s));
            }
            tc_commit_1(bar(Cfg::kBarDone));
        }
    } else {
        // ---- softmax warps: thread = query row r (TMEM lane 32 q + lane); group g
        // takes key blocks j = g, g + 2, .. into score buffer and P tile g
        const AWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_EPILOGUE};
        const uint32_t q = warp & 3u;
        const int g = (int)((warp - 3u) >> 2);
        const int r = 32 * (int)q + (int)lane;
        const int i = q0 + r;                              // query index
        const int lim = p.causal ? i + (p.Sk - p.Sq) : p.Sk - 1;   // last visible key
        const uint32_t lrow = (32u * q) << 16;             // TMEM lane offset of this warp
        volatile float* const hand = reinterpret_cast<volatile float*>(base_ptr + Cfg::kOffMisc + Cfg::kOffXch);
        volatile float* const sums = hand + 2 * kBQ;
        const float c2 = p.scale_log2;
        // m: the row's reference max (base 2) as last known here; l: this group's
        // share of the row sum, relative to m
        float m = -INFINITY, l = 0.0f;
        // the factor that moves sums from reference m_old to m_new (1 when equal)
        auto factor = [](float m_old, float m_new) { return m_new == m_old ? 1.0f : ex2_approx(m_old - m_new); };
        bool ok = true;
        for (int j = g; j < nkb && ok; j += 2) {
            const int sb = g;
            const uint32_t ph = ((uint32_t)j >> 1) & 1u;
            ok = __all_sync(0xffffffffu, w(bar(Cfg::kBarSFull + sb), ph));
            if (!ok) break;
            tc_fence_after();
            uint32_t v[4][32];
            const uint32_t tS = tmem + lrow + Cfg::kTmemS + (uint32_t)sb * 128u;
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(tS + (uint32_t)c * 32u, v[c]);
            tmem_ld_wait();
            // the scores are in registers: the buffer is free for S_{j+2}
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_local(bar(Cfg::kBarSFree + sb));
            const int k0 = j * kBKey;
            if (!__all_sync(0xffffffffu, k0 + kBKey - 1 <= lim)) {   // a block on the mask's edge
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        if (k0 + 32 * c + t > lim) v[c][t] = __float_as_uint(-INFINITY);
            }
            // block max of the raw scores, scaled once (the scale is positive)
            float mp[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) mp[t] = __uint_as_float(v[0][t]);
#pragma unroll
            for (int x = 8; x < 128; x += 16)
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    mp[t] = fmax3(mp[t], __uint_as_float(v[(x + t) >> 5][(x + t) & 31]),
                                  __uint_as_float(v[(x + 8 + t) >> 5][(x + 8 + t) & 31]));
            const float mx = fmaxf(fmax3(mp[0], mp[1], mp[2]), fmax3(fmax3(mp[3], mp[4], mp[5]), mp[6], mp[7])) * c2;
            // the reference max after block j - 1, from the other group
            if (j >= 1) {
                ok = __all_sync(0xffffffffu, w(bar(Cfg::kBarHand + 2 * (int)q + (g ^ 1)), ((uint32_t)(j - 1) >> 1) & 1u));
                if (!ok) break;
                const float mh = hand[(g ^ 1) * kBQ + r];
                l *= factor(m, mh);
                m = mh;
            }
            const bool grow = mx > m + 8.0f;      // false while nothing is visible
            float alpha = 1.0f;
            if (grow) {
                alpha = ex2_approx(m - mx);       // 0 on the row's first visible block
                m = mx;
                l *= alpha;
            }
            // pass the reference on to block j + 1
            hand[g * kBQ + r] = m;
            mbar_arrive_local(bar(Cfg::kBarHand + 2 * (int)q + g));
            const float mu = (m == -INFINITY) ? 0.0f : m;
            // P_j goes into the tile that P_{j-2} V_{j-2} read
            if (j >= 2) {
                ok = __all_sync(0xffffffffu, w(bar(Cfg::kBarODone + sb), (((uint32_t)j - 2) >> 1) & 1u));
                if (!ok) break;
                tc_fence_after();
            }
            // P = 2^(s - m) as 16-bit into the swizzled A tile, and its row sum
            const uint32_t prow = base + Cfg::kOffP + (uint32_t)sb * Cfg::kPBytes + (uint32_t)r * 128u;
            const uint64_t c2x2 = f2_pack(c2, c2), nmu2 = f2_pack(-mu, -mu);
            uint64_t sp[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) sp[t] = f2_pack(0.0f, 0.0f);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float e[32];
#pragma unroll
                for (int t = 0; t < 32; t += 2) {   // s * scale - m for two keys at once
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(v[c][t]), __uint_as_float(v[c][t + 1])), c2x2, nmu2), x0, x1);
                    e[t] = ex2_approx(x0);
                    e[t + 1] = ex2_approx(x1);
                    sp[(t >> 1) & 3] = f2_add(sp[(t >> 1) & 3], f2_pack(e[t], e[t + 1]));
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
            float s0, s1;
            f2_unpack(f2_add(f2_add(sp[0], sp[1]), f2_add(sp[2], sp[3])), s0, s1);
            l += s0 + s1;
            // a row whose reference max moved rescales its accumulator row, once
            // P_{j-1} V_{j-1} is in it (block 0 has nothing to rescale)
            if (j >= 1 && __any_sync(0xffffffffu, grow)) {
                ok = __all_sync(0xffffffffu, w(bar(Cfg::kBarODone + (sb ^ 1)), (((uint32_t)j - 1) >> 1) & 1u));
                if (!ok) break;
                tc_fence_after();
                const uint32_t tO = tmem + lrow + Cfg::kTmemO;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(tO + (uint32_t)c * 32u, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
                    tmem_st_32x32b_x32(tO + (uint32_t)c * 32u, o);
                }
                tmem_st_wait();
            }
            // P_j (generic-proxy stores) and the rescaled O are ready for the MMA
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_local(bar(Cfg::kBarPFull + sb));
        }
        // ---- the row sum: the group that did not take the last block brings its
        // share to the final reference, then the two shares are added
        if (ok && nkb > 0) {
            const int g_last = (nkb - 1) & 1;
            if (g != g_last && nkb >= 2) {
                ok = __all_sync(0xffffffffu,
                                w(bar(Cfg::kBarHand + 2 * (int)q + g_last), ((uint32_t)(nkb - 1) >> 1) & 1u));
                if (ok) l *= factor(m, hand[g_last * kBQ + r]);
            }
        }
        if (ok && nkb > 0) {
            sums[g * kBQ + r] = l;
            mbar_arrive_local(bar(Cfg::kBarFin + (int)q));
            ok = __all_sync(0xffffffffu, w(bar(Cfg::kBarFin + (int)q), 0u));
            if (ok) l = sums[r] + sums[kBQ + r];
        }
        // ---- O / l, stored by row, each group its D / 2 columns.  The TMEM loads
        // are warp-collective: the whole warp loads (conditions below are
        // warp-uniform); only the stores depend on the row being a real query.
        if (ok && nkb > 0) {
            ok = __all_sync(0xffffffffu,
                            w(bar(Cfg::kBarODone + ((nkb - 1) & 1)), (((uint32_t)nkb - 1) >> 1) & 1u));
            if (ok) tc_fence_after();
        }
        const bool store = i < p.Sq;
        OutT* orow = reinterpret_cast<OutT*>(p.O) + ((int64_t)bh * p.Sq + (store ? i : 0)) * D + g * (D / 2);
        const float inv = (ok && l > 0.0f) ? 1.0f / l : 0.0f;
        const uint32_t tO = tmem + lrow + Cfg::kTmemO + (uint32_t)g * (uint32_t)(D / 2);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
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
