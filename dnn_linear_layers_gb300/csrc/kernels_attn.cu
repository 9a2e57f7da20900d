// Fused attention forward: O = softmax(scale * Q K^T) V per (batch, head),
// never materialising the Sq x Sk score matrix -- the online-softmax
// recurrence of CMU 15-418 "DNNs and ML accelerators" notes, section 3.3
// (running max m, running sum l, accumulator rescaled by exp(m_old - m_new)
// whenever the max grows) and the FlashAttention tiling of youngju.dev "GEMM
// to FlashAttention" and the devpress.csdn.net notes, section 4 (Q, K, V in
// blocks that stay on chip).
//
// Design for sm_103a: persistent CTAs, one per SM, each walking work items of
// 128 queries of one head (see attn_item below); per CTA:
//   * warp 0: TMA producer -- Q of each item, K_j and V_j (128 keys each) into
//     3-slot rings (3-D tensor maps: keys past Sk read as zero).  K runs one
//     block ahead of V (a K slot frees when its score product is done, a V
//     slot only when its PV product is), and the next item's Q and first K
//     blocks load while the current item's last blocks run;
//   * warps 1 and 2: MMA issuers -- warp 1 S_j = Q K_j^T into one of two TMEM
//     score buffers (S_{j+1} is computed while the softmax works on S_j), warp
//     2 O += P_j V_j into the TMEM accumulator once P_j is ready, with P read
//     from TMEM as the A operand.  An MMA instruction is accepted only as the
//     tensor pipe drains, so one thread issuing both products would leave the
//     pipe idle while it waited for the other's operands; two threads keep it
//     fed from whichever is ready;
//   * warps 3..10: softmax in two groups of four warps that take the key blocks
//     in turn, one thread per query row (TMEM lane) in each, so the two warps
//     that share an SM sub-partition work on different blocks and hide each
//     other's latency.  A row's reference max passes from group to group once
//     per block through shared memory behind a (bounded) mbarrier; each group
//     keeps its share of the row sum until the end of the item, when the group
//     of the last block adds the other's share and writes O / l out while the
//     other group starts the next item.  Each thread reads its 128 scores from
//     TMEM once (the score buffer is handed back at once) and writes
//     P = 2^(s - m) as bf16 / fp16, two per column, into its group's 64-column
//     TMEM tile (two tiles, so P_j is written while P_{j-1} V runs).  The
//     reference max m of a row moves only when the block max exceeds it by more
//     than 8 (a factor 2^8): O = sum_j 2^(s_j - m) v_j / sum_j 2^(s_j - m) holds
//     for any m, so a stale m changes nothing but the rounding, and the
//     accumulator row is rescaled in TMEM only then.
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
    static constexpr int kStages = 3;             // K and V ring slots
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kOffMisc = kOffV + kStages * kKVBytes;
    // misc: 36 barriers (8 bytes each), then float hand-off [2 groups][128 rows],
    // the abort flag and the TMEM address
    static constexpr int kOffHand = 320;
    static constexpr int kAbort = kOffHand + 2 * kBQ * 4, kTmemPtr = kAbort + 4;
    static constexpr int kMiscBytes = kTmemPtr + 12;
    // the tiles want 1024-byte alignment; a window starting at a multiple of
    // 256 bytes fits (the kernel checks, and stops with a status bit if not)
    static constexpr int kSlack = 768;
    static constexpr int kSmem = kOffMisc + kMiscBytes + kSlack;
    // barriers: K / V ring slots indexed by global block index % 3, score and P
    // buffers by global block index & 1
    static constexpr int kBarQFull = 0, kBarQEmpty = 1, kBarK = 2, kBarV = 5, kBarKEmpty = 8, kBarVEmpty = 11,
                         kBarSFull = 14, kBarSFree = 16, kBarPFull = 18, kBarODone = 20, kBarDone = 22,
                         kBarOFree = 23,   // the item's O has been read out of TMEM
                         kBarHand = 24,    // [4 lane quarters][2 groups]: a group published a row max
                         kBarFin = 32;     // [4 lane quarters]: the other group's share of the row sums is in
    static constexpr int kTmemS = 0;      // two score buffers: columns 0..127 and 128..255
    static constexpr int kTmemO = 256;    // accumulator: columns 256 .. 256 + D - 1
    static constexpr int kTmemP = 384;    // two P tiles, 64 columns each (two 16-bit values per column)
    static_assert(36 * 8 <= kOffHand, "misc layout");
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


// 2^x on the special-function unit (ex2.approx: relative error about 2^-22,
// subnormal results flushed to zero, 2^-inf = +0)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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

// Work items of the persistent CTAs: 128 queries of one head each.  The query
// blocks of a head are consecutive items (CTAs working at the same time share
// that head's K and V in L2), taken in the order Q-1, 0, Q-2, 1, ... (Q blocks
// per head).  Under a causal mask block qb sees qb + 1 key blocks, so a CTA
// takes items in pairs: a pair costs about Q + 1 whatever it is, and the CTAs
// get even shares; otherwise every item costs the same and CTAs take them one
// by one.  Step `step` of CTA `cta` among `ctas`:
__device__ __forceinline__ int attn_item_index(bool paired, int cta, int ctas, int step) {
    return paired ? 2 * (cta + (step >> 1) * ctas) + (step & 1) : cta + step * ctas;
}
struct AttnItem {
    int bh, q0, nkb;
};
__device__ __forceinline__ AttnItem attn_item(const AttnParams& p, int qblocks, int item) {
    const int bh = item / qblocks;
    const int k = item - bh * qblocks;
    const int qb = (k & 1) ? (k >> 1) : qblocks - 1 - (k >> 1);
    return {bh, qb * kBQ, key_blocks(p, qb * kBQ)};
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
    const int qblocks = (p.Sq + kBQ - 1) / kBQ;
    const int items = p.BH * qblocks;

    if (threadIdx.x == 0) {
        mbar_init(bar(Cfg::kBarQFull), 1);
        mbar_init(bar(Cfg::kBarQEmpty), 1);
        for (int s = 0; s < Cfg::kStages; ++s) {
            mbar_init(bar(Cfg::kBarK + s), 1);
            mbar_init(bar(Cfg::kBarV + s), 1);
            mbar_init(bar(Cfg::kBarKEmpty + s), 1);
            mbar_init(bar(Cfg::kBarVEmpty + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(Cfg::kBarSFull + s), 1);
            mbar_init(bar(Cfg::kBarSFree + s), 4);   // the four warps of the group that owns buffer s
            mbar_init(bar(Cfg::kBarPFull + s), 4);
            mbar_init(bar(Cfg::kBarODone + s), 1);
        }
        mbar_init(bar(Cfg::kBarDone), 2);    // the two MMA issuers
        mbar_init(bar(Cfg::kBarOFree), 4);   // the four warps of the group that writes O out
        for (int x = 0; x < 8; ++x) mbar_init(bar(Cfg::kBarHand + x), 32);   // one warp
        for (int x = 0; x < 4; ++x) mbar_init(bar(Cfg::kBarFin + x), 32);    // one warp
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

    // Every role walks the same items in the same order.  Barrier phases follow
    // global counters: gb numbers the key blocks of all items this CTA has
    // taken (buffer gb & 1), qi / oi the items that have key blocks.
    if (warp == 0) {
        // ---- TMA producer
        if (lane == 0) {
            const AWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_PRODUCER};
            const uint64_t pol_q = l2_policy_evict_normal();
            const uint64_t pol_kv = l2_policy_evict_last();   // read by every query block of the head
            uint32_t qi = 0;
            int gb0 = 0;
            int k_issued = 0, v_issued = 0;   // key blocks whose K / V copies were issued
            bool ok = true;
            for (int step = 0, item; ok && (item = attn_item_index(p.causal != 0u, (int)blockIdx.x, (int)gridDim.x, step)) < items; ++step) {
                const AttnItem it = attn_item(p, qblocks, item);
                if (it.nkb == 0) continue;
                // Q: its tile frees once the previous item's last score product is done
                ok = w(bar(Cfg::kBarQEmpty), (qi & 1u) ^ 1u);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(Cfg::kBarQFull), Cfg::kQBytes);
#pragma unroll
                for (int b = 0; b < D / 64; ++b)
                    tma_load_3d(base + Cfg::kOffQ + b * kBox, &tmQ, bar(Cfg::kBarQFull), 64 * b, it.q0, it.bh, pol_q);
                ++qi;
                // block j (global gb) of K or V, into ring slot gb % 3: one 128-key box
                // per 64 columns
                auto load_kv = [&](const CUtensorMap* map, int off, int barid, int gb, int j) {
                    const int s = gb % Cfg::kStages;
                    mbar_arrive_expect_tx(bar(barid + s), Cfg::kKVBytes);
#pragma unroll
                    for (int b = 0; b < D / 64; ++b)
                        tma_load_3d(base + off + s * Cfg::kKVBytes + b * kBox, map, bar(barid + s), 64 * b,
                                    j * kBKey, it.bh, pol_kv);
                };
                // order K_0, K_1, V_0, K_2, V_1, ...: a K slot frees when the score
                // product three blocks back is done, a V slot when that PV product is
                auto ring_phase = [](int gb) { return ((uint32_t)(gb / Cfg::kStages) & 1u) ^ 1u; };
                ok = w(bar(Cfg::kBarKEmpty + gb0 % Cfg::kStages), ring_phase(gb0));
                if (!ok) break;
                load_kv(&tmK, Cfg::kOffK, Cfg::kBarK, gb0, 0);
                k_issued = gb0 + 1;
                for (int j = 0; j < it.nkb && ok; ++j) {
                    if (j + 1 < it.nkb) {
                        const int gn = gb0 + j + 1;
                        ok = w(bar(Cfg::kBarKEmpty + gn % Cfg::kStages), ring_phase(gn));
                        if (!ok) break;
                        load_kv(&tmK, Cfg::kOffK, Cfg::kBarK, gn, j + 1);
                        k_issued = gn + 1;
                    }
                    const int gb = gb0 + j;
                    ok = w(bar(Cfg::kBarVEmpty + gb % Cfg::kStages), ring_phase(gb));
                    if (!ok) break;
                    load_kv(&tmV, Cfg::kOffV, Cfg::kBarV, gb, j);
                    v_issued = gb + 1;
                }
                gb0 += it.nkb;
            }
            // Copies already issued land before shared memory is released:
            // wait (bounded, whatever the abort flag) for the last phase of the
            // Q tile and of each K and V slot -- immediately done in a run
            // without abort, where every copy was consumed.
            bool drained = qi == 0 || mbar_wait_bounded(bar(Cfg::kBarQFull), (qi - 1u) & 1u, p.timeout_ns);
            for (int i = k_issued - Cfg::kStages < 0 ? 0 : k_issued - Cfg::kStages; i < k_issued; ++i)
                drained &= mbar_wait_bounded(bar(Cfg::kBarK + i % Cfg::kStages), (uint32_t)(i / Cfg::kStages) & 1u,
                                             p.timeout_ns);
            for (int i = v_issued - Cfg::kStages < 0 ? 0 : v_issued - Cfg::kStages; i < v_issued; ++i)
                drained &= mbar_wait_bounded(bar(Cfg::kBarV + i % Cfg::kStages), (uint32_t)(i / Cfg::kStages) & 1u,
                                             p.timeout_ns);
            if (!drained) atomicOr(p.status, ST_TIMEOUT_PRODUCER);
        }
    } else if (warp == 1) {
        // ---- S issuer: S_j = Q K_j^T into score buffer gb & 1
        if (lane == 0) {
            const AWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_MMA};
            uint32_t qi = 0;
            int gb0 = 0;
            bool ok = true;
            for (int step = 0, item; ok && (item = attn_item_index(p.causal != 0u, (int)blockIdx.x, (int)gridDim.x, step)) < items; ++step) {
                const AttnItem it = attn_item(p, qblocks, item);
                if (it.nkb == 0) continue;
                ok = w(bar(Cfg::kBarQFull), qi & 1u);
                if (!ok) break;
                for (int j = 0; j < it.nkb && ok; ++j) {
                    const int gb = gb0 + j, s = gb & 1, r3 = gb % Cfg::kStages;
                    ok = w(bar(Cfg::kBarSFree + s), (((uint32_t)gb >> 1) & 1u) ^ 1u) &&
                         w(bar(Cfg::kBarK + r3), (uint32_t)(gb / Cfg::kStages) & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kq = base + Cfg::kOffQ, kk0 = base + Cfg::kOffK + r3 * Cfg::kKVBytes;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (uint32_t)((kk >> 2) * kBox + (kk & 3) * 32);
                        tc_mma<1>(tmem + Cfg::kTmemS + (uint32_t)s * 128u, smem_desc_sw128(kq + off, 16, 1024),
                                  smem_desc_sw128(kk0 + off, 16, 1024), p.idesc_s, kk ? 1u : 0u);
                    }
                    tc_commit_1(bar(Cfg::kBarSFull + s));
                    tc_commit_1(bar(Cfg::kBarKEmpty + r3));
                }
                if (!ok) break;
                tc_commit_1(bar(Cfg::kBarQEmpty));   // Q is free once these products are done
                ++qi;
                gb0 += it.nkb;
            }
            tc_commit_1(bar(Cfg::kBarDone));
            // every MMA of both issuers has finished before TMEM is released; this
            // wait ignores the abort flag (only its time budget ends it), so an
            // aborted run still lets the products in flight drain
            if (!mbar_try_wait(bar(Cfg::kBarDone), 0)) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(bar(Cfg::kBarDone), 0) && globaltimer_ns() - t0 < p.timeout_ns) { }
            }
        }
    } else if (warp == 2) {
        // ---- PV issuer: O += P_j V_j once the softmax has written P_j
        if (lane == 0) {
            const AWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_MMA};
            uint32_t oi = 0;
            int gb0 = 0;
            bool ok = true;
            const uint32_t tO = tmem + Cfg::kTmemO;
            for (int step = 0, item; ok && (item = attn_item_index(p.causal != 0u, (int)blockIdx.x, (int)gridDim.x, step)) < items; ++step) {
                const AttnItem it = attn_item(p, qblocks, item);
                if (it.nkb == 0) continue;
                // the accumulator holds the previous item's O until it has been read out
                ok = w(bar(Cfg::kBarOFree), (oi & 1u) ^ 1u);
                if (!ok) break;
                for (int j = 0; j < it.nkb && ok; ++j) {
                    const int gb = gb0 + j, s = gb & 1, r3 = gb % Cfg::kStages;
                    ok = w(bar(Cfg::kBarPFull + s), ((uint32_t)gb >> 1) & 1u) &&
                         w(bar(Cfg::kBarV + r3), (uint32_t)(gb / Cfg::kStages) & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t pt = tmem + Cfg::kTmemP + (uint32_t)s * 64u;
                    const uint32_t vv = base + Cfg::kOffV + r3 * Cfg::kKVBytes;
#pragma unroll
                    for (int kk = 0; kk < kBKey / 16; ++kk) {
                        // P from TMEM: 16 keys = 8 columns per step.  V is K x N = keys
                        // x D with D contiguous: MN-major, 64-column chunks one box
                        // apart, 16 key rows per step
                        tc_mma_ts(tO, pt + (uint32_t)kk * 8u, smem_desc_sw128(vv + (uint32_t)kk * 2048u, kBox, 1024),
                                  p.idesc_o, (j | kk) ? 1u : 0u);
                    }
                    if (!((p.debug & DBG_SKIP_FIRST_ACC_COMMIT) && gb == 0)) tc_commit_1(bar(Cfg::kBarODone + s));
                    tc_commit_1(bar(Cfg::kBarVEmpty + r3));
                }
                ++oi;
                gb0 += it.nkb;
            }
            tc_commit_1(bar(Cfg::kBarDone));
        }
    } else {
        // ---- softmax warps: thread = query row r (TMEM lane 32 q + lane); group g
        // takes the key blocks whose global index gb has parity g, into score
        // buffer and P tile g
        const AWait w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_EPILOGUE};
        const uint32_t q = warp & 3u;
        const int g = (int)((warp - 3u) >> 2);
        const int r = 32 * (int)q + (int)lane;
        const uint32_t lrow = (32u * q) << 16;             // TMEM lane offset of this warp
        volatile float* const hand = reinterpret_cast<volatile float*>(base_ptr + Cfg::kOffMisc + Cfg::kOffHand);
        const float c2 = p.scale_log2;
        // the factor that moves sums from reference m_old to m_new (1 when equal)
        auto factor = [](float m_old, float m_new) { return m_new == m_old ? 1.0f : ex2_approx(m_old - m_new); };
        uint32_t oi = 0;
        int gb0 = 0;
        bool ok = true;
        for (int step = 0, item; ok && (item = attn_item_index(p.causal != 0u, (int)blockIdx.x, (int)gridDim.x, step)) < items; ++step) {
            const AttnItem it = attn_item(p, qblocks, item);
            const int i = it.q0 + r;                       // query index
            const int lim = p.causal ? i + (p.Sk - p.Sq) : p.Sk - 1;   // last visible key
            const bool store = i < p.Sq;
            OutT* const orow = reinterpret_cast<OutT*>(p.O) + ((int64_t)it.bh * p.Sq + (store ? i : 0)) * D;
            if (it.nkb == 0) {   // no key is visible to any query of the item: zeros, from group 0
                if (g == 0 && store) {
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int t = 0; t < D * (int)sizeof(OutT) / 16; ++t) reinterpret_cast<uint4*>(orow)[t] = z;
                }
                continue;
            }
            const int nkb = it.nkb;
            const int gl = (gb0 + nkb - 1) & 1;            // the group that takes the item's last block
            // m: the row's reference max (base 2) as last known here; l: this
            // group's share of the row sum, relative to m
            float m = -INFINITY, l = 0.0f;
            for (int j = (g - gb0) & 1; j < nkb && ok; j += 2) {
                const int gb = gb0 + j, sb = g;
                const uint32_t ph = ((uint32_t)gb >> 1) & 1u;
                ok = __all_sync(0xffffffffu, w(bar(Cfg::kBarSFull + sb), ph));
                if (!ok) break;
                tc_fence_after();
                uint32_t v[4][32];
                const uint32_t tS = tmem + lrow + Cfg::kTmemS + (uint32_t)sb * 128u;
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(tS + (uint32_t)c * 32u, v[c]);
                tmem_ld_wait();
                // the scores are in registers: the buffer is free for the block after next
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
                    ok = __all_sync(0xffffffffu,
                                    w(bar(Cfg::kBarHand + 2 * (int)q + (g ^ 1)), ((uint32_t)(gb - 1) >> 1) & 1u));
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
                // P goes into the TMEM tile that the product of block gb - 2 read
                if (gb >= 2) {
                    ok = __all_sync(0xffffffffu, w(bar(Cfg::kBarODone + sb), (((uint32_t)gb - 2) >> 1) & 1u));
                    if (!ok) break;
                    tc_fence_after();
                }
                // P = 2^(s - m) as 16-bit values into the group's TMEM tile (two
                // per column, keys 2c and 2c + 1 in column c), and its row sum
                const uint32_t tP = tmem + lrow + Cfg::kTmemP + (uint32_t)sb * 64u;
                const uint64_t c2x2 = f2_pack(c2, c2), nmu2 = f2_pack(-mu, -mu);
                uint64_t sp[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) sp[t] = f2_pack(0.0f, 0.0f);
#pragma unroll
                for (int c = 0; c < 4; ++c) {    // keys 32 c .. 32 c + 31 -> columns 16 c .. 16 c + 15
                    // the packed pairs go into v[c] in place: entry t / 2 has been
                    // read by the time it is written
#pragma unroll
                    for (int t = 0; t < 32; t += 2) {   // s * scale - m for two keys at once
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(v[c][t]), __uint_as_float(v[c][t + 1])), c2x2, nmu2),
                                  x0, x1);
                        x0 = ex2_approx(x0);
                        x1 = ex2_approx(x1);
                        sp[(t >> 1) & 3] = f2_add(sp[(t >> 1) & 3], f2_pack(x0, x1));
                        v[c][t >> 1] = pack2<InT>(x0, x1);
                    }
                    tmem_st_32x32b_x16(tP + 16u * (uint32_t)c, v[c]);
                }
                tmem_st_wait();
                float s0, s1;
                f2_unpack(f2_add(f2_add(sp[0], sp[1]), f2_add(sp[2], sp[3])), s0, s1);
                l += s0 + s1;
                // a row whose reference max moved rescales its accumulator row, once
                // the product of block j - 1 is in it (block 0 has nothing to rescale)
                if (j >= 1 && __any_sync(0xffffffffu, grow)) {
                    ok = __all_sync(0xffffffffu, w(bar(Cfg::kBarODone + (sb ^ 1)), (((uint32_t)gb - 1) >> 1) & 1u));
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
                // P and the rescaled O are in TMEM, ready for the MMA
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_local(bar(Cfg::kBarPFull + sb));
            }
            if (!ok) break;
            if (g != gl) {
                // this group's share of the row sum, at the final reference, goes to
                // the group of the last block through that group's hand-off slot
                // (its max has just been read from there); then on to the next item
                ok = __all_sync(0xffffffffu,
                                w(bar(Cfg::kBarHand + 2 * (int)q + gl), ((uint32_t)(gb0 + nkb - 1) >> 1) & 1u));
                if (!ok) break;
                l *= factor(m, hand[gl * kBQ + r]);   // l = 0 if this group took no block of the item
                hand[gl * kBQ + r] = l;
                mbar_arrive_local(bar(Cfg::kBarFin + (int)q));
            } else {
                // the group of the last block adds the other share, writes O / l out
                // (the whole row) and frees the accumulator for the next item.  The
                // TMEM loads are warp-collective: the whole warp loads; only the
                // stores depend on the row being a real query.
                ok = __all_sync(0xffffffffu, w(bar(Cfg::kBarFin + (int)q), oi & 1u));
                if (!ok) break;
                l += hand[gl * kBQ + r];
                const int gbl = gb0 + nkb - 1;
                ok = __all_sync(0xffffffffu, w(bar(Cfg::kBarODone + (gbl & 1)), ((uint32_t)gbl >> 1) & 1u));
                if (!ok) break;
                tc_fence_after();
                const float inv = l > 0.0f ? 1.0f / l : 0.0f;
                const uint32_t tO = tmem + lrow + Cfg::kTmemO;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tO + (uint32_t)c * 32u, v);
                    tmem_ld_wait();
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
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_local(bar(Cfg::kBarOFree));
            }
            ++oi;
            gb0 += nkb;
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
    // persistent: one CTA per SM (at most one per item, or per pair of items
    // under a causal mask)
    static int sms[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (sms[dev] == 0) {
        e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    const int64_t items = (int64_t)p.BH * ((p.Sq + kBQ - 1) / kBQ);
    const int64_t units = p.causal ? (items + 1) / 2 : items;
    const unsigned grid = (unsigned)(units < sms[dev] ? units : sms[dev]);
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
