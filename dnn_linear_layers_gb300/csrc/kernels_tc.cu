// Persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   C[m][n] = epilogue( sum_k A[m][k] * B[k][n] )   epilogue = (+bias[n]) (ReLU) cast
//
// The algorithm is the tiled product of youngju.dev "GEMM to FlashAttention"
// (tiling diagram: each output tile is the sum over k-tiles of A-tile x
// B-tile) mapped onto the Blackwell primitives of the CMU 15-418 notes,
// section 2.9 (TMA copies into shared memory completing on mbarriers, one
// thread issuing tensor-core MMAs into a TMEM accumulator).  Tile sizes are
// chosen for sm_103a, not the pages' CPU blocking:
//
//   * one CTA owns 128 rows x 256 columns of the output; with cta_group::2 a
//     pair of CTAs (a 2-CTA cluster) issues 256 x 256 x 16 MMAs, each CTA
//     holding half of A's rows and half of B's columns in its own smem;
//   * a k-atom is one 128-byte swizzle row: 64 16-bit elements (kind::f16),
//     128 fp8 (kind::f8f6f4) or 32 tf32 (kind::tf32), four MMAs of 32 bytes
//     each; a ring of stages (3 stages of two atoms for a pair, 4 of one atom
//     for a single CTA) keeps TMA loads ahead of the MMAs.  A (M x K, or K x M read MN-major) and B (N x K, or
//     K x N read MN-major) come from 2-D tensor maps; for an implicit-GEMM
//     convolution A comes through an im2col map of the NHWC activations (two
//     maps, top and bottom rows of each row pair, for the fused max-pool);
//   * warp 0 issues TMA loads, warp 1 issues MMAs (leader CTA only) and owns
//     the TMEM allocation, warps 2-5 run the epilogue: TMEM -> registers ->
//     (alpha, per-column scale, +bias, +beta C, ReLU, cast) -> swizzled smem ->
//     TMA store, or for the fused max-pool the 2 x 2 maximum of each window;
//   * the accumulator is double buffered in TMEM (2 x 256 fp32 columns), so
//     the epilogue of one tile overlaps the main loop of the next;
//   * the grid is persistent (one CTA per SM) and walks the output tiles in
//     groups of `group_m` tile-rows so that the B panel stays in L2 while the
//     group is swept (wave-quantisation and even-load concerns of the
//     devpress.csdn.net notes, sections 3.6-3.7).
//
// Tails: A, B and C are described by TMA tensor maps with their true extents,
// so loads past M, N or K read zeros and stores past M or N are clipped.
//
// Every mbarrier wait is bounded by a %globaltimer budget; a wait that runs
// out records a status bit, raises a CTA-local abort flag and the roles fall
// through to a common exit that releases TMEM.  No trap, no endless spin.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace gb300 {

namespace {

constexpr int kThreads = 192;          // 6 warps
constexpr int kEpiWarps = 4;
constexpr int kTmemCols = 512;         // 2 accumulators x 256 fp32 columns

template <int CG>
struct TcCfg {
    // k-atoms (one 128-byte swizzle row per operand row: 64 16-bit, 128 fp8 or
    // 32 tf32 elements) per ring stage.  A CTA pair takes two per stage: one
    // full-barrier wait and one release per eight MMAs instead of four, which
    // measured 6% faster at 8192^3 (the MMA thread's barrier round trip per
    // stage, not the loads, held the tensor pipe back).  A single CTA keeps
    // four one-atom stages (two slots would not cover the copy latency).
    static constexpr int kAtoms = (CG == 2) ? 2 : 1;
    static constexpr int kStages = (CG == 2) ? 3 : 4;
    static constexpr int kBnCta = TC_BN / CG;                    // B columns held per CTA
    static constexpr int kAAtom = TC_BM * TC_BK * 2;            // 16 KB
    static constexpr int kBAtom = kBnCta * TC_BK * 2;           // 16 or 32 KB
    static constexpr int kAStage = kAtoms * kAAtom;
    static constexpr int kBStage = kAtoms * kBAtom;
    static constexpr int kCStage = 32 * 128;                     // one warp's 32 rows x 128 B
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kAStage;
    static constexpr int kOffC = kOffB + kStages * kBStage;
    static constexpr int kOffMisc = kOffC + kEpiWarps * 2 * kCStage;
    static constexpr int kMiscBytes = 1024;
    static constexpr int kSmem = kOffMisc + kMiscBytes + 1024;  // + alignment slack
    // misc region layout (bytes from kOffMisc)
    static constexpr int kBarFull = 0;
    static constexpr int kBarEmpty = kBarFull + 8 * kStages;
    static constexpr int kBarTFull = kBarEmpty + 8 * kStages;
    static constexpr int kBarTEmpty = kBarTFull + 16;
    static constexpr int kBarDone = kBarTEmpty + 16;
    static constexpr int kTmemPtr = kBarDone + 8;
    static constexpr int kAbort = kTmemPtr + 4;
    // max-pool hand-over between the lane quarters holding the two output rows
    static constexpr int kBarXFull = (kAbort + 4 + 7) / 8 * 8;
    static constexpr int kBarXEmpty = kBarXFull + 16;
    // ring iterations each producer of the pair issued (read by the leader on exit)
    static constexpr int kIssued = kBarXEmpty + 16;
    static_assert(kIssued + 8 <= kMiscBytes, "misc layout");
    static_assert(kEpiWarps * 2 * kCStage >= 2 * 16384, "pool hand-over needs 16 KB per warp pair");
    static_assert(kSmem <= 232448, "shared memory budget");
};

struct Waiter {
    uint64_t budget_ns;
    volatile int* abort;
    int* status;
    int bit;
    // true once the barrier phase completed; false on timeout or abort.
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
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

__device__ __forceinline__ void tile_coords(int tile, int num_m_tiles, int num_n_tiles, int group_m,
                                            int& tm, int& tn) {
    const int per_group = group_m * num_n_tiles;
    const int g = tile / per_group;
    const int first_m = g * group_m;
    const int rows = min(num_m_tiles - first_m, group_m);
    const int r = tile - g * per_group;
    tm = first_m + r % rows;
    tn = r / rows;
}

// Whole-tile work item -> output region.  Items [0, num_full) are whole
// 256-column tiles in raster order from tile sk_tiles on; each later tile is
// split into two 128-column halves (two consecutive items), which evens out
// the last, partial wave of the persistent grid when stream-K is off.
__device__ __forceinline__ void work_item(int item, const TcParams& p, int& tm, int& n0, int& nw) {
    int tile, half = -1;
    if (item < p.num_full) {
        tile = p.sk_tiles + item;
    } else {
        const int j = item - p.num_full;
        tile = p.sk_tiles + p.num_full + (j >> 1);
        half = j & 1;
    }
    int tn;
    tile_coords(tile, p.num_m_tiles, p.num_n_tiles, p.group_m, tm, tn);
    n0 = tn * TC_BN + (half > 0 ? TC_BN / 2 : 0);
    nw = half < 0 ? TC_BN : TC_BN / 2;
}

// One piece of a worker's sequence: a k-range of a split tile (stream-K) or
// a whole tile (or N-half).
struct Piece {
    int tm, n0, nw;          // output region: tile row, first column, width
    int kb0, nkb;            // k-atoms [kb0, kb0 + nkb) of the tile
    int tile;                // split tiles: tile index (< sk_tiles)
    int contrib, ncontrib;   // split tiles: this worker's rank among the contributors (k order), their number
    bool partial;            // the tile has other contributors
    bool rev;                // walk the tile's k-stages backwards (serpentine order)
};

// Worker owning stream-K atom a when A atoms are split over W workers in
// equal ranges [w A / W, (w + 1) A / W): the largest w with w A / W <= a.
__device__ __forceinline__ int sk_owner(int64_t a, int64_t A, int64_t W) { return (int)(((a + 1) * W - 1) / A); }

// Piece idx of worker `unit`'s sequence (stream-K pieces, then whole tiles
// every num_units); false past its end.  Producer, MMA issuer and epilogue
// walk the same sequence.
__device__ __forceinline__ bool piece_at(const TcParams& p, int unit, int num_units, int idx, Piece& pc) {
    const int nkb = p.num_k_blocks;
    const int64_t A = (int64_t)p.sk_tiles * nkb, W = p.sk_workers;
    int n_sk = 0;
    int64_t s = 0, e = 0;
    if (unit < p.sk_workers) {                 // W <= A: every range is non-empty
        s = (int64_t)unit * A / W;
        e = (int64_t)(unit + 1) * A / W;
        n_sk = (int)((e - 1) / nkb - s / nkb + 1);
    }
    if (idx < n_sk) {
        const int t = (int)(s / nkb) + idx;
        const int64_t t0 = (int64_t)t * nkb;
        const int64_t lo = s > t0 ? s : t0, hi = e < t0 + nkb ? e : t0 + nkb;
        pc.kb0 = (int)(lo - t0);
        pc.nkb = (int)(hi - lo);
        const int wf = sk_owner(t0, A, W), wl = sk_owner(t0 + nkb - 1, A, W);
        pc.ncontrib = wl - wf + 1;
        pc.contrib = unit - wf;
        pc.partial = pc.ncontrib > 1;
        pc.tile = t;
        pc.rev = false;
        int tn;
        tile_coords(t, p.num_m_tiles, p.num_n_tiles, p.group_m, pc.tm, tn);
        pc.n0 = tn * TC_BN;
        pc.nw = TC_BN;
        return true;
    }
    const int j = idx - n_sk;
    const int dp_items = p.num_full + 2 * (p.num_m_tiles * p.num_n_tiles - p.sk_tiles - p.num_full);
    const int item = unit + j * num_units;
    if (item >= dp_items) return false;
    work_item(item, p, pc.tm, pc.n0, pc.nw);
    pc.kb0 = 0;
    pc.nkb = nkb;
    pc.tile = -1;
    pc.contrib = 0;
    pc.ncontrib = 1;
    pc.partial = false;
    pc.rev = p.k_snake && (j & 1);
    return true;
}

template <typename OutT> struct OutTraits;
template <> struct OutTraits<float> {
    static constexpr int kCols = 32;   // 128-byte row chunk
    static __device__ __forceinline__ float cvt(float v) { return v; }
};
template <> struct OutTraits<__nv_bfloat16> {
    static constexpr int kCols = 64;
    static __device__ __forceinline__ __nv_bfloat16 cvt(float v) { return __float2bfloat16_rn(v); }
};
template <> struct OutTraits<__half> {
    static constexpr int kCols = 64;
    static __device__ __forceinline__ __half cvt(float v) { return __float2half_rn(v); }
};

template <typename InT> __device__ __forceinline__ float to_f32(InT v);
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
__device__ __forceinline__ float out_to_f32(float v) { return v; }
__device__ __forceinline__ float out_to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float out_to_f32(__half v) { return __half2float(v); }

__device__ __forceinline__ uint32_t pack2(float a, float b, __nv_bfloat16*) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack2(float a, float b, __half*) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_shared_v4f(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

// CG = CTAs per cluster (1, or 2 for a CTA pair issuing cta_group::2 MMAs).
// Each CTA fetches its own operand tiles: no copy is shared across CTAs.
template <int CG, typename InT, typename OutT, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
               const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, const TcParams p) {
    using Cfg = TcCfg<CG>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle pattern.
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw_addr);

    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = lane_id();
    const uint32_t crank = (CG == 2) ? cluster_ctarank() : 0u;   // rank within the pair
    const int unit = (int)(blockIdx.x / CG);
    const int num_units = (int)(gridDim.x / CG);

    const uint32_t misc = base + Cfg::kOffMisc;
    auto bar_full = [&](int s) { return misc + Cfg::kBarFull + 8u * s; };
    auto bar_empty = [&](int s) { return misc + Cfg::kBarEmpty + 8u * s; };
    auto bar_tfull = [&](int a) { return misc + Cfg::kBarTFull + 8u * a; };
    auto bar_tempty = [&](int a) { return misc + Cfg::kBarTEmpty + 8u * a; };
    const uint32_t bar_done = misc + Cfg::kBarDone;
    auto bar_xfull = [&](uint32_t i) { return misc + Cfg::kBarXFull + 8u * i; };
    auto bar_xempty = [&](uint32_t i) { return misc + Cfg::kBarXEmpty + 8u * i; };

    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + Cfg::kOffMisc + Cfg::kAbort);
    volatile uint32_t* issued = reinterpret_cast<volatile uint32_t*>(base_ptr + Cfg::kOffMisc + Cfg::kIssued);
    uint32_t* tmem_ptr_smem = reinterpret_cast<uint32_t*>(base_ptr + Cfg::kOffMisc + Cfg::kTmemPtr);

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::kStages; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_tfull(a), 1);
            mbar_init(bar_tempty(a), kEpiWarps * CG);
        }
        mbar_init(bar_done, 1);
        for (uint32_t i = 0; i < 2; ++i) {
            mbar_init(bar_xfull(i), 1);
            mbar_init(bar_xempty(i), 1);
        }
        *abort_flag = 0;
        issued[0] = issued[1] = 0u;
        fence_mbarrier_init_cluster();
        tma_prefetch_desc(&tmA);
        if (p.conv_pool) tma_prefetch_desc(&tmA2);
        tma_prefetch_desc(&tmB);
        if (!p.c_direct) tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(tmem_ptr_smem), kTmemCols);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    if constexpr (CG == 2) cluster_sync_all(); else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_ptr_smem;
    // The prologue above may overlap the previous kernel of the stream; no
    // operand, bias or output is touched until that kernel has finished.
    grid_dependency_wait();
    grid_launch_dependents();

    const int nkb = p.num_k_blocks;
    // elements per 128-byte k-block row: 64 16-bit, 128 fp8 or 32 tf32
    constexpr int kBk = KIND == 1 ? 2 * TC_BK : (KIND == 2 ? TC_BK / 2 : TC_BK);

    // MN-major operands (K x N B, K x M A) arrive as boxes one 128-byte
    // swizzle row wide (kBk columns) and kBk k-rows high, kBox bytes apart:
    // 2 boxes per 128 columns for 16-bit types, 1 for fp8, 4 for tf32.  An
    // N x K B is one full-height box (a half tile uses its top rows).
    constexpr uint32_t kBox = (uint32_t)kBk * 128u;
    const bool boxes64 = p.b_mn_major != 0;
    // ring iterations (stages) of a piece, and the k-atoms of its stage stk
    auto stages_of = [](const Piece& pc) { return (pc.nkb + Cfg::kAtoms - 1) / Cfg::kAtoms; };
    auto atoms_of = [](const Piece& pc, int stk) { return min(Cfg::kAtoms, pc.nkb - stk * Cfg::kAtoms); };
    // bytes one CTA's copies bring per k-atom of a piece nw columns wide
    auto atom_bytes = [&](int nw) -> uint32_t {
        return (uint32_t)Cfg::kAAtom +
               (boxes64 && !p.b_chunks ? (uint32_t)(nw / CG / kBk) * kBox : (uint32_t)Cfg::kBAtom);
    };
    // bytes of ring iteration i (counted over the worker's whole sequence)
    auto iter_bytes = [&](int i) -> uint32_t {
        for (int idx = 0;; ++idx) {
            Piece pc;
            if (!piece_at(p, unit, num_units, idx, pc)) return 0u;
            const int n = stages_of(pc);
            if (i < n) return (uint32_t)atoms_of(pc, pc.rev ? n - 1 - i : i) * atom_bytes(pc.nw);
            i -= n;
        }
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            const Waiter w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_PRODUCER};
            // The group walk reuses each A panel across every N tile of the group and
            // each B panel only across the group's rows, so A is the operand to keep.
            const uint64_t pol_a = p.l2_policy == 0 ? l2_policy_evict_last() : l2_policy_evict_normal();
            const uint64_t pol_b = p.l2_policy == 1 ? l2_policy_evict_last() : l2_policy_evict_normal();
            uint32_t it = 0;
            bool ok = true;
            for (int idx = 0; ok; ++idx) {
                Piece pc;
                if (!piece_at(p, unit, num_units, idx, pc)) break;
                const int tm = pc.tm, n0 = pc.n0, nw = pc.nw;
                // serpentine k order (whole tiles): a tile starts on the k-slabs the
                // previous one ended on, which are the ones most likely still in L2
                const bool rev = pc.rev;
                const int nst = stages_of(pc);
                const int m0 = tm * TC_BM * CG + (int)crank * TC_BM;
                const int nb = n0 + (int)crank * (nw / CG);
                // implicit GEMM: base pixel (top-left of the filter window) of row m0
                int px_n = 0, px_h = 0, px_w = 0;
                if (p.conv && p.conv_pool) {
                    // CTA tile u: positions 64 u .. 64 u + 63 of the sequence (image, row
                    // pair ph, column); the top-row map walks rows 2 ph, the bottom-row
                    // map rows 2 ph + 1 (both step two rows and run on across images)
                    const int k0 = (m0 / TC_BM) * 64;
                    const int per_img = p.pool_ph * p.conv_out_w;
                    px_n = k0 / per_img;
                    const int rem = k0 - px_n * per_img;
                    const int ph = rem / p.conv_out_w;
                    px_h = 2 * ph - p.conv_pad;
                    px_w = rem - ph * p.conv_out_w - p.conv_pad;
                } else if (p.conv) {
                    px_n = m0 / p.conv_out_hw;
                    const int rem = m0 - px_n * p.conv_out_hw;
                    px_h = rem / p.conv_out_w - p.conv_pad;
                    px_w = rem % p.conv_out_w - p.conv_pad;
                }
                // A tile of k-block k0: a 2-D box of the matrix, or the tap's
                // channel block through the im2col map
                auto load_a = [&](uint32_t dst, uint32_t bar, int k0, bool pair_bar) {
                    if (p.conv) {
                        const int kbi = k0 / TC_BK;
                        const int tap = kbi / p.conv_cb;
                        const int c0 = (kbi - tap * p.conv_cb) * TC_BK;
                        const int r = tap / p.conv_s;
                        const uint16_t off_w = (uint16_t)(tap - r * p.conv_s), off_h = (uint16_t)r;
                        if (p.conv_pool) {
                            // two boxes of 64 pixels, top rows then bottom rows, 8 KB apart
                            for (int h = 0; h < 2; ++h) {
                                const uint32_t d = dst + (uint32_t)h * 8192u;
                                const CUtensorMap* map = h ? &tmA2 : &tmA;
                                if (pair_bar)
                                    tma_load_im2col_pair(d, map, bar, c0, px_w, px_h + h, px_n, off_w, off_h, pol_a);
                                else
                                    tma_load_im2col(d, map, bar, c0, px_w, px_h + h, px_n, off_w, off_h, pol_a);
                            }
                        } else {
                            if (pair_bar) tma_load_im2col_pair(dst, &tmA, bar, c0, px_w, px_h, px_n, off_w, off_h, pol_a);
                            else tma_load_im2col(dst, &tmA, bar, c0, px_w, px_h, px_n, off_w, off_h, pol_a);
                        }
                    } else if (p.a_chunks) {
                        // K x M operand, M a multiple of 64: the tile's two 64-column
                        // chunks in one copy
                        if (pair_bar) tma_load_3d_pair(dst, &tmA, bar, 0, k0, m0 / 64, pol_a);
                        else tma_load_3d(dst, &tmA, bar, 0, k0, m0 / 64, pol_a);
                    } else if (p.a_mn_major) {
                        // K x M operand: TC_BM / kBk boxes of kBk rows (M) x kBk k
                        for (int c = 0; c < TC_BM / kBk; ++c) {
                            if (pair_bar) tma_load_2d_pair(dst + (uint32_t)c * kBox, &tmA, bar, m0 + kBk * c, k0, pol_a);
                            else tma_load_2d(dst + (uint32_t)c * kBox, &tmA, bar, m0 + kBk * c, k0, pol_a);
                        }
                    } else {
                        if (pair_bar) tma_load_2d_pair(dst, &tmA, bar, k0, m0, pol_a);
                        else tma_load_2d(dst, &tmA, bar, k0, m0, pol_a);
                    }
                };
                // (a chunked K x N B always copies all of a CTA's chunks, also
                // for a half tile, whose MMAs read only the first)
                const int b_boxes = boxes64 ? nw / CG / kBk : 1;
                const uint32_t b_bytes = boxes64 && !p.b_chunks ? (uint32_t)b_boxes * kBox : (uint32_t)Cfg::kBAtom;
                for (int st = 0; st < nst; ++st, ++it) {
                    const int s = (int)(it % Cfg::kStages);
                    const uint32_t ph = (it / Cfg::kStages) & 1u;
                    if (!w.wait(bar_empty(s), ph ^ 1u)) { ok = false; break; }
                    const int stk = rev ? nst - 1 - st : st;
                    const int na = atoms_of(pc, stk);
                    const uint32_t bytes = (uint32_t)na * ((uint32_t)Cfg::kAAtom + b_bytes);
                    if constexpr (CG == 2) {
                        if (crank == 0) mbar_arrive_expect_tx(bar_full(s), 2u * bytes);
                    } else {
                        mbar_arrive_expect_tx(bar_full(s), bytes);
                    }
                    for (int j = 0; j < na; ++j) {
                        const uint32_t sa = base + Cfg::kOffA + s * Cfg::kAStage + j * Cfg::kAAtom;
                        const uint32_t sb = base + Cfg::kOffB + s * Cfg::kBStage + j * Cfg::kBAtom;
                        const int k0 = (pc.kb0 + stk * Cfg::kAtoms + j) * kBk;
                        if constexpr (CG == 2) {
                            const uint32_t fb = mapa_shared(bar_full(s), 0);
                            load_a(sa, fb, k0, true);
                            if (p.b_chunks) {
                                tma_load_3d_pair(sb, &tmB, fb, 0, k0, nb / 64, pol_b);
                            } else if (boxes64) {
                                for (int c = 0; c < b_boxes; ++c)
                                    tma_load_2d_pair(sb + c * kBox, &tmB, fb, nb + kBk * c, k0, pol_b);
                            } else {
                                tma_load_2d_pair(sb, &tmB, fb, k0, nb, pol_b);
                            }
                        } else {
                            load_a(sa, bar_full(s), k0, false);
                            if (p.b_chunks) {
                                tma_load_3d(sb, &tmB, bar_full(s), 0, k0, nb / 64, pol_b);
                            } else if (p.b_mn_major) {
                                for (int c = 0; c < b_boxes; ++c)
                                    tma_load_2d(sb + c * kBox, &tmB, bar_full(s), nb + kBk * c, k0, pol_b);
                            } else {
                                tma_load_2d(sb, &tmB, bar_full(s), k0, nb, pol_b);
                            }
                        }
                    }
                }
            }
            // iterations issued (a failed wait breaks before its copies): the
            // leader reconciles both counts on exit (teardown below)
            if (crank == 0) issued[0] = it;
            else st_shared_cluster_u32(mapa_shared(smem_u32((const void*)(issued + 1)), 0), it);
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer ----
        if (crank == 0 && lane == 0) {
            const Waiter w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_MMA};
            // stage release and accumulator hand-over reach both CTAs of the pair
            const uint16_t pair_mask = 0x3u;
            uint32_t it = 0, tcount = 0;
            bool ok = true;
            for (int idx = 0; ok; ++idx, ++tcount) {
                Piece pc;
                if (!piece_at(p, unit, num_units, idx, pc)) break;
                const uint32_t idesc = pc.nw == TC_BN ? p.idesc : p.idesc_half;
                const int nst = stages_of(pc);
                const uint32_t a = tcount & 1u;
                const uint32_t aph = (tcount >> 1) & 1u;
                if (!w.wait(bar_tempty(a), aph ^ 1u)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + a * TC_BN;
                const bool rev = pc.rev;
                // descriptors built once; per stage, atom and MMA only the start
                // address field (bits 0-13, address >> 4) moves
                // (MN-major: leading byte offset = the distance between boxes)
                const uint64_t a0 = p.a_mn_major ? smem_desc_sw128(base + Cfg::kOffA, kBox, 1024)
                                                 : smem_desc_sw128(base + Cfg::kOffA, 16, 1024);
                const uint64_t b0 = p.b_mn_major ? smem_desc_sw128(base + Cfg::kOffB, kBox, 1024)
                                                 : smem_desc_sw128(base + Cfg::kOffB, 16, 1024);
                // one MMA takes a quarter of the k-atom: 32 bytes along a K-major
                // row, or kBk / 4 k-rows of 128 bytes of an MN-major box
                const uint32_t a_kstep = p.a_mn_major ? (uint32_t)(kBk * 32) >> 4 : 32u >> 4;
                const uint32_t b_kstep = p.b_mn_major ? (uint32_t)(kBk * 32) >> 4 : 32u >> 4;
                for (int st = 0; st < nst; ++st, ++it) {
                    const int s = (int)(it % Cfg::kStages);
                    const uint32_t ph = (it / Cfg::kStages) & 1u;
                    // the stage's bytes arrived through the async proxy that the MMA
                    // reads with; the barrier wait alone orders them (no tcgen05 fence,
                    // which would hold the tensor pipe at every stage)
                    if (!w.wait(bar_full(s), ph)) { ok = false; break; }
                    const int na = atoms_of(pc, rev ? nst - 1 - st : st);
                    const uint64_t as = a0 + (uint64_t)((s * Cfg::kAStage) >> 4);
                    const uint64_t bs = b0 + (uint64_t)((s * Cfg::kBStage) >> 4);
                    // four MMAs per k-atom
                    for (int j = 0; j < na; ++j)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma<CG, KIND>(d_tmem, as + (uint64_t)((j * Cfg::kAAtom) >> 4) + kk * a_kstep,
                                             bs + (uint64_t)((j * Cfg::kBAtom) >> 4) + kk * b_kstep, idesc,
                                             (st | j | kk) != 0 ? 1u : 0u);
                    if constexpr (CG == 2) tc_commit_2(bar_empty(s), pair_mask); else tc_commit_1(bar_empty(s));
                }
                if (!ok) break;
                if (!((p.debug & DBG_SKIP_FIRST_ACC_COMMIT) && tcount == 0)) {
                    if constexpr (CG == 2) tc_commit_2(bar_tfull(a), pair_mask); else tc_commit_1(bar_tfull(a));
                }
            }
            // Every MMA this thread issued has finished before TMEM can be released.
            if constexpr (CG == 2) tc_commit_2(bar_done, (uint16_t)(1u << crank)); else tc_commit_1(bar_done);
            const Waiter wd{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_MMA};
            if (!mbar_try_wait(bar_done, 0)) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(bar_done, 0) && globaltimer_ns() - t0 < wd.budget_ns) { }
            }
        }
    } else {
        // --------------------------------------------------- epilogue ----
        const Waiter w{p.timeout_ns, abort_flag, p.status, ST_TIMEOUT_EPILOGUE};
        const uint32_t q = warp & 3u;                 // TMEM lane quarter of this warp
        constexpr int kCols = OutTraits<OutT>::kCols;

        const uint32_t cbuf0 = base + Cfg::kOffC + (warp - 2) * 2 * Cfg::kCStage;
        const bool has_bias = (p.epi & EPI_BIAS) != 0;
        const bool relu = (p.epi & EPI_RELU) != 0;
        const InT* bias = reinterpret_cast<const InT*>(p.bias);
        const uint32_t tempty_leader0 = (CG == 2) ? mapa_shared(bar_tempty(0), 0) : bar_tempty(0);
        const uint32_t tempty_leader1 = (CG == 2) ? mapa_shared(bar_tempty(1), 0) : bar_tempty(1);
        uint32_t tcount = 0, cstore = 0;
        for (int idx = 0;; ++idx, ++tcount) {
            Piece pc;
            if (!piece_at(p, unit, num_units, idx, pc)) break;
            const int tm = pc.tm, n0 = pc.n0, nw = pc.nw;
            const int kChunks = nw / kCols;
            const int m0 = tm * TC_BM * CG + (int)crank * TC_BM;
            const int row0 = m0 + 32 * (int)q;
            const uint32_t a = tcount & 1u;
            const uint32_t aph = (tcount >> 1) & 1u;
            // all lanes poll; the warp leaves together if any lane gave up
            const bool ready = w.wait(bar_tfull(a), aph);
            if (!__all_sync(0xffffffffu, ready)) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + ((32u * q) << 16) + a * TC_BN;
            if (p.conv_pool) {
                // Lanes 0..63 of the accumulator hold the top pixels of positions
                // 64 u + lane, lanes 64..127 the bottom pixels of the same positions;
                // position k is pooled output row k / 2 (OW is even).  Every warp applies the
                // epilogue and takes the max with its horizontal neighbour (lane ^ 1);
                // the row 2 ph + 1 quarters (q = 2, 3) then leave their even lanes' values
                // for the whole tile in shared memory (16 KB each, one hand-over per
                // tile), and the row 2 ph quarters (q = 0, 1) take the vertical max and
                // store the pooled pixels from their even lanes.
                const int kpos = (m0 / TC_BM) * 64 + 32 * (int)(q & 1u) + (int)lane;
                const bool writer = (q >> 1) != 0;
                const bool even = (lane & 1u) == 0;
                // 16 rows (even lanes) x 128 B per 32-column chunk, 16 KB per tile
                const uint32_t xrow = base + Cfg::kOffC + (q & 1u) * 4 * Cfg::kCStage + (lane >> 1) * 128u;
                const uint32_t xf = bar_xfull(q & 1u), xe = bar_xempty(q & 1u);
                const uint32_t xph = tcount & 1u;
                const bool out_ok = !writer && even && kpos < 2 * p.pool_rows;
                OutT* const yrow = reinterpret_cast<OutT*>(p.pool_y) + (int64_t)(kpos >> 1) * p.pool_ldy;
                const InT* sc = reinterpret_cast<const InT*>(p.ex.scale);
                const int chunks = nw / 32;
                bool ok = true;
                if (writer) {   // the previous tile's values must have been read
                    ok = w.wait(xe, xph ^ 1u);
                    ok = __all_sync(0xffffffffu, ok);
                } else {        // this tile's values must have been written
                    ok = w.wait(xf, xph);
                    ok = __all_sync(0xffffffffu, ok);
                }
                for (int c = 0; c < chunks; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + c * 32, r);
                    tmem_ld_wait();
                    if (c == chunks - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster(a ? tempty_leader1 : tempty_leader0);
                    }
                    const int cb = n0 + c * 32;
                    float sv[32], bv[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) { sv[j] = 1.0f; bv[j] = 0.0f; }
                    if (cb + 32 <= p.N && (!has_bias || p.bias_vec16) && (!(p.epi & EPI_SCALE) || p.ex.scale_vec16)) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (p.epi & EPI_SCALE) {
                                const uint4 us = __ldg(reinterpret_cast<const uint4*>(sc + cb) + j);
                                const InT* es = reinterpret_cast<const InT*>(&us);
#pragma unroll
                                for (int t = 0; t < 8; ++t) sv[8 * j + t] = to_f32<InT>(es[t]);
                            }
                            if (has_bias) {
                                const uint4 ub = __ldg(reinterpret_cast<const uint4*>(bias + cb) + j);
                                const InT* eb = reinterpret_cast<const InT*>(&ub);
#pragma unroll
                                for (int t = 0; t < 8; ++t) bv[8 * j + t] = to_f32<InT>(eb[t]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            if (cb + j < p.N) {
                                if (p.epi & EPI_SCALE) sv[j] = to_f32<InT>(sc[cb + j]);
                                if (has_bias) bv[j] = to_f32<InT>(bias[cb + j]);
                            }
                        }
                    }
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        float t = __uint_as_float(r[j]);
                        if (p.epi & EPI_ALPHA) t *= p.ex.alpha;
                        t = t * sv[j] + bv[j];
                        if (relu) t = fmaxf(t, 0.0f);
                        v[j] = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 1));
                    }
                    const uint32_t xa = xrow + (uint32_t)c * 2048u;   // 16 rows x 128 B per chunk
                    if (writer) {
                        if (ok && even) {
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                st_shared_v4(xa + ((j ^ ((lane >> 1) & 7u)) << 4), __float_as_uint(v[4 * j]),
                                             __float_as_uint(v[4 * j + 1]), __float_as_uint(v[4 * j + 2]),
                                             __float_as_uint(v[4 * j + 3]));
                        }
                    } else if (ok && out_ok) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 o = ld_shared_v4f(xa + ((j ^ ((lane >> 1) & 7u)) << 4));
                            v[4 * j] = fmaxf(v[4 * j], o.x); v[4 * j + 1] = fmaxf(v[4 * j + 1], o.y);
                            v[4 * j + 2] = fmaxf(v[4 * j + 2], o.z); v[4 * j + 3] = fmaxf(v[4 * j + 3], o.w);
                        }
                        OutT* dst = yrow + cb;
                        if (p.pool_vec16 && cb + 32 <= p.N) {
                            constexpr int kPer = 16 / (int)sizeof(OutT);
#pragma unroll
                            for (int j = 0; j < 32 / kPer; ++j) {
                                OutT o[kPer];
#pragma unroll
                                for (int t = 0; t < kPer; ++t) o[t] = OutTraits<OutT>::cvt(v[kPer * j + t]);
                                *reinterpret_cast<uint4*>(dst + kPer * j) = *reinterpret_cast<const uint4*>(o);
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (cb + j < p.N) dst[j] = OutTraits<OutT>::cvt(v[j]);
                        }
                    }
                }
                __syncwarp();
                if (ok && lane == 0) mbar_arrive_local(writer ? xf : xe);
                if (!ok) break;
                continue;
            }
            // A chunk of kCols columns (each lane its row's values): alpha, scale,
            // bias, beta * previous C, ReLU, cast, swizzled staging, TMA store.
            auto finish_chunk = [&](int c, float (&v)[kCols]) {
                const int cb = n0 + c * kCols;
                if (p.epi & EPI_ALPHA) {
#pragma unroll
                    for (int j = 0; j < kCols; ++j) v[j] *= p.ex.alpha;
                }
                if (p.epi & EPI_SCALE) {
                    // per-column factors, like the bias: one broadcast load per vector
                    const InT* sc = reinterpret_cast<const InT*>(p.ex.scale);
                    if (p.ex.scale_vec16 && cb + kCols <= p.N) {
                        const uint4* sv = reinterpret_cast<const uint4*>(sc + cb);
#pragma unroll
                        for (int j = 0; j < kCols / 8; ++j) {
                            const uint4 u = __ldg(sv + j);
                            const InT* e = reinterpret_cast<const InT*>(&u);
#pragma unroll
                            for (int t = 0; t < 8; ++t) v[8 * j + t] *= to_f32<InT>(e[t]);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < kCols; ++j)
                            if (cb + j < p.N) v[j] *= to_f32<InT>(sc[cb + j]);
                    }
                }
                if (has_bias) {
                    // every lane reads the same addresses: one broadcast load per vector
                    if (p.bias_vec16 && cb + kCols <= p.N) {
                        const uint4* bv = reinterpret_cast<const uint4*>(bias + cb);
#pragma unroll
                        for (int j = 0; j < kCols / 8; ++j) {
                            const uint4 u = __ldg(bv + j);
                            const InT* e = reinterpret_cast<const InT*>(&u);
#pragma unroll
                            for (int t = 0; t < 8; ++t) v[8 * j + t] += to_f32<InT>(e[t]);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < kCols; ++j)
                            if (cb + j < p.N) v[j] += to_f32<InT>(bias[cb + j]);
                    }
                }
                if (p.epi & EPI_BETA) {
                    // lane = row of the chunk: its 128 bytes of the previous C, read
                    // before this warp's store of the same elements is issued
                    const int row = row0 + (int)lane;
                    if (row < p.M) {
                        const OutT* crow = reinterpret_cast<const OutT*>(p.ex.c_old) + (int64_t)row * p.ex.ldc_old + cb;
                        if (p.ex.c_old_vec16 && cb + kCols <= p.N) {
                            constexpr int kPer = 16 / (int)sizeof(OutT);
#pragma unroll
                            for (int j = 0; j < kCols / kPer; ++j) {
                                const uint4 u = *reinterpret_cast<const uint4*>(crow + kPer * j);
                                const OutT* e = reinterpret_cast<const OutT*>(&u);
#pragma unroll
                                for (int t = 0; t < kPer; ++t) v[kPer * j + t] += p.ex.beta * out_to_f32(e[t]);
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < kCols; ++j)
                                if (cb + j < p.N) v[j] += p.ex.beta * out_to_f32(crow[j]);
                        }
                    }
                }
                if (relu) {
#pragma unroll
                    for (int j = 0; j < kCols; ++j) v[j] = fmaxf(v[j], 0.0f);
                }
                const uint32_t buf = cbuf0 + (cstore & 1u) * Cfg::kCStage;
                if (lane == 0) bulk_wait_group_read<1>();
                __syncwarp();
                const uint32_t row_addr = buf + lane * 128u;
#pragma unroll
                for (int j = 0; j < 8; ++j) {            // eight 16-byte pieces of the 128-byte row
                    uint32_t w0, w1, w2, w3;
                    if constexpr (sizeof(OutT) == 4) {
                        w0 = __float_as_uint(v[4 * j + 0]); w1 = __float_as_uint(v[4 * j + 1]);
                        w2 = __float_as_uint(v[4 * j + 2]); w3 = __float_as_uint(v[4 * j + 3]);
                    } else {
                        w0 = pack2(v[8 * j + 0], v[8 * j + 1], (OutT*)nullptr);
                        w1 = pack2(v[8 * j + 2], v[8 * j + 3], (OutT*)nullptr);
                        w2 = pack2(v[8 * j + 4], v[8 * j + 5], (OutT*)nullptr);
                        w3 = pack2(v[8 * j + 6], v[8 * j + 7], (OutT*)nullptr);
                    }
                    st_shared_v4(row_addr + ((j ^ (lane & 7u)) << 4), w0, w1, w2, w3);
                }
                if (p.c_direct) {
                    // C breaks the TMA rule (pitch or base): the warp writes its 32
                    // staged rows itself, one row at a time, lane l the l-th 4-byte
                    // word of the row's 128 bytes (coalesced; 16-bit halves where a
                    // word of C is not 4-byte aligned)
                    __syncwarp();
                    OutT* const Cg = reinterpret_cast<OutT*>(p.c_ptr);
                    constexpr int kPerWord = 4 / (int)sizeof(OutT);
                    const int col = cb + (int)lane * kPerWord;
                    for (int r = 0; r < 32 && row0 + r < p.M; ++r) {
                        const uint32_t word = ld_shared_u32(buf + r * 128u + ((((lane >> 2) ^ (uint32_t)(r & 7)) << 4) |
                                                                            ((lane & 3u) << 2)));
                        OutT* dst = Cg + (int64_t)(row0 + r) * p.ldc + col;
                        if constexpr (kPerWord == 1) {
                            if (col < p.N) *reinterpret_cast<uint32_t*>(dst) = word;
                        } else if (col + 1 < p.N && (reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
                            *reinterpret_cast<uint32_t*>(dst) = word;
                        } else {
                            if (col < p.N) *reinterpret_cast<uint16_t*>(dst) = (uint16_t)(word & 0xFFFFu);
                            if (col + 1 < p.N) *reinterpret_cast<uint16_t*>(dst + 1) = (uint16_t)(word >> 16);
                        }
                    }
                    __syncwarp();
                } else {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int col = n0 + c * kCols;
                        if (row0 < p.M && col < p.N) tma_store_2d(&tmC, buf, col, row0);
                        bulk_commit_group();
                    }
                }
                ++cstore;
            };
            if (pc.partial) {
                // Stream-K: this worker holds part of the tile's K range.  The warp
                // writes its fp32 partial (32 rows x 256 columns) into its slot of
                // the tile: 16-byte piece j (columns 4j .. 4j + 3) of 32-column chunk
                // cc of lane l's row at float4 (cc * 8 + j) * 32 + l, so each warp
                // access covers 512 contiguous bytes (coalesced),
                // frees the accumulator, and counts its arrival once its stores are
                // visible (fence, then atomic).  The last arrival of the slot (which
                // waits for no one) adds the contributors' partials in k order,
                // its own included, so the sum does not depend on arrival order,
                // runs the epilogue and resets the counter for the next launch.
                const int g = (int)crank * 4 + (int)q;
                auto slot = [&](int c) {
                    return p.sk_part + ((((int64_t)pc.tile * p.sk_maxc + c) * 8 + g) << 13);
                };
                float* const mine = slot(pc.contrib);
                for (int cc = 0; cc < TC_BN / 32; ++cc) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + cc * 32, r);
                    tmem_ld_wait();
                    float4* dst = reinterpret_cast<float4*>(mine) + cc * 256 + (int)lane;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        __stcg(dst + 32 * j, make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                    __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(a ? tempty_leader1 : tempty_leader0);
                __threadfence();
                __syncwarp();
                int old = 0;
                if (lane == 0) old = atomicAdd(p.sk_cnt + pc.tile * 8 + g, 1);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (old != pc.ncontrib - 1) continue;
                __threadfence();
                for (int c = 0; c < kChunks; ++c) {
                    float v[kCols];
#pragma unroll
                    for (int j = 0; j < kCols; ++j) v[j] = 0.0f;
                    for (int k = 0; k < pc.ncontrib; ++k) {
                        const float* src = slot(k);
#pragma unroll
                        for (int h = 0; h < kCols / 32; ++h) {
                            const float4* s4 =
                                reinterpret_cast<const float4*>(src) + (c * (kCols / 32) + h) * 256 + (int)lane;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float4 x = __ldcg(s4 + 32 * j);
                                v[h * 32 + 4 * j] += x.x;
                                v[h * 32 + 4 * j + 1] += x.y;
                                v[h * 32 + 4 * j + 2] += x.z;
                                v[h * 32 + 4 * j + 3] += x.w;
                            }
                        }
                    }
                    finish_chunk(c, v);
                }
                if (lane == 0) p.sk_cnt[pc.tile * 8 + g] = 0;
                continue;
            }
            for (int c = 0; c < kChunks; ++c) {
                float v[kCols];
#pragma unroll
                for (int h = 0; h < kCols / 32; ++h) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + c * kCols + h * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[h * 32 + j] = __uint_as_float(r[j]);
                }
                if (c == kChunks - 1) {
                    // accumulator fully read: hand it back to the MMA warp
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(a ? tempty_leader1 : tempty_leader0);
                }
                finish_chunk(c, v);
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    // ------------------------------------------------------------ teardown ----
    __syncwarp();
    tc_fence_before();
    if constexpr (CG == 2) cluster_sync_all(); else __syncthreads();
    if (warp == 0 && lane == 0 && crank == 0) {
        // No CTA may release shared memory while one of its copies is in
        // flight.  Every copy of the pair completes on the leader's full
        // barriers, so the leader waits (bounded) for the last phase of each
        // stage.  After an abort the two producers may have issued different
        // numbers of iterations (at most one ring apart): phases only the peer
        // issued are armed here with the peer's bytes; phases the leader armed
        // for both but the peer never issued are credited the peer's bytes.
        // In a run without abort both counts match and every phase is done.
        const int nl = (int)issued[0];
        const int np = CG == 2 ? (int)issued[1] : nl;
        const int lo = nl < np ? nl : np, hi = nl < np ? np : nl;
        for (int i = lo; i < hi; ++i) {
            const uint32_t b = iter_bytes(i);
            if (i >= nl) mbar_arrive_expect_tx(bar_full(i % Cfg::kStages), b);
            else mbar_complete_tx(bar_full(i % Cfg::kStages), b);
        }
        for (int i = hi - Cfg::kStages < 0 ? 0 : hi - Cfg::kStages; i < hi; ++i)
            if (!mbar_wait_bounded(bar_full(i % Cfg::kStages), (uint32_t)(i / Cfg::kStages) & 1u, p.timeout_ns))
                atomicOr(p.status, ST_TIMEOUT_PRODUCER);
    }
    __syncwarp();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, kTmemCols);
    }
    if constexpr (CG == 2) cluster_sync_all();
}

template <int CG, typename InT, typename OutT, int KIND = 0>
cudaError_t launch_impl(const CUtensorMap& tmA, const CUtensorMap& tmA2, const CUtensorMap& tmB, const CUtensorMap& tmC,
                        const TcParams& p, int grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = TcCfg<CG>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<CG, InT, OutT, KIND>, tmA, tmA2, tmB, tmC, p);
}

template <int CG, typename InT, typename OutT, int KIND = 0>
cudaError_t prepare_impl(int* max_units) {
    auto fn = gemm_tc_kernel<CG, InT, OutT, KIND>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<CG>::kSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CG, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = TcCfg<CG>::kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
    if (e != cudaSuccess) return e;
    *max_units = n;
    return cudaSuccess;
}

template <int CG>
cudaError_t launch_dt(int dtype, const CUtensorMap& tmA, const CUtensorMap& tmA2, const CUtensorMap& tmB, const CUtensorMap& tmC,
                      const TcParams& p, int grid, cudaStream_t stream) {
    switch (dtype) {
        case DT_BF16_F32: return launch_impl<CG, __nv_bfloat16, float>(tmA, tmA2, tmB, tmC, p, grid, stream);
        case DT_BF16_BF16: return launch_impl<CG, __nv_bfloat16, __nv_bfloat16>(tmA, tmA2, tmB, tmC, p, grid, stream);
        case DT_F16_F32: return launch_impl<CG, __half, float>(tmA, tmA2, tmB, tmC, p, grid, stream);
        case DT_F16_F16: return launch_impl<CG, __half, __half>(tmA, tmA2, tmB, tmC, p, grid, stream);
        // fp8 operands (the format is in the instruction descriptor); bf16 bias / scale
        case DT_E4M3_F32:
        case DT_E5M2_F32: return launch_impl<CG, __nv_bfloat16, float, 1>(tmA, tmA2, tmB, tmC, p, grid, stream);
        case DT_E4M3_BF16:
        case DT_E5M2_BF16: return launch_impl<CG, __nv_bfloat16, __nv_bfloat16, 1>(tmA, tmA2, tmB, tmC, p, grid, stream);
        // fp32 operands multiplied as tf32; bf16 bias / scale
        case DT_TF32_F32: return launch_impl<CG, __nv_bfloat16, float, 2>(tmA, tmA2, tmB, tmC, p, grid, stream);
        case DT_TF32_BF16: return launch_impl<CG, __nv_bfloat16, __nv_bfloat16, 2>(tmA, tmA2, tmB, tmC, p, grid, stream);
    }
    return cudaErrorInvalidValue;
}

template <int CG>
cudaError_t prepare_dt(int dtype, int* max_units) {
    switch (dtype) {
        case DT_BF16_F32: return prepare_impl<CG, __nv_bfloat16, float>(max_units);
        case DT_BF16_BF16: return prepare_impl<CG, __nv_bfloat16, __nv_bfloat16>(max_units);
        case DT_F16_F32: return prepare_impl<CG, __half, float>(max_units);
        case DT_F16_F16: return prepare_impl<CG, __half, __half>(max_units);
        case DT_E4M3_F32:
        case DT_E5M2_F32: return prepare_impl<CG, __nv_bfloat16, float, 1>(max_units);
        case DT_E4M3_BF16:
        case DT_E5M2_BF16: return prepare_impl<CG, __nv_bfloat16, __nv_bfloat16, 1>(max_units);
        case DT_TF32_F32: return prepare_impl<CG, __nv_bfloat16, float, 2>(max_units);
        case DT_TF32_BF16: return prepare_impl<CG, __nv_bfloat16, __nv_bfloat16, 2>(max_units);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

int tc_smem_bytes(int cta_group) {
    return cta_group == 2 ? TcCfg<2>::kSmem : TcCfg<1>::kSmem;
}

cudaError_t launch_tc_gemm(int cta_group, int dtype, const CUtensorMap& tmA, const CUtensorMap& tmB,
                           const CUtensorMap& tmC, const TcParams& p, int grid, cudaStream_t stream,
                           const CUtensorMap* tmA2) {
    const CUtensorMap& a2 = tmA2 ? *tmA2 : tmA;
    if (cta_group == 2) return launch_dt<2>(dtype, tmA, a2, tmB, tmC, p, grid, stream);
    if (cta_group == 1) return launch_dt<1>(dtype, tmA, a2, tmB, tmC, p, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t tc_prepare(int cta_group, int dtype, int* max_units) {
    if (cta_group == 2) return prepare_dt<2>(dtype, max_units);
    if (cta_group == 1) return prepare_dt<1>(dtype, max_units);
    return cudaErrorInvalidValue;
}

}  // namespace gb300
