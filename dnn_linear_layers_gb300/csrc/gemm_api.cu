// C-ABI layer: plans, argument validation, TMA tensor maps, operand packing
// and kernel dispatch.  The interface mirrors the BLAS GEMM call of
// youngju.dev "GEMM to FlashAttention" ("GEMM interface": m, n, k, alpha, lda,
// ldb, beta, ldc, transa / transb) and the handle create/use/destroy pattern of
// its cuBLAS example, for row-major operands: gemm_run is the alpha = 1,
// beta = 0 form, gemm_run_ex the general one; plan flags give transa
// (GEMM_A_KM) and transb (GEMM_B_NK).  The convolution and attention entry
// points build their tensor maps here too.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "../../include/gemm.h"
#include "internal.h"

using namespace gb300;

struct gemm_plan {
    int device = 0;
    unsigned flags = 0;
    int sm_count = 0;
    int max_pairs[kNumDtypes] = {};     // co-resident 2-CTA clusters, per operand type
    int max_singles[kNumDtypes] = {};   // co-resident single CTAs, per operand type
    int* status_dev = nullptr;
    void* workspace = nullptr;
    size_t workspace_bytes = 0;
    int forced_kernel = GEMM_KERNEL_AUTO;
    int last_kernel = -1;
    int64_t launches = 0;
    int last_cuda_error = 0;
    uint64_t timeout_ns = 1000000000ull;
    int packing = 1;
    unsigned debug = 0;
    int group_m = 0;                // 0: auto_group_m
    unsigned l2_policy = 0;
    unsigned pdl = 1;             // programmatic dependent launch of the GEMM kernels
    int debug_log = 0;            // GEMM_OPT_LOG: one line per launch on stderr
    int tail_split = 1;           // split the last wave's tiles into N-halves
    int k_snake = 1;              // serpentine k order across a worker's tiles (measured: -30% DRAM reads)
    // stream-K: fewest k-atoms per worker, 0 = off.  Off by default: measured on
    // GB300 it is within run-to-run noise or slower (FFN down 603 vs 589 us,
    // 3000 x 5000 x 2048 53.2 vs 51.8 us): the partials' traffic and the
    // reductions cost about what the balanced last wave gains.
    int sk_min_atoms = 0;
    int skinny_splits = 0;        // 0: automatic; otherwise forced split count (sweeps)
    int skinny_stages = 0;        // 0: automatic; otherwise forced ring depth (sweeps)
    // M up to which an N x K Linear layer runs on the CUDA-core GEMV.  Measured
    // on GB300 (4096 -> 14336, bf16): M = 1 0.93 of HBM against 0.80 on the
    // tensor-core small-M kernel; M = 4 0.55 against 0.79 (the CUDA cores run
    // out of issue slots for 4 tokens per weight element), so only M = 1.
    int gemv_max_m = 1;
    // largest M for the warp-MMA kernel (16-bit, N x K weight): from 9 tokens
    // its two MMAs per k-step run into the warp-level MMA rate (4096 -> 14336:
    // M = 4 19.2 us against 22.3 on the tensor-core small-M kernel, M = 16 31.3
    // against 22.7)
    int warp_mma_max_m = 8;
    int gemv_mma_blocks[2][4][8] = {};   // co-resident warp-MMA CTAs per SM: [groups - 1][log2 ks][dtype]
    int gemv_blocks[3][kNumDtypes] = {};   // co-resident GEMV CTAs per SM, by tokens held (1, 2, 4)
    int smem_per_sm = 0;          // shared memory of one SM (bytes)
    int smem_reserved = 0;        // shared memory the system reserves per CTA (bytes)
    cudaStream_t last_stream = nullptr;
    bool have_stream = false;
};

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;
typedef CUresult (*EncodeIm2colFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const int*, const int*, cuuint32_t, cuuint32_t,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeIm2colFn g_encode_im2col = nullptr;

int record(gemm_plan* p, cudaError_t e) {
    if (p) p->last_cuda_error = (int)e;
    return GEMM_ERR_CUDA;
}

bool get_encode() {
    if (g_encode) return true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    // optional: without it, convolutions take the explicit im2col path
    void* fn2 = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &fn2, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess && fn2 != nullptr)
        g_encode_im2col = reinterpret_cast<EncodeIm2colFn>(fn2);
    else
        cudaGetLastError();
    return true;
}

// 2-D tensor map: `inner` contiguous elements per row, `outer` rows, row pitch
// in bytes; box of box_inner x box_outer elements, 128-byte swizzle, zero fill
// out of bounds.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
              uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer) {
    cuuint64_t gdim[2] = {inner, outer};
    cuuint64_t gstride[1] = {pitch_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, dt, 2, const_cast<void*>(ptr), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// MN-major operand of 16-bit elements (K x N B, K x M A; mn a multiple of 64)
// seen as [mn / 64][k][64]: one box of `chunks` 64-column chunks x 64 k-rows is
// the same shared-memory image as `chunks` 2-D boxes of 64 x 64 placed 8 KB
// apart, in one copy instead of `chunks` (the chunk stride, 128 bytes, is
// smaller than the row pitch; columns past mn are never addressed because mn
// is a multiple of 64, and chunks past the end read as zero).
bool make_map_mn_chunks(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t mn, uint64_t k,
                        uint64_t pitch_bytes, uint32_t chunks) {
    cuuint64_t gdim[3] = {64, k, mn / 64};
    cuuint64_t gstride[2] = {pitch_bytes, 128};
    cuuint32_t box[3] = {64, 64, chunks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, dt, 3, const_cast<void*>(ptr), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D tensor map over a [n2][n1][n0] row-major tensor of 16-bit elements: boxes
// of 64 x 128 x 1 elements, 128-byte swizzle, zero fill past the ends.
bool make_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t n0, uint64_t n1, uint64_t n2) {
    cuuint64_t gdim[3] = {n0, n1, n2};
    cuuint64_t gstride[2] = {n0 * 2, n0 * n1 * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, dt, 3, const_cast<void*>(ptr), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}


// A operand of an implicit-GEMM convolution: NHWC activations read through an
// im2col tensor map (stride 1, square filter, C a multiple of TC_BK).
struct ConvA {
    const void* x;
    int64_t Nb, H, W, C;
    int R, S, pad;
    bool pool = false;     // fused 2 x 2 max-pool: tiles of two output rows x 64 columns
    void* pool_y = nullptr;
    int64_t pool_ldy = 0;
};

// im2col tensor map over x (Nb x H x W x C): tiles of TC_BM consecutive output
// pixels x TC_BK channels, 128-byte swizzle.  The bounding box holds the
// top-left pixels of the filter windows walked: from -pad to (dim - 1) + pad -
// (filter - 1) in W and H.  For the fused max-pool, `rows` 1 / 2 gives the
// maps of the top / bottom rows of the row pairs: 64 pixels per box, two rows
// per step in H, the bottom map's box one row lower.  Corner arrays run W, H.
bool make_im2col_map(CUtensorMap* m, CUtensorMapDataType dt, const ConvA& c, int rows = 0) {
    if (!g_encode_im2col) return false;
    cuuint64_t gdim[4] = {(cuuint64_t)c.C, (cuuint64_t)c.W, (cuuint64_t)c.H, (cuuint64_t)c.Nb};
    cuuint64_t gstride[3] = {(cuuint64_t)c.C * 2, (cuuint64_t)(c.W * c.C * 2), (cuuint64_t)(c.H * c.W * c.C * 2)};
    const int oh_last = (int)(c.H + 2 * c.pad - c.R);                // last output row
    int lower[2] = {-c.pad, -c.pad};
    int upper[2] = {c.pad - (c.S - 1), c.pad - (c.R - 1)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (rows == 1) {          // top rows 0, 2, .., OH - 2
        upper[1] = (oh_last - 1 - c.pad) - (int)(c.H - 1);
        estr[2] = 2;
    } else if (rows == 2) {   // bottom rows 1, 3, .., OH - 1
        lower[1] = 1 - c.pad;
        upper[1] = (oh_last - c.pad) - (int)(c.H - 1);
        estr[2] = 2;
    }
    const cuuint32_t pixels = rows ? 64 : TC_BM;
    CUresult r = g_encode_im2col(m, dt, 4, const_cast<void*>(c.x), gdim, gstride, lower, upper, TC_BK, pixels, estr,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Device block owned by a plan: the status word, then the stream-K arrival
// counters (zero between launches).
constexpr size_t kStatusBlockBytes = 16384;
constexpr int kSkCounterOffset = 64;                                  // ints
constexpr int64_t kSkMaxTiles = (int64_t)(kStatusBlockBytes / 4 - kSkCounterOffset) / 8;

// Stream-K split of a persistent launch of T >= U tiles on U workers with
// nkb k-atoms per tile: the T mod U tiles of the last, partial wave are cut
// into equal ranges of atoms over W <= U workers, at least min_atoms each, so
// every worker carries the same number of atoms; the split pieces run first
// and their reductions overlap the whole tiles that follow.  A grid of fewer
// than U tiles is not split: measured on GB300, the reductions at the end of
// such a launch (2048^3: 29 us against 17.4 us unsplit) cost more than the
// balance gains.  maxc is the most workers sharing one tile; no split
// (tiles = 0) when no tile would be shared.
struct SkSplit { int64_t tiles = 0, workers = 0, maxc = 0; };
SkSplit plan_stream_k(int64_t T, int64_t U, int64_t nkb, int64_t min_atoms) {
    SkSplit sk;
    if (min_atoms <= 0 || U < 2 || nkb < 1 || T < U) return sk;
    const int64_t Tsk = T % U;
    if (Tsk == 0 || Tsk > kSkMaxTiles) return sk;
    const int64_t A = Tsk * nkb;
    int64_t W = A / min_atoms;
    if (W > U) W = U;
    if (W < 2) return sk;
    int64_t maxc = 1;
    for (int64_t t = 0; t < Tsk; ++t) {
        const int64_t wf = ((t * nkb + 1) * W - 1) / A, wl = ((t + 1) * nkb * W - 1) / A;
        if (wl - wf + 1 > maxc) maxc = wl - wf + 1;
    }
    if (maxc < 2) return sk;
    sk.tiles = Tsk; sk.workers = W; sk.maxc = maxc;
    return sk;
}

bool in_is_bf16(int dtype) { return dtype == DT_BF16_F32 || dtype == DT_BF16_BF16; }
int in_bytes(int dtype) { return dtype_is_fp8(dtype) ? 1 : (dtype_is_tf32(dtype) ? 4 : 2); }
int out_bytes(int dtype) {
    return (dtype == DT_BF16_F32 || dtype == DT_F16_F32 || dtype == DT_E4M3_F32 || dtype == DT_E5M2_F32 ||
            dtype == DT_TF32_F32) ? 4 : 2;
}
CUtensorMapDataType in_map_type(int dtype) {
    if (dtype_is_tf32(dtype)) return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;   // fp32 bits, read by the MMA as tf32
    if (dtype_is_fp8(dtype)) return CU_TENSOR_MAP_DATA_TYPE_UINT8;   // bytes, read by the MMA as e4m3 / e5m2
    return in_is_bf16(dtype) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}
CUtensorMapDataType out_map_type(int dtype) {
    if (out_bytes(dtype) == 4) return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    return dtype == DT_F16_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

uint32_t make_idesc(int dtype, bool b_mn_major, int mma_m, int mma_n, bool a_mn_major = false) {
    // operand format: kind::f16 bf16 = 1 / fp16 = 0; kind::f8f6f4 e5m2 = 1 / e4m3 = 0;
    // kind::tf32 tf32 = 2
    const uint32_t ab = dtype_is_tf32(dtype) ? 2u
                      : (in_is_bf16(dtype) || dtype == DT_E5M2_F32 || dtype == DT_E5M2_BF16) ? 1u : 0u;
    return (1u << 4)                       // accumulator fp32
         | (ab << 7) | (ab << 10)          // A and B formats
         | ((a_mn_major ? 1u : 0u) << 15)  // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)  // B major-ness
         | ((uint32_t)(mma_n >> 3) << 17)
         | ((uint32_t)(mma_m >> 4) << 24);
}

struct DeviceGuard {
    int prev = -1;
    bool changed = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) changed = (cudaSetDevice(dev) == cudaSuccess);
    }
    ~DeviceGuard() {
        if (changed) cudaSetDevice(prev);
    }
};

int ensure_workspace(gemm_plan* p, size_t bytes) {
    if (bytes <= p->workspace_bytes) return GEMM_OK;
    if (p->workspace) {
        if (p->have_stream) cudaStreamSynchronize(p->last_stream);
        cudaFree(p->workspace);
        p->workspace = nullptr;
        p->workspace_bytes = 0;
    }
    const size_t want = (size_t)round_up((int64_t)bytes, 1 << 20);
    cudaError_t e = cudaMalloc(&p->workspace, want);
    if (e != cudaSuccess) {
        p->workspace = nullptr;
        p->last_cuda_error = (int)e;
        cudaGetLastError();
        return GEMM_ERR_NO_MEMORY;
    }
    p->workspace_bytes = want;
    return GEMM_OK;
}

// Number of trailing tiles to run as two N-halves.  With items dealt round
// robin to `units` persistent workers (whole tiles first, then halves), the
// busiest worker carries ceil((T - t) / U) + ceil((T + t) / U) half-tiles;
// pick the smallest t that minimises it (0 when splitting does not help).
int64_t tail_split(int64_t T, int64_t U, int enabled) {
    if (!enabled || U <= 0 || T <= U) return 0;
    int64_t best_t = 0, best = 2 * ((T + U - 1) / U);
    const int64_t lim = T < 2 * U ? T : 2 * U;
    for (int64_t t = 1; t <= lim; ++t) {
        const int64_t ms = (T - t + U - 1) / U + (T + t + U - 1) / U;
        if (ms < best) { best = ms; best_t = t; }
    }
    return best_t;
}

// Skinny-M launch: feature tiles of 128 weight rows, split-K over a cluster of
// S CTAs chosen so the whole grid is resident at once.
int run_skinny(gemm_plan* p, int64_t M, int64_t N, int64_t K, const void* X, int64_t ldx, const void* W,
               int64_t ldw, const void* bias, void* Y, int64_t ldy, uint32_t epi, const EpiArgs& ex, int dtype,
               bool w_nk, CUtensorMapDataType in_dt, cudaStream_t stream) {
    const int mpad = (int)round_up(M, 16);
    const int tmem_cols = mpad <= 32 ? 32 : (mpad <= 64 ? 64 : 128);
    const int64_t n_tiles = (N + 127) / 128;
    const int es = in_bytes(dtype);                   // 2, or 1 for fp8 (N x K W only)
    const int kbk = 128 / es;                         // elements per 128-byte k-block row
    const int64_t nkb = (K + kbk - 1) / kbk;
    if (n_tiles > INT32_MAX / 8) return GEMM_ERR_UNSUPPORTED;
    // Bandwidth follows the weight bytes in flight, and only resident CTAs have
    // loads in flight.  Candidates (splits S <= 8, ring depth 3..4, or 2 for an
    // unsplit K) are kept when the whole grid fits on the SMs with 20% headroom
    // for placing clusters inside GPCs; the one with the most weight bytes in
    // flight wins, ties going to more CTAs.  (Measured on GB300: grids at the
    // residency limit fall into a second wave, and 16-CTA clusters were slower.)
    const int64_t stage_bytes = 16384 + (int64_t)mpad * 128;
    int S = 1, stages = 2;
    int64_t best = -1;
    for (int cand = 8; cand >= 1; cand /= 2) {
        if (cand > nkb && cand > 1) continue;
        if (p->skinny_splits && cand != p->skinny_splits) continue;
        const int64_t ctas = n_tiles * cand;
        const int64_t kb_per_slice = nkb / cand;
        // rings deeper than four stages earn nothing (below) and measured slower
        // (M = 1 and 16 at 4096 -> 14336: 2 x 4 beats 2 x 6 by 2%): the search
        // starts at four unless a depth is forced
        for (int st = p->skinny_stages ? 8 : 4; st >= 2; --st) {
            if (p->skinny_stages && st != p->skinny_stages) continue;
            if (st < 3 && !p->skinny_stages && cand > 1) continue;
            const int64_t smem = skinny_smem_bytes(mpad, st);
            if (smem > 227 * 1024) continue;
            int64_t per_sm = p->smem_per_sm / (smem + p->smem_reserved);
            if (per_sm > kSkinnyMaxCtasPerSm) per_sm = kSkinnyMaxCtasPerSm;   // registers
            if (per_sm > 512 / tmem_cols) per_sm = 512 / tmem_cols;
            if (ctas * 10 > (int64_t)p->sm_count * per_sm * 8) continue;   // not resident with headroom
            // depth beyond four stages earns nothing: more CTAs beat a deeper ring
            int64_t depth = st < kb_per_slice ? st : kb_per_slice;
            if (depth > 4) depth = 4;
            const int64_t score = ctas * depth;
            if (score > best) { best = score; S = cand; stages = st; }
            break;
        }
    }
    if (best < 0) {   // nothing resident in one wave: one slice per tile, shallow ring, several waves
        S = p->skinny_splits ? (int)(p->skinny_splits <= nkb ? p->skinny_splits : 1) : 1;
        stages = p->skinny_stages ? p->skinny_stages : 3;
    }
    CUtensorMap tmW, tmX;
    const bool okw = w_nk ? make_map(&tmW, in_dt, W, (uint64_t)K, (uint64_t)N, (uint64_t)ldw * es, kbk, 128)
                          : make_map(&tmW, in_dt, W, (uint64_t)N, (uint64_t)K, (uint64_t)ldw * es, kbk, kbk);
    if (!okw) return GEMM_ERR_CUDA;
    if (!make_map(&tmX, in_dt, X, (uint64_t)K, (uint64_t)M, (uint64_t)ldx * es, kbk, (uint32_t)mpad))
        return GEMM_ERR_CUDA;
    SkinnyParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.M = (int32_t)M; sp.N = (int32_t)N; sp.K = (int32_t)K;
    sp.mpad = mpad; sp.stages = stages;
    sp.w_prefetch = (p->pdl && (p->flags & GEMM_B_CONST)) ? 1u : 0u;
    sp.pdl = p->pdl; sp.splits = S; sp.num_k_blocks = (int32_t)nkb; sp.tmem_cols = tmem_cols;
    sp.epi = epi;
    sp.ex = ex;
    // A = W (128 features; MN-major when stored K x N), B = X (mpad tokens, K-major)
    sp.idesc = make_idesc(dtype, false, 128, mpad, !w_nk);
    sp.w_mn_major = w_nk ? 0u : 1u;
    sp.bias = bias;
    sp.Y = Y; sp.ldy = ldy;
    sp.status = p->status_dev;
    sp.timeout_ns = p->timeout_ns;
    if (p->debug_log)
        std::fprintf(stderr, "[gemm] skinny M=%lld N=%lld K=%lld mpad=%d tiles=%lld splits=%d stages=%d smem=%d "
                     "prefetch=%u pdl=%u\n", (long long)M, (long long)N, (long long)K, mpad, (long long)n_tiles, S,
                     stages, skinny_smem_bytes(mpad, stages), sp.w_prefetch, sp.pdl);
    cudaError_t e = launch_skinny(dtype, tmW, tmX, sp, (int)(n_tiles * S), stream);
    if (e != cudaSuccess) return record(p, e);
    p->launches += 1;
    return GEMM_OK;
}

// GEMV launch (M <= 4, W stored N x K): the rows of W split evenly over a
// grid that is resident at once.
int run_gemv(gemm_plan* p, int64_t M, int64_t N, int64_t K, const void* X, int64_t ldx, const void* W,
             int64_t ldw, const void* bias, void* Y, int64_t ldy, uint32_t epi, const EpiArgs& ex, int dtype,
             cudaStream_t stream) {
    const int mt = gemv_tokens_held((int)M);
    const int bps = p->gemv_blocks[mt == 1 ? 0 : (mt == 2 ? 1 : 2)][dtype];
    if (mt == 0 || bps < 1) return GEMM_ERR_UNSUPPORTED;
    const int warps = kGemvThreads / 32;
    int64_t grid = (int64_t)p->sm_count * bps;
    const int64_t need = (N + warps - 1) / warps;   // one row per warp at least
    if (grid > need) grid = need;
    GemvParams gp;
    std::memset(&gp, 0, sizeof(gp));
    gp.M = (int32_t)M; gp.N = (int32_t)N; gp.K = (int32_t)K;
    gp.X = X; gp.ldx = ldx; gp.W = W; gp.ldw = ldw;
    gp.bias = bias; gp.Y = Y; gp.ldy = ldy;
    gp.epi = epi; gp.ex = ex;
    gp.pdl = p->pdl;
    gp.w_prefetch = (p->pdl && (p->flags & GEMM_B_CONST)) ? 1u : 0u;
    if (p->debug_log)
        std::fprintf(stderr, "[gemm] gemv M=%lld N=%lld K=%lld tokens=%d grid=%lld prefetch=%u pdl=%u\n",
                     (long long)M, (long long)N, (long long)K, mt, (long long)grid, gp.w_prefetch, gp.pdl);
    cudaError_t e = launch_gemv(dtype, gp, (int)grid, stream);
    if (e != cudaSuccess) return record(p, e);
    p->launches += 1;
    return GEMM_OK;
}

// Warp-MMA small-M kernel.  k-slices per row group: the fewest (1, 2, 4, 8)
// that give every warp resident on the GPU a (row group, slice) unit, so the
// whole grid streams at once; each slice keeps at least 256 k.
int run_gemv_mma(gemm_plan* p, int64_t M, int64_t N, int64_t K, const void* X, int64_t ldx, const void* W,
                 int64_t ldw, const void* bias, void* Y, int64_t ldy, uint32_t epi, const EpiArgs& ex, int dtype,
                 cudaStream_t stream) {
    const int nh = gemv_mma_groups((int)M);
    if (nh == 0 || dtype > DT_E5M2_BF16) return GEMM_ERR_UNSUPPORTED;
    const int64_t groups = (N + 15) / 16;
    const int warps = kGemvThreads / 32;
    int j = 0;
    for (; j < 3; ++j) {
        const int64_t resident = (int64_t)p->sm_count * p->gemv_mma_blocks[nh - 1][j][dtype] * warps;
        if (groups * (1 << j) >= resident || K < 256 * (2 << j)) break;
    }
    const int ks = 1 << j;
    const int bps = p->gemv_mma_blocks[nh - 1][j][dtype];
    if (bps < 1) return GEMM_ERR_UNSUPPORTED;
    int64_t grid = (int64_t)p->sm_count * bps;
    const int64_t need = (groups + warps / ks - 1) / (warps / ks);
    if (grid > need) grid = need;
    GemvParams gp;
    std::memset(&gp, 0, sizeof(gp));
    gp.M = (int32_t)M; gp.N = (int32_t)N; gp.K = (int32_t)K;
    gp.X = X; gp.ldx = ldx; gp.W = W; gp.ldw = ldw;
    gp.bias = bias; gp.Y = Y; gp.ldy = ldy;
    gp.epi = epi; gp.ex = ex;
    gp.pdl = p->pdl;
    gp.w_prefetch = (p->pdl && (p->flags & GEMM_B_CONST)) ? 1u : 0u;
    if (p->debug_log)
        std::fprintf(stderr, "[gemm] warp-mma M=%lld N=%lld K=%lld groups=%lld ks=%d grid=%lld prefetch=%u pdl=%u\n",
                     (long long)M, (long long)N, (long long)K, (long long)groups, ks, (long long)grid, gp.w_prefetch,
                     gp.pdl);
    cudaError_t e = launch_gemv_mma(dtype, ks, gp, (int)grid, stream);
    if (e != cudaSuccess) return record(p, e);
    p->launches += 1;
    return GEMM_OK;
}

}  // namespace

extern "C" {

int gemm_validate(unsigned flags, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                  int64_t ldb, const void* bias, const void* C, int64_t ldc, int epilogue, int dtype) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (epilogue < GEMM_EPI_NONE || epilogue > GEMM_EPI_BIAS_RELU) return GEMM_ERR_INVALID_ARG;
    if (dtype < GEMM_BF16_F32OUT || dtype > GEMM_TF32_BF16OUT) return GEMM_ERR_INVALID_ARG;
    if (flags & ~(GEMM_B_NK | GEMM_B_CONST | GEMM_A_KM)) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (C == nullptr || ldc < N) return GEMM_ERR_INVALID_ARG;
    if ((epilogue & GEMM_EPI_BIAS) && bias == nullptr) return GEMM_ERR_INVALID_ARG;
    if (K > 0) {
        if (A == nullptr || B == nullptr) return GEMM_ERR_INVALID_ARG;
        if (lda < ((flags & GEMM_A_KM) ? M : K)) return GEMM_ERR_INVALID_ARG;
        if (ldb < ((flags & GEMM_B_NK) ? K : N)) return GEMM_ERR_INVALID_ARG;
    }
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
    // every pointer on a boundary of its element size (bias: bf16 for the fp8
    // and tf32 types)
    const uintptr_t ie = (uintptr_t)in_bytes(dtype), oe = (uintptr_t)out_bytes(dtype);
    const uintptr_t ve = (dtype_is_fp8(dtype) || dtype_is_tf32(dtype)) ? 2u : ie;
    if (reinterpret_cast<uintptr_t>(C) % oe) return GEMM_ERR_INVALID_ARG;
    if (bias && reinterpret_cast<uintptr_t>(bias) % ve) return GEMM_ERR_INVALID_ARG;
    if (K > 0 && (reinterpret_cast<uintptr_t>(A) % ie || reinterpret_cast<uintptr_t>(B) % ie))
        return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

int gemm_plan_create(gemm_plan_t* plan, int device, unsigned flags) {
    if (plan == nullptr || device < 0 || (flags & ~(GEMM_B_NK | GEMM_B_CONST | GEMM_A_KM)))
        return GEMM_ERR_INVALID_ARG;
    int ndev = 0;
    cudaError_t e = cudaGetDeviceCount(&ndev);
    if (e != cudaSuccess) { cudaGetLastError(); return GEMM_ERR_CUDA; }
    if (device >= ndev) return GEMM_ERR_INVALID_ARG;
    if (!get_encode()) return GEMM_ERR_CUDA;
    gemm_plan* p = new (std::nothrow) gemm_plan();
    if (!p) return GEMM_ERR_NO_MEMORY;
    p->device = device;
    p->flags = flags;
    DeviceGuard g(device);
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, device);
    if (e != cudaSuccess) { delete p; return GEMM_ERR_CUDA; }
    if (prop.major * 10 + prop.minor < 100) { delete p; return GEMM_ERR_UNSUPPORTED; }
    p->sm_count = prop.multiProcessorCount;
    // co-residency of the tensor-core kernels, kept per operand type (each type
    // is its own instantiation, with its own register count)
    for (int dt = 0; dt < kNumDtypes; ++dt) {
        int n2 = 0, n1 = 0;
        e = tc_prepare(2, dt, &n2);
        if (e == cudaSuccess) e = tc_prepare(1, dt, &n1);
        if (e != cudaSuccess) { cudaGetLastError(); delete p; return GEMM_ERR_CUDA; }
        if (n2 < 1 || n1 < 1) { delete p; return GEMM_ERR_UNSUPPORTED; }
        p->max_pairs[dt] = n2;
        p->max_singles[dt] = n1;
    }
    for (int dt = 0; dt < 4; ++dt) {
        e = attention_prepare(dt);
        if (e != cudaSuccess) { cudaGetLastError(); delete p; return GEMM_ERR_CUDA; }
    }
    for (int dt = 0; dt <= DT_E5M2_BF16; ++dt) {
        e = skinny_prepare(dt);
        if (e != cudaSuccess) { cudaGetLastError(); delete p; return GEMM_ERR_CUDA; }
        for (int i = 0; i < 3; ++i) {
            e = gemv_prepare(1 << i, dt, &p->gemv_blocks[i][dt]);
            if (e != cudaSuccess) { cudaGetLastError(); delete p; return GEMM_ERR_CUDA; }
        }
        for (int nh = 1; nh <= 2; ++nh)
            for (int j = 0; j < 4; ++j) {
                e = gemv_mma_prepare(nh, 1 << j, dt, &p->gemv_mma_blocks[nh - 1][j][dt]);
                if (e != cudaSuccess) { cudaGetLastError(); delete p; return GEMM_ERR_CUDA; }
            }
    }
    p->smem_per_sm = (int)prop.sharedMemPerMultiprocessor;
    p->smem_reserved = (int)prop.reservedSharedMemPerBlock;
    e = cudaMalloc(&p->status_dev, kStatusBlockBytes);
    if (e != cudaSuccess) { delete p; return GEMM_ERR_NO_MEMORY; }
    e = cudaMemset(p->status_dev, 0, kStatusBlockBytes);
    if (e != cudaSuccess) { cudaFree(p->status_dev); delete p; return GEMM_ERR_CUDA; }
    *plan = p;
    return GEMM_OK;
}

int gemm_plan_destroy(gemm_plan_t p) {
    if (!p) return GEMM_OK;
    DeviceGuard g(p->device);
    if (p->have_stream) cudaStreamSynchronize(p->last_stream);
    if (p->workspace) cudaFree(p->workspace);
    if (p->status_dev) cudaFree(p->status_dev);
    delete p;
    return GEMM_OK;
}

int gemm_plan_set_kernel(gemm_plan_t p, int kernel) {
    if (!p || kernel < GEMM_KERNEL_AUTO || kernel > GEMM_KERNEL_WARP_MMA) return GEMM_ERR_INVALID_ARG;
    p->forced_kernel = kernel;
    return GEMM_OK;
}

int gemm_plan_last_kernel(gemm_plan_t p) { return p ? p->last_kernel : -1; }
int64_t gemm_plan_launch_count(gemm_plan_t p) { return p ? p->launches : -1; }
int gemm_plan_last_cuda_error(gemm_plan_t p) { return p ? p->last_cuda_error : 0; }
int64_t gemm_plan_workspace_bytes(gemm_plan_t p) { return p ? (int64_t)p->workspace_bytes : -1; }

int gemm_plan_set_timeout_ns(gemm_plan_t p, uint64_t ns) {
    if (!p || ns == 0) return GEMM_ERR_INVALID_ARG;
    p->timeout_ns = ns;
    return GEMM_OK;
}

int gemm_plan_set_packing(gemm_plan_t p, int enabled) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    p->packing = enabled ? 1 : 0;
    return GEMM_OK;
}

int gemm_plan_set_debug(gemm_plan_t p, unsigned flags) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    p->debug = flags;
    return GEMM_OK;
}

int gemm_plan_set_option(gemm_plan_t p, int option, int64_t v) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    const bool b01 = v == 0 || v == 1;
    switch (option) {
        case GEMM_OPT_GROUP_M:
            if (v < 0 || v > 1024) return GEMM_ERR_INVALID_ARG;
            p->group_m = (int)v; return GEMM_OK;
        case GEMM_OPT_TAIL_SPLIT:
            if (!b01) return GEMM_ERR_INVALID_ARG;
            p->tail_split = (int)v; return GEMM_OK;
        case GEMM_OPT_K_SNAKE:
            if (!b01) return GEMM_ERR_INVALID_ARG;
            p->k_snake = (int)v; return GEMM_OK;
        case GEMM_OPT_PDL:
            if (!b01) return GEMM_ERR_INVALID_ARG;
            p->pdl = (unsigned)v; return GEMM_OK;
        case GEMM_OPT_L2_POLICY:
            if (v < 0 || v > 2) return GEMM_ERR_INVALID_ARG;
            p->l2_policy = (unsigned)v; return GEMM_OK;
        case GEMM_OPT_SKINNY_SPLITS:
            if (v != 0 && v != 1 && v != 2 && v != 4 && v != 8) return GEMM_ERR_INVALID_ARG;
            p->skinny_splits = (int)v; return GEMM_OK;
        case GEMM_OPT_SKINNY_STAGES:
            if (v != 0 && (v < 2 || v > 8)) return GEMM_ERR_INVALID_ARG;
            p->skinny_stages = (int)v; return GEMM_OK;
        case GEMM_OPT_LOG:
            if (!b01) return GEMM_ERR_INVALID_ARG;
            p->debug_log = (int)v; return GEMM_OK;
        case GEMM_OPT_GEMV_MAX_M:
            if (v < 0 || v > kGemvMaxM) return GEMM_ERR_INVALID_ARG;
            p->gemv_max_m = (int)v; return GEMM_OK;
        case GEMM_OPT_WARP_MMA_MAX_M:
            if (v < 0 || v > kWarpMmaMaxM) return GEMM_ERR_INVALID_ARG;
            p->warp_mma_max_m = (int)v; return GEMM_OK;
        case GEMM_OPT_STREAM_K:
            if (v < 0 || v > 4096) return GEMM_ERR_INVALID_ARG;
            p->sk_min_atoms = (int)v; return GEMM_OK;
    }
    return GEMM_ERR_INVALID_ARG;
}

int gemm_plan_get_option(gemm_plan_t p, int option, int64_t* v) {
    if (!p || !v) return GEMM_ERR_INVALID_ARG;
    switch (option) {
        case GEMM_OPT_GROUP_M: *v = p->group_m; return GEMM_OK;
        case GEMM_OPT_TAIL_SPLIT: *v = p->tail_split; return GEMM_OK;
        case GEMM_OPT_K_SNAKE: *v = p->k_snake; return GEMM_OK;
        case GEMM_OPT_PDL: *v = p->pdl; return GEMM_OK;
        case GEMM_OPT_L2_POLICY: *v = p->l2_policy; return GEMM_OK;
        case GEMM_OPT_SKINNY_SPLITS: *v = p->skinny_splits; return GEMM_OK;
        case GEMM_OPT_SKINNY_STAGES: *v = p->skinny_stages; return GEMM_OK;
        case GEMM_OPT_LOG: *v = p->debug_log; return GEMM_OK;
        case GEMM_OPT_GEMV_MAX_M: *v = p->gemv_max_m; return GEMM_OK;
        case GEMM_OPT_WARP_MMA_MAX_M: *v = p->warp_mma_max_m; return GEMM_OK;
        case GEMM_OPT_STREAM_K: *v = p->sk_min_atoms; return GEMM_OK;
    }
    return GEMM_ERR_INVALID_ARG;
}

int gemm_plan_status(gemm_plan_t p) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    DeviceGuard g(p->device);
    cudaError_t e = p->have_stream ? cudaStreamSynchronize(p->last_stream) : cudaDeviceSynchronize();
    if (e != cudaSuccess) return record(p, e);
    int st = 0;
    e = cudaMemcpy(&st, p->status_dev, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return record(p, e);
    if (st != 0) {
        // an aborted launch may leave stream-K arrival counters behind: clear
        // them with the status word
        cudaMemset(p->status_dev, 0, kStatusBlockBytes);
        cudaDeviceSynchronize();
        return GEMM_ERR_DEVICE_TIMEOUT;
    }
    return GEMM_OK;
}

const char* gemm_strerror(int code) {
    switch (code) {
        case GEMM_OK: return "ok";
        case GEMM_ERR_INVALID_ARG: return "invalid argument";
        case GEMM_ERR_ALIGNMENT: return "operand not 16-byte aligned and packing disabled";
        case GEMM_ERR_UNSUPPORTED: return "unsupported configuration";
        case GEMM_ERR_CUDA: return "CUDA call failed";
        case GEMM_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case GEMM_ERR_NO_MEMORY: return "out of memory";
        default: return "unknown error";
    }
}

int gemm_im2col(const void* x, int64_t Nb, int64_t H, int64_t W, int64_t C, int R, int S, int pad, int stride,
                void* out, int64_t ld_out, int elem_bytes, void* stream) {
    if (Nb < 0 || H < 0 || W < 0 || C < 0 || R < 1 || S < 1 || pad < 0 || stride < 1) return GEMM_ERR_INVALID_ARG;
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4) return GEMM_ERR_INVALID_ARG;
    const int64_t OH = H + 2 * pad >= R ? (H + 2 * pad - R) / stride + 1 : 0;
    const int64_t OW = W + 2 * pad >= S ? (W + 2 * pad - S) / stride + 1 : 0;
    if (Nb == 0 || OH == 0 || OW == 0 || C == 0) return GEMM_OK;
    if (x == nullptr || out == nullptr || ld_out < (int64_t)R * S * C) return GEMM_ERR_INVALID_ARG;
    cudaError_t e = launch_im2col(x, Nb, H, W, C, R, S, pad, stride, out, ld_out, elem_bytes,
                                  reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) { cudaGetLastError(); return GEMM_ERR_CUDA; }
    return GEMM_OK;
}

}  // extern "C"

namespace {

EpiArgs plain_epilogue() {
    EpiArgs ex;
    std::memset(&ex, 0, sizeof(ex));
    ex.alpha = 1.0f;
    return ex;
}

// Epilogue flags and operands of gemm_epilogue_args_t; C is also the previous C.
int extended_epilogue(const gemm_epilogue_args_t* a, int dtype, const void* C, int64_t ldc, uint32_t* flags,
                      EpiArgs* ex) {
    *ex = plain_epilogue();
    uint32_t f = 0;
    if (a->bias) f |= EPI_BIAS;
    if (a->relu) f |= EPI_RELU;
    if (a->scale) { f |= EPI_SCALE; ex->scale = a->scale; ex->scale_vec16 = aligned16(a->scale) ? 1u : 0u; }
    if (a->alpha != 1.0f) { f |= EPI_ALPHA; ex->alpha = a->alpha; }
    if (a->beta != 0.0f) {
        if (C == nullptr) return GEMM_ERR_INVALID_ARG;
        f |= EPI_BETA;
        ex->beta = a->beta;
        ex->c_old = C;
        ex->ldc_old = ldc;
        ex->c_old_vec16 = (aligned16(C) && (ldc * out_bytes(dtype)) % 16 == 0) ? 1u : 0u;
    }
    *flags = f;
    return GEMM_OK;
}

// Validated arguments; M, N > 0.  b_nk: B is N x K.  conv: A is the im2col
// view of an activation tensor (then A and lda are unused).  a_km: A is K x M.
int run_impl(gemm_plan* p, bool b_nk, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
             int64_t ldb, const void* bias, void* C, int64_t ldc, uint32_t epi, const EpiArgs& ex, int dtype,
             cudaStream_t stream, const ConvA* conv, bool a_km = false) {
    int rc = GEMM_OK;
    cudaError_t e;

    if (K == 0) {
        e = launch_fill_epilogue(dtype, M, N, bias, epi, ex, C, ldc, stream);
        if (e != cudaSuccess) return record(p, e);
        p->launches += 1;
        p->last_kernel = GEMM_KERNEL_FILL;
        p->last_stream = stream; p->have_stream = true;
        return GEMM_OK;
    }

    // fp8 and tf32 take every operand layout (MN-major operands through the
    // instruction descriptor's major-ness bits), but no convolution
    const bool fp8 = dtype_is_fp8(dtype) || dtype_is_tf32(dtype);
    if (fp8 && conv) return GEMM_ERR_UNSUPPORTED;
    if (a_km && conv) return GEMM_ERR_UNSUPPORTED;
    // the small-M kernels take 16-bit and fp8 operands with an M x K A; the
    // CUDA-core GEMV also needs the weight stored N x K
    const bool tf32 = dtype_is_tf32(dtype);
    const bool small_ok = !conv && !tf32 && !a_km;
    // the warp-MMA kernel: 16-bit or fp8 operands, an N x K weight, M <= 16
    const bool mma_ok = small_ok && b_nk;
    int kernel = p->forced_kernel;
    if (kernel == GEMM_KERNEL_AUTO)
        kernel = (small_ok && b_nk && M <= p->gemv_max_m) ? GEMM_KERNEL_GEMV
               : (mma_ok && M <= p->warp_mma_max_m) ? GEMM_KERNEL_WARP_MMA
               : (small_ok && M <= 128) ? GEMM_KERNEL_SKINNY : GEMM_KERNEL_TC_PAIR;
    if (kernel == GEMM_KERNEL_SKINNY && (M > 128 || !small_ok)) return GEMM_ERR_UNSUPPORTED;
    if (kernel == GEMM_KERNEL_GEMV && (M > kGemvMaxM || !small_ok || !b_nk)) return GEMM_ERR_UNSUPPORTED;
    if (kernel == GEMM_KERNEL_WARP_MMA && (M > kWarpMmaMaxM || !mma_ok)) return GEMM_ERR_UNSUPPORTED;
    if (kernel != GEMM_KERNEL_TC_PAIR && kernel != GEMM_KERNEL_TC_SINGLE && kernel != GEMM_KERNEL_SKINNY &&
        kernel != GEMM_KERNEL_GEMV && kernel != GEMM_KERNEL_WARP_MMA)
        return GEMM_ERR_UNSUPPORTED;
    // both weight-streaming kernels on the CUDA-core path store C with plain stores
    const bool gemv = kernel == GEMM_KERNEL_GEMV || kernel == GEMM_KERNEL_WARP_MMA;
    const bool skinny = kernel == GEMM_KERNEL_SKINNY;
    const int cg = (kernel == GEMM_KERNEL_TC_PAIR) ? 2 : 1;
    const int kbk = 128 / in_bytes(dtype);          // elements per 128-byte k-atom row
    // persistent grid of the tensor-core kernels, and the stream-K split of its
    // last wave (not for the fused max-pool, whose epilogue pools whole tiles)
    const int64_t num_m_tiles = (M + TC_BM * cg - 1) / (TC_BM * cg), num_n_tiles = (N + TC_BN - 1) / TC_BN;
    const int64_t num_kb = (K + kbk - 1) / kbk;
    const int64_t tiles = num_m_tiles * num_n_tiles;
    const int64_t cap = cg == 2 ? p->max_pairs[dtype] : p->max_singles[dtype];
    SkSplit sk;
    if (!gemv && !skinny && !(conv && conv->pool)) sk = plan_stream_k(tiles, cap, num_kb, p->sk_min_atoms);
    const size_t sk_bytes = (size_t)(sk.tiles * sk.maxc) * 8u * 32u * (size_t)TC_BN * 4u;

    // ---- operand alignment: pack anything that breaks the TMA 16-byte rule
    const int ob = out_bytes(dtype);
    const int64_t b_rows = b_nk ? N : K, b_cols = b_nk ? K : N;
    const int64_t a_rows = a_km ? K : M, a_cols = a_km ? M : K;
    const int es = in_bytes(dtype);                 // element size of A and B
    // tf32 operands stored MN-major (K x N B, K x M A) are first transposed
    // into the workspace: the tensor cores take tf32 K-major only (MMAs with
    // an MN-major tf32 operand gave wrong sums on GB300; 16-bit and fp8
    // MN-major operands are read directly)
    const bool t_a = tf32 && a_km, t_b = tf32 && !b_nk;
    const int64_t ld_t = round_up(K, 4);            // 16-byte rows of the transposed copies
    const bool a_ok = conv || t_a || (aligned16(A) && (lda * es) % 16 == 0);
    const bool b_ok = t_b || (aligned16(B) && (ldb * es) % 16 == 0);
    // the small-M kernels store C with plain stores, and so does the
    // tensor-core epilogue when C breaks the TMA rule: any pitch is fine.  A
    // TMA store also needs the right edge of C on a 16-byte boundary: at an
    // edge inside a 16-byte granule it writes the whole granule, i.e. up to
    // 15 bytes of each row past column N (measured on GB300).
    const bool c_tma = aligned16(C) && (ldc * ob) % 16 == 0 && (N * ob) % 16 == 0;
    const bool c_direct = !skinny && !gemv && !c_tma && !(conv && conv->pool);
    const bool c_ok = skinny || gemv || c_tma || c_direct;
    const void* A_use = A; int64_t lda_use = lda;
    const void* B_use = B; int64_t ldb_use = ldb;
    void* C_use = C; int64_t ldc_use = ldc;
    float* sk_part = nullptr;
    if (!a_ok || !b_ok || !c_ok || t_a || t_b) {
        if ((!a_ok || !b_ok || !c_ok) && !p->packing) return GEMM_ERR_ALIGNMENT;
        const int64_t lda_p = round_up(a_cols, 16 / es), ldb_p = round_up(b_cols, 16 / es),
                      ldc_p = round_up(N, 16 / ob);
        const size_t a_bytes = t_a ? (size_t)round_up(M * ld_t * 4, 256)
                             : a_ok ? 0 : (size_t)round_up(a_rows * lda_p * es, 256);
        const size_t b_bytes = t_b ? (size_t)round_up(N * ld_t * 4, 256)
                             : b_ok ? 0 : (size_t)round_up(b_rows * ldb_p * es, 256);
        const size_t c_bytes = c_ok ? 0 : (size_t)round_up(M * ldc_p * ob, 256);
        rc = ensure_workspace(p, a_bytes + b_bytes + c_bytes + sk_bytes);
        if (rc != GEMM_OK) return rc;
        char* ws = static_cast<char*>(p->workspace);
        if (sk_bytes) sk_part = reinterpret_cast<float*>(ws + a_bytes + b_bytes + c_bytes);
        // MN-major tf32 operands transposed (both in one launch); from here on
        // the GEMM sees them K-major
        if (t_a || t_b) {
            TransJob ja = {}, jb = {};
            if (t_a) {
                ja = {static_cast<const uint32_t*>(A), lda, reinterpret_cast<uint32_t*>(ws), ld_t, K, M};
                A_use = ws; lda_use = ld_t; a_km = false;
            }
            if (t_b) {
                jb = {static_cast<const uint32_t*>(B), ldb, reinterpret_cast<uint32_t*>(ws + a_bytes), ld_t, K, N};
                B_use = ws + a_bytes; ldb_use = ld_t; b_nk = true;
            }
            e = t_a ? launch_transpose2(ja, jb, stream) : launch_transpose2(jb, TransJob{}, stream);
            if (e != cudaSuccess) return record(p, e);
            p->launches += 1;
        }
        // A and B packed in one launch
        PackJob ja = {}, jb = {};
        if (!a_ok) {
            ja = pack_job(A, lda, ws, lda_p, a_rows, a_cols, es);
            A_use = ws; lda_use = lda_p;
        }
        if (!b_ok) {
            jb = pack_job(B, ldb, ws + a_bytes, ldb_p, b_rows, b_cols, es);
            B_use = ws + a_bytes; ldb_use = ldb_p;
        }
        if (!a_ok || !b_ok) {
            e = launch_pack2(ja, jb, stream);
            if (e != cudaSuccess) return record(p, e);
            p->launches += 1;
        }
        if (!c_ok) { C_use = ws + a_bytes + b_bytes; ldc_use = ldc_p; }
    } else if (sk_bytes) {
        rc = ensure_workspace(p, sk_bytes);
        if (rc != GEMM_OK) return rc;
        sk_part = static_cast<float*>(p->workspace);
    }

    if (gemv) {
        rc = kernel == GEMM_KERNEL_WARP_MMA
                 ? run_gemv_mma(p, M, N, K, A_use, lda_use, B_use, ldb_use, bias, C, ldc, epi, ex, dtype, stream)
                 : run_gemv(p, M, N, K, A_use, lda_use, B_use, ldb_use, bias, C, ldc, epi, ex, dtype, stream);
        if (rc != GEMM_OK) return rc;
        p->last_kernel = kernel;
        p->last_stream = stream; p->have_stream = true;
        return GEMM_OK;
    }
    const CUtensorMapDataType in_dt = in_map_type(dtype);
    if (skinny) {
        rc = run_skinny(p, M, N, K, A_use, lda_use, B_use, ldb_use, bias, C, ldc, epi, ex, dtype, b_nk, in_dt, stream);
        if (rc != GEMM_OK) return rc;
        p->last_kernel = kernel;
        p->last_stream = stream; p->have_stream = true;
        return GEMM_OK;
    }
    const CUtensorMapDataType out_dt = out_map_type(dtype);
    // 16-bit MN-major operands whose MN extent is a multiple of 64 take one
    // copy per k-atom (measured 1.5% faster at 8192^3 with a K x N B)
    const bool a_chunks = a_km && es == 2 && M % 64 == 0;
    const bool b_chunks = !b_nk && es == 2 && N % 64 == 0;
    CUtensorMap tmA, tmA2, tmB, tmC;
    if (conv && conv->pool) {
        if (!make_im2col_map(&tmA, in_dt, *conv, 1) || !make_im2col_map(&tmA2, in_dt, *conv, 2))
            return GEMM_ERR_CUDA;
    } else if (conv) {
        if (!make_im2col_map(&tmA, in_dt, *conv)) return GEMM_ERR_CUDA;
    } else if (a_km && a_chunks) {
        if (!make_map_mn_chunks(&tmA, in_dt, A_use, (uint64_t)M, (uint64_t)K, (uint64_t)lda_use * es, TC_BM / 64))
            return GEMM_ERR_CUDA;
    } else if (a_km) {   // boxes of kbk columns of the M x K operand (128 bytes) x kbk k-rows
        if (!make_map(&tmA, in_dt, A_use, (uint64_t)M, (uint64_t)K, (uint64_t)lda_use * es, kbk, kbk))
            return GEMM_ERR_CUDA;
    } else if (!make_map(&tmA, in_dt, A_use, (uint64_t)K, (uint64_t)M, (uint64_t)lda_use * es, kbk, TC_BM)) {
        return GEMM_ERR_CUDA;
    }
    // N x K B: one box of the CTA's columns per k-block row; K x N B: boxes
    // of kbk columns (128 bytes) x kbk k-rows, or all of a CTA's 64-column
    // chunks in one box
    bool okb = b_nk     ? make_map(&tmB, in_dt, B_use, (uint64_t)K, (uint64_t)N, (uint64_t)ldb_use * es, kbk, TC_BN / cg)
             : b_chunks ? make_map_mn_chunks(&tmB, in_dt, B_use, (uint64_t)N, (uint64_t)K, (uint64_t)ldb_use * es,
                                             (uint32_t)(TC_BN / cg / 64))
                        : make_map(&tmB, in_dt, B_use, (uint64_t)N, (uint64_t)K, (uint64_t)ldb_use * es, kbk, kbk);
    if (!okb) return GEMM_ERR_CUDA;
    if (c_direct) {
        std::memset(&tmC, 0, sizeof(tmC));   // not used: the epilogue stores C itself
    } else if (!make_map(&tmC, out_dt, C_use, (uint64_t)N, (uint64_t)M, (uint64_t)ldc_use * ob, 128 / ob, 32)) {
        return GEMM_ERR_CUDA;
    }

    TcParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.M = (int32_t)M; prm.N = (int32_t)N; prm.K = (int32_t)K;
    prm.num_m_tiles = (int32_t)num_m_tiles;
    prm.num_n_tiles = (int32_t)num_n_tiles;
    prm.num_k_blocks = (int32_t)num_kb;
    prm.epi = epi;
    prm.ex = ex;
    prm.idesc = make_idesc(dtype, !b_nk, TC_BM * cg, TC_BN, a_km);
    prm.b_mn_major = b_nk ? 0u : 1u;
    prm.a_mn_major = a_km ? 1u : 0u;
    prm.a_chunks = a_chunks ? 1u : 0u;
    prm.b_chunks = b_chunks ? 1u : 0u;
    prm.bias = bias;
    prm.bias_vec16 = (bias != nullptr && aligned16(bias)) ? 1u : 0u;
    prm.status = p->status_dev;
    prm.timeout_ns = p->timeout_ns;
    prm.debug = p->debug;
    prm.l2_policy = p->l2_policy;
    prm.pdl = p->pdl;
    prm.k_snake = p->k_snake ? 1u : 0u;
    if (c_direct) {
        prm.c_direct = 1u;
        prm.c_ptr = C;
        prm.ldc = ldc;
    }
    if (conv) {
        prm.conv = 1u;
        prm.conv_cb = (int32_t)(conv->C / TC_BK);
        prm.conv_s = conv->S;
        prm.conv_pad = conv->pad;
        prm.conv_out_w = (int32_t)(conv->W + 2 * conv->pad - conv->S + 1);
        prm.conv_out_hw = (int32_t)((conv->H + 2 * conv->pad - conv->R + 1) * prm.conv_out_w);
        if (conv->pool) {
            prm.conv_pool = 1u;
            prm.pool_ph = (int32_t)((conv->H + 2 * conv->pad - conv->R + 1) / 2);
            prm.pool_rows = (int32_t)(conv->Nb * prm.pool_ph * (prm.conv_out_w / 2));
            prm.pool_y = conv->pool_y;
            prm.pool_ldy = conv->pool_ldy;
            prm.pool_vec16 = (aligned16(conv->pool_y) && (conv->pool_ldy * ob) % 16 == 0) ? 1u : 0u;
        }
    }
    if (tiles > INT32_MAX / 2) return GEMM_ERR_UNSUPPORTED;
    // workers: one per co-resident CTA (pair), fewer for small problems
    int64_t units = tiles < cap ? tiles : cap;
    prm.group_m = p->group_m ? p->group_m : auto_group_m(num_n_tiles, cap);
    if (sk.tiles) {
        if (sk.workers > units) units = sk.workers;
        prm.sk_tiles = (int32_t)sk.tiles;
        prm.sk_workers = (int32_t)sk.workers;
        prm.sk_maxc = (int32_t)sk.maxc;
        prm.sk_cnt = p->status_dev + kSkCounterOffset;
        prm.sk_part = sk_part;
        prm.num_full = (int32_t)(tiles - sk.tiles);   // the rest are whole waves
    } else if (cg == 2 && !b_nk && dtype_is_fp8(dtype)) {
        // a CTA's share of a half tile, 64 fp8 columns, is narrower than one
        // 128-byte box of a K x N B: whole tiles only
        prm.num_full = (int32_t)tiles;
    } else {
        prm.num_full = (int32_t)(tiles - tail_split(tiles, units, p->tail_split));
    }
    prm.idesc_half = make_idesc(dtype, !b_nk, TC_BM * cg, TC_BN / 2, a_km);
    if (p->debug_log)
        std::fprintf(stderr, "[gemm] tc cta_group=%d conv=%u M=%lld N=%lld K=%lld tiles=%lld sk=%lldx%lld/%lld "
                     "split=%lld grid=%lld packed=%d%d%d\n",
                     cg, prm.conv, (long long)M, (long long)N, (long long)K, (long long)tiles, (long long)sk.tiles,
                     (long long)sk.maxc, (long long)sk.workers, (long long)(tiles - sk.tiles - prm.num_full),
                     (long long)(units * cg), A_use != A, B_use != B, C_use != C);
    e = launch_tc_gemm(cg, dtype, tmA, tmB, tmC, prm, (int)(units * cg), stream,
                       (conv && conv->pool) ? &tmA2 : nullptr);
    if (e != cudaSuccess) return record(p, e);
    p->launches += 1;

    if (C_use != C) {
        e = launch_copy2d(C_use, ldc_use, C, ldc, M, N, ob, stream);
        if (e != cudaSuccess) return record(p, e);
        p->launches += 1;
    }
    p->last_kernel = kernel;
    p->last_stream = stream; p->have_stream = true;
    return GEMM_OK;
}

}  // namespace

extern "C" {

int gemm_run(gemm_plan_t p, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
             int64_t ldb, const void* bias, void* C, int64_t ldc, int epilogue, int dtype, void* stream_v) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    int rc = gemm_validate(p->flags, M, N, K, A, lda, B, ldb, bias, C, ldc, epilogue, dtype);
    if (rc != GEMM_OK) return rc;
    if (M == 0 || N == 0) return GEMM_OK;
    DeviceGuard g(p->device);
    return run_impl(p, (p->flags & GEMM_B_NK) != 0, M, N, K, A, lda, B, ldb, bias, C, ldc, (uint32_t)epilogue,
                    plain_epilogue(), dtype, reinterpret_cast<cudaStream_t>(stream_v), nullptr,
                    (p->flags & GEMM_A_KM) != 0);
}

int gemm_run_ex(gemm_plan_t p, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                int64_t ldb, void* C, int64_t ldc, const gemm_epilogue_args_t* epi, int dtype, void* stream_v) {
    if (!p || !epi) return GEMM_ERR_INVALID_ARG;
    uint32_t flags = 0;
    EpiArgs ex;
    int rc = extended_epilogue(epi, dtype, C, ldc, &flags, &ex);
    if (rc != GEMM_OK) return rc;
    rc = gemm_validate(p->flags, M, N, K, A, lda, B, ldb, epi->bias, C, ldc, (int)(flags & 3u), dtype);
    if (rc != GEMM_OK) return rc;
    if (M == 0 || N == 0) return GEMM_OK;
    DeviceGuard g(p->device);
    return run_impl(p, (p->flags & GEMM_B_NK) != 0, M, N, K, A, lda, B, ldb, epi->bias, C, ldc, flags, ex, dtype,
                    reinterpret_cast<cudaStream_t>(stream_v), nullptr, (p->flags & GEMM_A_KM) != 0);
}

int gemm_conv2d(gemm_plan_t p, int64_t Nb, int64_t H, int64_t W, int64_t C, int64_t Cout, int R, int S, int pad,
                const void* x, const void* w, void* y, int64_t ldy, const gemm_epilogue_args_t* epi_args, int dtype,
                void* stream_v) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    uint32_t epi = 0;
    EpiArgs ex = plain_epilogue();
    const void* bias = nullptr;
    if (epi_args) {
        int rc0 = extended_epilogue(epi_args, dtype, y, ldy, &epi, &ex);
        if (rc0 != GEMM_OK) return rc0;
        bias = epi_args->bias;
    }
    const int epilogue = (int)(epi & 3u);
    if (Nb < 0 || H < 0 || W < 0 || C < 0 || Cout < 0 || R < 1 || S < 1 || pad < 0) return GEMM_ERR_INVALID_ARG;
    const int64_t OH = H + 2 * pad - R + 1, OW = W + 2 * pad - S + 1;
    if (OH < 0 || OW < 0) return GEMM_ERR_INVALID_ARG;
    if (dtype_is_fp8(dtype) || dtype_is_tf32(dtype)) return GEMM_ERR_UNSUPPORTED;
    const int64_t M = Nb * OH * OW, N = Cout, K = (int64_t)R * S * C;
    // the weights w[f][r][s][c] are the N x K operand
    int rc = gemm_validate(GEMM_B_NK, M, N, K, x, K, w, K, bias, y, ldy, epilogue, dtype);
    if (rc != GEMM_OK) return rc;
    if (M == 0 || N == 0) return GEMM_OK;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
    DeviceGuard g(p->device);
    // implicit GEMM: channel blocks of TC_BK, square filter (the map's
    // bounding box is symmetric), corner offsets in the 8-bit range of a 4-D
    // im2col map, 16-byte aligned activations, more rows than the small-M path
    const bool implicit = K > 0 && C % TC_BK == 0 && R == S && pad <= 127 && (S - 1 - pad) <= 128 &&
                          aligned16(x) && M > 128 && Nb <= INT32_MAX && H <= INT32_MAX && W <= INT32_MAX &&
                          p->forced_kernel != GEMM_KERNEL_SKINNY && g_encode_im2col != nullptr;
    if (implicit) {
        const ConvA cv{x, Nb, H, W, C, R, S, pad};
        return run_impl(p, true, M, N, K, nullptr, 0, w, K, bias, y, ldy, epi, ex, dtype, stream, &cv);
    }
    // otherwise: explicit im2col matrix in the plan workspace, then the GEMM
    if (K == 0) return run_impl(p, true, M, N, K, nullptr, 0, w, K, bias, y, ldy, epi, ex, dtype, stream, nullptr);
    const int64_t ldk = round_up(K, 8);
    rc = ensure_workspace(p, (size_t)(M * ldk * 2));
    if (rc != GEMM_OK) return rc;
    cudaError_t e = launch_im2col(x, Nb, H, W, C, R, S, pad, 1, p->workspace, ldk, 2, stream);
    if (e != cudaSuccess) return record(p, e);
    p->launches += 1;
    return run_impl(p, true, M, N, K, p->workspace, ldk, w, K, bias, y, ldy, epi, ex, dtype, stream, nullptr);
}

int gemm_attention(gemm_plan_t p, int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t D, const void* Q,
                   const void* K, const void* V, void* O, float scale, int causal, int dtype, void* stream_v) {
    if (!p || B < 0 || H < 0 || Sq < 0 || Sk < 0) return GEMM_ERR_INVALID_ARG;
    if (dtype < GEMM_BF16_F32OUT || dtype > GEMM_F16_F16OUT) return GEMM_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return GEMM_ERR_UNSUPPORTED;
    const int64_t BH = B * H;
    if (BH == 0 || Sq == 0) return GEMM_OK;
    if (O == nullptr || Q == nullptr || (Sk > 0 && (K == nullptr || V == nullptr))) return GEMM_ERR_INVALID_ARG;
    if (BH > 65535 || Sq > INT32_MAX - 128 || Sk > INT32_MAX - 128) return GEMM_ERR_UNSUPPORTED;
    if (!aligned16(Q) || !aligned16(O) || (Sk > 0 && (!aligned16(K) || !aligned16(V)))) return GEMM_ERR_ALIGNMENT;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
    DeviceGuard g(p->device);
    const int ob = out_bytes(dtype);
    cudaError_t e;
    if (Sk == 0) {   // every query sees nothing: zeros
        e = cudaMemsetAsync(O, 0, (size_t)(BH * Sq * D * ob), stream);
        if (e != cudaSuccess) return record(p, e);
        p->last_stream = stream; p->have_stream = true;
        return GEMM_OK;
    }
    const CUtensorMapDataType dt = in_map_type(dtype);
    CUtensorMap tmQ, tmK, tmV;
    if (!make_map_3d(&tmQ, dt, Q, (uint64_t)D, (uint64_t)Sq, (uint64_t)BH) ||
        !make_map_3d(&tmK, dt, K, (uint64_t)D, (uint64_t)Sk, (uint64_t)BH) ||
        !make_map_3d(&tmV, dt, V, (uint64_t)D, (uint64_t)Sk, (uint64_t)BH))
        return GEMM_ERR_CUDA;
    AttnParams ap;
    std::memset(&ap, 0, sizeof(ap));
    ap.BH = (int32_t)BH; ap.Sq = (int32_t)Sq; ap.Sk = (int32_t)Sk;
    const float s = scale > 0.0f ? scale : 1.0f / std::sqrt((float)D);
    ap.scale_log2 = s * 1.4426950408889634f;   // log2(e)
    ap.causal = causal ? 1u : 0u;
    ap.idesc_s = make_idesc(dtype, false, 128, 128);       // Q K^T: both operands K-major
    ap.idesc_o = make_idesc(dtype, true, 128, (int)D);     // P V: V is MN-major (D contiguous)
    ap.O = O;
    ap.status = p->status_dev;
    ap.timeout_ns = p->timeout_ns;
    ap.debug = p->debug;
    e = launch_attention(dtype, (int)D, tmQ, tmK, tmV, ap, stream);
    if (e != cudaSuccess) return record(p, e);
    p->launches += 1;
    p->last_stream = stream; p->have_stream = true;
    return GEMM_OK;
}

int gemm_conv2d_maxpool(gemm_plan_t p, int64_t Nb, int64_t H, int64_t W, int64_t C, int64_t Cout, int R, int S,
                        int pad, const void* x, const void* w, void* y, int64_t ldy,
                        const gemm_epilogue_args_t* epi_args, int dtype, void* stream_v) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    if (Nb < 0 || H < 0 || W < 0 || C < 0 || Cout < 0 || R < 1 || S < 1 || pad < 0) return GEMM_ERR_INVALID_ARG;
    const int64_t OH = H + 2 * pad - R + 1, OW = W + 2 * pad - S + 1;
    if (OH < 0 || OW < 0 || (OH & 1) || (OW & 1)) return GEMM_ERR_INVALID_ARG;   // whole 2 x 2 windows
    if (dtype_is_fp8(dtype) || dtype_is_tf32(dtype)) return GEMM_ERR_UNSUPPORTED;
    uint32_t epi = 0;
    EpiArgs ex = plain_epilogue();
    const void* bias = nullptr;
    if (epi_args) {
        if (epi_args->beta != 0.0f) return GEMM_ERR_INVALID_ARG;   // the pooled output is only written
        int rc0 = extended_epilogue(epi_args, dtype, y, ldy, &epi, &ex);
        if (rc0 != GEMM_OK) return rc0;
        bias = epi_args->bias;
    }
    const int64_t PH = OH / 2, PW = OW / 2;
    const int64_t rows = Nb * PH * PW, N = Cout, K = (int64_t)R * S * C;
    int rc = gemm_validate(GEMM_B_NK, rows, N, K, x, K, w, K, bias, y, ldy, (int)(epi & 3u), dtype);
    if (rc != GEMM_OK) return rc;
    if (rows == 0 || N == 0) return GEMM_OK;
    // the fused form needs the implicit-GEMM operand (channel blocks of 64, a
    // square filter, aligned activations) and K > 0
    // and the pooled rows are stored with 16-byte vectors (no pack workspace)
    if (K == 0 || C % TC_BK != 0 || R != S || pad > 127 || (S - 1 - pad) > 128 || !aligned16(x) ||
        !aligned16(y) || (ldy * out_bytes(dtype)) % 16 != 0 || g_encode_im2col == nullptr || Nb > INT32_MAX / 2)
        return GEMM_ERR_UNSUPPORTED;
    DeviceGuard g(p->device);
    // virtual GEMM rows: one 128-row tile per 64 positions of the sequence
    // (image, row pair, column), top pixels then bottom pixels.  (Tiles of 8 or
    // 16 columns x 16 or 8 rows, which hold every window inside one warp, measured
    // 2.7x slower: one small im2col copy per row makes the loads the limit.)
    const int64_t units = (Nb * PH * OW + 63) / 64;
    if (units > INT32_MAX / TC_BM || Nb * PH * OW > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
    ConvA cv{x, Nb, H, W, C, R, S, pad};
    cv.pool = true;
    cv.pool_y = y;
    cv.pool_ldy = ldy;
    return run_impl(p, true, units * TC_BM, N, K, nullptr, 0, w, K, bias, y, ldy, epi, ex, dtype,
                    reinterpret_cast<cudaStream_t>(stream_v), &cv);
}

}  // extern "C"
