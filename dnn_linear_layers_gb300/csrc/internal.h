// Host-side declarations shared by the C-ABI layer and the kernel translation
// units.  Not part of the public interface (that is include/gemm.h).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gb300 {

// Output/input type combinations, same numbering as gemm_dtype_t.  The fp8
// inputs (A and B in one format) take bf16 bias and scale vectors.
enum Dtype : int {
    DT_BF16_F32 = 0, DT_BF16_BF16 = 1, DT_F16_F32 = 2, DT_F16_F16 = 3,
    DT_E4M3_F32 = 4, DT_E4M3_BF16 = 5, DT_E5M2_F32 = 6, DT_E5M2_BF16 = 7, DT_TF32_F32 = 8, DT_TF32_BF16 = 9
};
constexpr bool dtype_is_fp8(int dt) { return dt >= DT_E4M3_F32 && dt <= DT_E5M2_BF16; }
constexpr bool dtype_is_tf32(int dt) { return dt == DT_TF32_F32 || dt == DT_TF32_BF16; }
constexpr int kNumDtypes = 10;

// Epilogue on the fp32 accumulator, in this order: t = alpha * acc (EPI_ALPHA);
// t *= scale[n] (EPI_SCALE); t += bias[n] (EPI_BIAS); t += beta * C_old[m][n]
// (EPI_BETA); t = max(t, 0) (EPI_RELU); then the single cast to the output type.
enum EpiFlags : uint32_t { EPI_BIAS = 1u, EPI_RELU = 2u, EPI_SCALE = 4u, EPI_ALPHA = 8u, EPI_BETA = 16u };

// Operands of the extended epilogue (unused fields are ignored).
struct EpiArgs {
    float alpha;           // EPI_ALPHA
    float beta;            // EPI_BETA
    const void* scale;     // EPI_SCALE: N per-column factors of the input type
    const void* c_old;     // EPI_BETA: previous C (output type), row pitch ldc_old elements
    int64_t ldc_old;
    uint32_t scale_vec16;  // scale is 16-byte aligned
    uint32_t c_old_vec16;  // c_old and ldc_old * element size are 16-byte aligned
};

// Bits written into the device status word by a wait that ran out of time.
enum StatusBits : int {
    ST_TIMEOUT_PRODUCER = 1,
    ST_TIMEOUT_MMA = 2,
    ST_TIMEOUT_EPILOGUE = 4,
    ST_SMEM_LAYOUT = 8,     // shared window too misaligned for the kernel's tiles (it did nothing)
};

// Fault-injection flags (tests only): make one wait run out on purpose.
enum DebugFlags : uint32_t {
    DBG_SKIP_FIRST_ACC_COMMIT = 1u,   // MMA warp never signals the first accumulator (attention: the first PV product)
};

// Tile shape of the tensor-core kernels: each CTA owns 128 rows of C, the
// tile is 256 columns wide, k-blocks are 64 elements (one 128-byte swizzle row).
constexpr int TC_BM = 128;
constexpr int TC_BN = 256;
constexpr int TC_BK = 64;

struct TcParams {
    int32_t M, N, K;
    int32_t num_m_tiles;   // tiles of TC_BM * cta_group rows
    int32_t num_n_tiles;   // tiles of TC_BN columns
    int32_t num_k_blocks;  // ceil(K / TC_BK)
    int32_t group_m;       // rasterisation: m-tiles per group
    int32_t num_full;      // tiles after the split ones run whole; the rest as two N-halves
    uint32_t idesc_half;   // instruction descriptor for a half tile (N = TC_BN / 2)
    uint32_t epi;          // EpiFlags
    uint32_t idesc;        // tcgen05 instruction descriptor
    uint32_t b_mn_major;   // 1: B is K x N (N contiguous); 0: B is N x K
    uint32_t a_mn_major;   // 1: A is K x M (M contiguous); 0: A is M x K
    uint32_t a_chunks;     // 1: MN-major A tile in one copy ([M/64][K][64] map)
    uint32_t b_chunks;     // 1: MN-major B tile in one copy ([N/64][K][64] map)
    const void* bias;      // N elements of the input type, or null
    uint32_t bias_vec16;   // 1: bias is 16-byte aligned (vector loads allowed)
    int* status;           // device status word (StatusBits)
    uint64_t timeout_ns;   // bound on any single wait
    uint32_t debug;        // DebugFlags
    uint32_t l2_policy;    // 0: A evict_last, B evict_normal; 1: A normal, B last; 2: both normal
    uint32_t pdl;          // host only: launch with programmatic stream serialisation
    uint32_t k_snake;      // 1: every other tile of a worker walks k backwards
    uint32_t c_direct;     // 1: C breaks the TMA rule: the epilogue stores it with plain stores
    void* c_ptr;           // c_direct: C (M x N, row pitch ldc elements, any alignment of its type)
    int64_t ldc;
    EpiArgs ex;            // alpha / scale / beta operands of the epilogue
    // Stream-K (sk_tiles > 0): tiles [0, sk_tiles) of the raster are split into
    // equal ranges of k-atoms over workers [0, sk_workers) (worker w takes atoms
    // [w A / W, (w + 1) A / W) of the A = sk_tiles * num_k_blocks atoms, in tile
    // order); each worker runs its pieces of them first, then whole tiles from
    // sk_tiles on.  A split tile's contributors leave fp32 partials in sk_part
    // (sk_tiles x sk_maxc x 8 slots of 32 rows x 256 columns) and count their
    // arrival in sk_cnt (sk_tiles x 8, zero between launches); the last arrival
    // of each 32-row slot adds the partials in contributor order and applies
    // the epilogue.
    int32_t sk_tiles;
    int32_t sk_workers;
    int32_t sk_maxc;
    int* sk_cnt;
    float* sk_part;
    // Implicit-GEMM convolution (conv != 0): A is not a matrix but an NHWC
    // activation tensor read through an im2col tensor map; row m of A is
    // output pixel m = (n * out_h + oh) * out_w + ow and k-block kb is channel
    // block kb % conv_cb of filter tap kb / conv_cb = r * conv_s + s (stride 1).
    uint32_t conv;
    int32_t conv_cb;       // channel blocks of TC_BK per tap (C / 64)
    int32_t conv_s;        // filter width S
    int32_t conv_pad;      // zero padding (rows and columns)
    int32_t conv_out_w;    // output width  (= W for stride 1, pad (S-1)/2)
    int32_t conv_out_hw;   // output pixels per image
    // Fused 2 x 2 max-pool (conv_pool != 0): the output pixels are taken as
    // positions k = (n * pool_ph + ph) * out_w + ow of row pairs (2 ph, 2 ph + 1);
    // CTA tile u holds positions 64 u .. 64 u + 63, rows 0..63 the top pixels
    // (A through the first im2col map, which steps two rows) and rows 64..127
    // the bottom pixels (the second map, one row lower).  Only pooled values are
    // written: position k to row k / 2 of pool_y (pitch pool_ldy).
    uint32_t conv_pool;
    int32_t pool_ph;       // out_h / 2
    int32_t pool_rows;     // pooled output rows: images * out_h / 2 * out_w / 2
    void* pool_y;
    int64_t pool_ldy;
    uint32_t pool_vec16;   // pool_y and pool_ldy * element size are 16-byte aligned
};

// Launch the persistent tcgen05 GEMM.  cta_group is 1 or 2; grid is the
// number of CTAs (a multiple of cta_group).  Returns the launch's cudaError_t.
cudaError_t launch_tc_gemm(int cta_group, int dtype, const CUtensorMap& tmA, const CUtensorMap& tmB,
                           const CUtensorMap& tmC, const TcParams& p, int grid, cudaStream_t stream,
                           const CUtensorMap* tmA2 = nullptr);   // second A map (fused max-pool only)

// Dynamic shared memory the tensor-core kernel needs for a cta_group.
int tc_smem_bytes(int cta_group);

// Configure kernel attributes (dynamic smem) and report the largest number of
// co-resident clusters (cta_group 2: CTA pairs) or CTAs (cta_group 1) on this
// device.
cudaError_t tc_prepare(int cta_group, int dtype, int* max_units);

// Skinny-M (M <= 128) Linear layer: weight-streaming tcgen05 kernel ------
struct SkinnyParams {
    int32_t M, N, K;
    int32_t mpad;          // M rounded up to a multiple of 16 (MMA N), <= 128
    int32_t stages;        // depth of the operand ring (2..8)
    int32_t splits;        // k-slices per feature tile = cluster size (1, 2, 4, 8)
    int32_t num_k_blocks;  // ceil(K / 64)
    int32_t tmem_cols;     // TMEM columns allocated (power of two >= 32, >= mpad)
    uint32_t epi;          // EpiFlags
    uint32_t idesc;        // tcgen05 instruction descriptor (M = 128, N = mpad)
    uint32_t w_mn_major;   // 1: W stored K x N (features contiguous); 0: N x K
    const void* bias;      // N elements of the input type, or null
    void* Y;               // output, M x N, row pitch ldy (elements)
    int64_t ldy;
    int* status;
    uint64_t timeout_ns;
    uint32_t pdl;          // host only: launch with programmatic stream serialisation
    uint32_t w_prefetch;   // 1: W may be read before the previous kernel of the stream ends
    EpiArgs ex;            // alpha / scale / beta operands of the epilogue
};

// at most this many skinny CTAs share an SM (the kernel's launch bounds size
// its registers for it)
constexpr int kSkinnyMaxCtasPerSm = 4;
int skinny_smem_bytes(int mpad, int stages);
cudaError_t skinny_prepare(int dtype);
cudaError_t launch_skinny(int dtype, const CUtensorMap& tmW, const CUtensorMap& tmX, const SkinnyParams& p,
                          int grid, cudaStream_t stream);

// GEMV / very-small-M Linear layer on the CUDA cores (M <= 4, W stored N x K)
struct GemvParams {
    int32_t M, N, K;
    const void* X;         // M x K, row pitch ldx elements (rows 16-byte aligned)
    int64_t ldx;
    const void* W;         // N x K, row pitch ldw elements (rows 16-byte aligned)
    int64_t ldw;
    const void* bias;      // N elements (bf16 for fp8 operands), or null
    void* Y;               // M x N, row pitch ldy elements
    int64_t ldy;
    uint32_t epi;          // EpiFlags
    EpiArgs ex;
    uint32_t pdl;          // host only: launch with programmatic stream serialisation
    uint32_t w_prefetch;   // 1: W may be read before the previous kernel of the stream ends
};
constexpr int kGemvThreads = 256;
constexpr int kGemvMaxM = 4;
// tokens a kernel instantiation holds for M tokens (1, 2 or 4; 0 if M > 4)
int gemv_tokens_held(int M);
cudaError_t gemv_prepare(int M, int dtype, int* blocks_per_sm);
cudaError_t launch_gemv(int dtype, const GemvParams& p, int grid, cudaStream_t stream);
// Warp-MMA small-M kernel (16-bit or fp8 operands, 2 <= M <= 16, W stored N x K):
// groups of 8 tokens held (1 or 2; 0 if M > 16); ks = warps of a CTA
// splitting K (1, 2, 4 or 8).
constexpr int kWarpMmaMaxM = 16;
int gemv_mma_groups(int M);
cudaError_t gemv_mma_prepare(int nh, int ks, int dtype, int* blocks_per_sm);
cudaError_t launch_gemv_mma(int dtype, int ks, const GemvParams& p, int grid, cudaStream_t stream);

// Fused attention forward -------------------------------------------------
// O = softmax(scale * Q K^T (masked)) V per (batch, head); Q, K, V, O are
// [B*H][S][D] row-major (D = 64 or 128); one CTA per 128 queries of one head.
struct AttnParams {
    int32_t BH;            // batch * heads
    int32_t Sq, Sk;        // query / key sequence lengths
    float scale_log2;      // softmax scale * log2(e): scores are taken in base 2
    uint32_t causal;       // key j visible to query i iff j <= i + (Sk - Sq)
    uint32_t idesc_s;      // tcgen05 descriptor of S = Q K^T (M 128, N 128, both K-major)
    uint32_t idesc_o;      // tcgen05 descriptor of O += P V (M 128, N = D, V MN-major)
    void* O;
    int* status;
    uint64_t timeout_ns;
    uint32_t debug;        // DebugFlags (tests only)
};
cudaError_t attention_prepare(int dtype);
cudaError_t launch_attention(int dtype, int D, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                             const CUtensorMap& tmV, const AttnParams& p, cudaStream_t stream);

// Auxiliary kernels ------------------------------------------------------
// C[i][j] = epilogue(0) for K == 0 (bias and/or ReLU of an empty sum).
cudaError_t launch_fill_epilogue(int dtype, int64_t M, int64_t N, const void* bias, uint32_t epi,
                                 const EpiArgs& ex, void* C, int64_t ldc, cudaStream_t stream);

// Copy a rows x cols matrix of elem_bytes-sized elements between strides.
// When the destination is 16-byte aligned with ld_dst >= cols rounded up to
// 16 bytes, the columns up to that boundary are zero-filled as well.
cudaError_t launch_copy2d(const void* src, int64_t ld_src, void* dst, int64_t ld_dst,
                          int64_t rows, int64_t cols, int elem_bytes, cudaStream_t stream);

// Rasterisation group (tile-rows walked together) for a grid of tile columns
// run by `workers` co-resident CTAs or CTA pairs: when one wave of tiles spans
// three or more whole tile-rows, row-major order (1) measured best (4096^3 3.3%,
// 6144^3 4.4%, 8192 x 4096 x 4096 5% faster than groups of 8); when it spans
// fewer, groups of 16 tile-rows keep the panels of a wave in L2 (against 1:
// 8192^3 8%, 8192 x 4096 x 12288 10%; against 8: 1-3%, e.g. 8192 x 4096 x
// 14336 2.8%, e4m3 8192^3 2.2%; 24 and 32 were slower again).
inline int auto_group_m(int64_t num_n_tiles, int64_t workers) {
    return num_n_tiles * 3 <= workers ? 1 : 16;
}

// Packing job: rows x row_bytes bytes from src (row pitch ld_src_bytes, any
// alignment) into dst (16-byte aligned, pitch ld_dst_bytes a multiple of 16
// and at least row_bytes rounded up to 16), zero-filling each row up to its
// 16-byte boundary; chunks = 16-byte pieces per row.  A job with rows = 0 is
// empty.
struct PackJob {
    const uint8_t* src;
    int64_t ld_src_bytes;
    uint8_t* dst;
    int64_t ld_dst_bytes;
    int64_t rows;
    int64_t row_bytes;
    int64_t chunks;
};
PackJob pack_job(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows, int64_t cols,
                 int elem_bytes);
// Run up to two packing jobs in one launch.
cudaError_t launch_pack2(const PackJob& j0, const PackJob& j1, cudaStream_t stream);

// Transposition job of 32-bit elements: dst[c * ld_dst + r] = src[r * ld_src +
// c] for r < rows, c < cols (pitches in elements; dst columns past rows are not
// written).  src on a 4-byte boundary, dst on a 16-byte one with ld_dst a
// multiple of 4.  A job with rows or cols = 0 is empty; j1 may be empty.
struct TransJob {
    const uint32_t* src;
    int64_t ld_src;
    uint32_t* dst;
    int64_t ld_dst;
    int64_t rows;
    int64_t cols;
};
cudaError_t launch_transpose2(const TransJob& j0, const TransJob& j1, cudaStream_t stream);

// im2col of an NHWC tensor for an R x S convolution (zero padding `pad`,
// stride `stride`): out[(n*OH + oh)*OW + ow][(r*S + s)*C + c], row pitch ld_out.
cudaError_t launch_im2col(const void* x, int64_t Nb, int64_t H, int64_t W, int64_t C, int R, int S, int pad,
                          int stride, void* out, int64_t ld_out, int elem_bytes, cudaStream_t stream);

}  // namespace gb300
