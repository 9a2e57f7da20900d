// gemm_run_noalloc: the GEMM entry point for callers that cannot allocate
// device memory.
//
// Who needs it: processes whose device memory is fully reserved up front by a
// pool or framework allocator (a serving process that pre-allocates HBM and
// forbids allocation afterwards), and latency-sensitive callers for whom
// cudaMalloc / cudaFree are off limits because they may synchronise the whole
// device and stall other streams.  gemm_run, by contrast, needs a plan (whose
// creation allocates a status word) and may grow the plan's workspace with
// cudaMalloc when an operand must be packed.
//
// How: the scratch this path needs -- a device status word and the packed,
// 16-byte-aligned copies of operands whose base address or row pitch breaks
// the TMA rule -- lives in one file-scope __device__ array of fixed size that
// every GPU loading the library keeps until the process exits.  Host code
// cannot use the array's name as a device address, so the first call on each
// device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it.  Nothing here calls cudaMalloc, cudaFree or any
// allocating library routine.
//
// All calls on a device share the array and it keeps the last call's
// contents; the status word is cleared at the start of every call.  Calls
// whose work overlaps on the GPU (different streams, or another thread) race
// on the array: callers must order them.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/gemm.h"
#include "internal.h"

namespace {

constexpr size_t kStatusBytes = 256;   // status word, padded to keep the packed area aligned
static_assert(GEMM_NOALLOC_SCRATCH_BYTES > kStatusBytes, "scratch size");

static __device__ __align__(256) unsigned char g_noalloc_scratch[GEMM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool ready = false;
    unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch on this device
    int max_pairs[4] = {};     // co-resident CTA pairs, per 16-bit operand type
    int max_singles[4] = {};   // co-resident single CTAs, per 16-bit operand type
};

DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode_na = nullptr;

// One-time set-up for the current device: scratch address, kernel attributes,
// co-residency limits and the tensor-map encoder.  Returns a GEMM_* code.
int setup_device(int dev, DeviceSetup** out) {
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceSetup& s = g_setup[dev];
    if (!s.ready) {
        void* addr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
        if (e != cudaSuccess || addr == nullptr) { cudaGetLastError(); return GEMM_ERR_CUDA; }
        int n2[4] = {}, n1[4] = {};
        for (int dt = 0; dt < 4; ++dt) {
            e = gb300::tc_prepare(2, dt, &n2[dt]);
            if (e == cudaSuccess) e = gb300::tc_prepare(1, dt, &n1[dt]);
            if (e != cudaSuccess) { cudaGetLastError(); return GEMM_ERR_CUDA; }
            if (n2[dt] < 1 || n1[dt] < 1) return GEMM_ERR_UNSUPPORTED;
        }
        if (!g_encode_na) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
                return GEMM_ERR_CUDA;
            g_encode_na = reinterpret_cast<EncodeTiledFn>(fn);
        }
        s.scratch = static_cast<unsigned char*>(addr);
        for (int dt = 0; dt < 4; ++dt) {
            s.max_pairs[dt] = n2[dt];
            s.max_singles[dt] = n1[dt];
        }
        s.ready = true;
    }
    *out = &s;
    return GEMM_OK;
}

bool map2d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
           uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer) {
    cuuint64_t gdim[2] = {inner, outer};
    cuuint64_t gstride[1] = {pitch_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return g_encode_na(m, dt, 2, const_cast<void*>(ptr), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int64_t rup(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

}  // namespace

extern "C" int gemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                                int64_t ldb, const void* bias, void* C, int64_t ldc, int epilogue, int dtype,
                                unsigned flags, int* dev_status, void* stream_v) {
    // only the B-layout flag applies here: no plan to hold constant weights
    // or a transposed A
    if (flags & ~GEMM_B_NK) return GEMM_ERR_INVALID_ARG;
    int rc = gemm_validate(flags, M, N, K, A, lda, B, ldb, bias, C, ldc, epilogue, dtype);
    if (rc == GEMM_OK && (gb300::dtype_is_fp8(dtype) || gb300::dtype_is_tf32(dtype)))
        rc = GEMM_ERR_UNSUPPORTED;   // 16-bit inputs only
    if (rc != GEMM_OK) return rc;
    if (M == 0 || N == 0) return GEMM_OK;
    const bool b_nk = (flags & GEMM_B_NK) != 0;
    const int ob = (dtype == GEMM_BF16_F32OUT || dtype == GEMM_F16_F32OUT) ? 4 : 2;

    // Scratch needed for packed operands, checked before anything is launched.
    const int64_t b_rows = b_nk ? N : K, b_cols = b_nk ? K : N;
    const bool a_ok = K == 0 || (al16(A) && (lda * 2) % 16 == 0);
    const bool b_ok = K == 0 || (al16(B) && (ldb * 2) % 16 == 0);
    // C that breaks the TMA rule (base, pitch, or a right edge inside a
    // 16-byte granule, where a TMA store would write past column N) is stored
    // by the epilogue itself
    const bool c_direct = !(al16(C) && (ldc * ob) % 16 == 0 && (N * ob) % 16 == 0);
    const int64_t lda_p = rup(K, 8), ldb_p = rup(b_cols, 8);
    const int64_t a_bytes = a_ok ? 0 : rup(M * lda_p * 2, 256);
    const int64_t b_bytes = b_ok ? 0 : rup(b_rows * ldb_p * 2, 256);
    if (a_bytes + b_bytes > (int64_t)(GEMM_NOALLOC_SCRATCH_BYTES - kStatusBytes))
        return GEMM_ERR_UNSUPPORTED;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { cudaGetLastError(); return GEMM_ERR_CUDA; }
    DeviceSetup* s = nullptr;
    rc = setup_device(dev, &s);
    if (rc != GEMM_OK) return rc;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
    const uint32_t epi = (uint32_t)epilogue;

    if (K == 0) {
        gb300::EpiArgs ex;
        std::memset(&ex, 0, sizeof(ex));
        e = gb300::launch_fill_epilogue(dtype, M, N, bias, epi, ex, C, ldc, stream);
        return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    }

    int* status = dev_status;
    if (status == nullptr) {
        status = reinterpret_cast<int*>(s->scratch);
        e = cudaMemsetAsync(status, 0, sizeof(int), stream);
        if (e != cudaSuccess) return GEMM_ERR_CUDA;
    }
    unsigned char* ws = s->scratch + kStatusBytes;
    const void* A_use = A; int64_t lda_use = lda;
    const void* B_use = B; int64_t ldb_use = ldb;
    gb300::PackJob ja = {}, jb = {};
    if (!a_ok) {
        ja = gb300::pack_job(A, lda, ws, lda_p, M, K, 2);
        A_use = ws; lda_use = lda_p;
    }
    if (!b_ok) {
        jb = gb300::pack_job(B, ldb, ws + a_bytes, ldb_p, b_rows, b_cols, 2);
        B_use = ws + a_bytes; ldb_use = ldb_p;
    }
    if (!a_ok || !b_ok) {
        e = gb300::launch_pack2(ja, jb, stream);
        if (e != cudaSuccess) return GEMM_ERR_CUDA;
    }

    const int cg = (M <= 128) ? 1 : 2;
    const bool bf16_in = (dtype == GEMM_BF16_F32OUT || dtype == GEMM_BF16_BF16OUT);
    const CUtensorMapDataType in_dt = bf16_in ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUtensorMapDataType out_dt = (ob == 4) ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : in_dt;
    CUtensorMap tmA, tmB, tmC;
    if (!map2d(&tmA, in_dt, A_use, (uint64_t)K, (uint64_t)M, (uint64_t)lda_use * 2, gb300::TC_BK, gb300::TC_BM))
        return GEMM_ERR_CUDA;
    const bool okb = b_nk ? map2d(&tmB, in_dt, B_use, (uint64_t)K, (uint64_t)N, (uint64_t)ldb_use * 2, gb300::TC_BK,
                                  gb300::TC_BN / cg)
                          : map2d(&tmB, in_dt, B_use, (uint64_t)N, (uint64_t)K, (uint64_t)ldb_use * 2, 64, gb300::TC_BK);
    if (!okb) return GEMM_ERR_CUDA;
    if (c_direct) std::memset(&tmC, 0, sizeof(tmC));   // not used: the epilogue stores C itself
    else if (!map2d(&tmC, out_dt, C, (uint64_t)N, (uint64_t)M, (uint64_t)ldc * ob, 128 / ob, 32))
        return GEMM_ERR_CUDA;

    gb300::TcParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.M = (int32_t)M; prm.N = (int32_t)N; prm.K = (int32_t)K;
    prm.num_m_tiles = (int32_t)((M + gb300::TC_BM * cg - 1) / (gb300::TC_BM * cg));
    prm.num_n_tiles = (int32_t)((N + gb300::TC_BN - 1) / gb300::TC_BN);
    prm.num_k_blocks = (int32_t)((K + gb300::TC_BK - 1) / gb300::TC_BK);
    prm.epi = epi;
    const uint32_t ab = bf16_in ? 1u : 0u;
    prm.idesc = (1u << 4) | (ab << 7) | (ab << 10) | ((b_nk ? 0u : 1u) << 16) |
                ((uint32_t)(gb300::TC_BN >> 3) << 17) | ((uint32_t)((gb300::TC_BM * cg) >> 4) << 24);
    prm.b_mn_major = b_nk ? 0u : 1u;
    prm.bias = bias;
    prm.bias_vec16 = (bias != nullptr && al16(bias)) ? 1u : 0u;
    prm.status = status;
    prm.timeout_ns = 1000000000ull;
    prm.debug = 0;
    prm.l2_policy = 0;
    prm.num_full = prm.num_m_tiles * prm.num_n_tiles;   // whole tiles only
    if (c_direct) {
        prm.c_direct = 1u;
        prm.c_ptr = C;
        prm.ldc = ldc;
    }
    const int64_t tiles = (int64_t)prm.num_m_tiles * prm.num_n_tiles;
    if (tiles > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
    const int64_t cap = (cg == 2) ? s->max_pairs[dtype] : s->max_singles[dtype];
    const int64_t units = tiles < cap ? tiles : cap;
    prm.group_m = gb300::auto_group_m(prm.num_n_tiles, cap);
    e = gb300::launch_tc_gemm(cg, dtype, tmA, tmB, tmC, prm, (int)(units * cg), stream);
    if (e != cudaSuccess) return GEMM_ERR_CUDA;
    return GEMM_OK;
}
