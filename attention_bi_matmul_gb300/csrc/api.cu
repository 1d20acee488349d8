// api.cu -- the C ABI of include/bi.h: argument validation, configuration
// choice, tensor-map encoding and launches on the caller's stream.
//
// Routing rule (the batch-invariance contract): the kernel and its tile
// configuration are functions of (dtype, N, K, weight layout) for GEMMs and of
// (dtype, head_dim, group size, mask) for attention.  M, the batch, the query
// length, the context length, pointer values and the environment never select
// a different route; an argument the built kernels cannot take is an error,
// never a fallback.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace bi {

// The device error word: written by kernels (atomicOr), read and cleared by
// bi_last_device_error.  Static storage, one copy per device context.
__device__ uint32_t g_error_word;

namespace {

std::atomic<int64_t> g_launches{0};

// Per-device state, filled once under g_init_mutex and published by the release store
// of g_ready[dev]; entry points called from several host threads read it after the
// acquire load in check_device.
constexpr int MAX_DEV = 64;
std::mutex g_init_mutex;
std::atomic<uint32_t *> g_err_ptr[MAX_DEV] = {};
std::atomic<int> g_sm_count[MAX_DEV] = {};
std::atomic<int> g_arch_ok[MAX_DEV] = {};  // 0 unknown, 1 sm_103, -1 other
std::atomic<int> g_ready[MAX_DEV] = {};    // per-device initialisation done

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return (dev >= 0 && dev < MAX_DEV) ? dev : -1;
}

std::atomic<PFN_cuTensorMapEncodeTiled_v12000> g_encode{nullptr};

// The driver's tensor-map encoder (the same function for every device).  Two threads
// may both look it up; they store the same pointer.
PFN_cuTensorMapEncodeTiled_v12000 load_encode() {
    PFN_cuTensorMapEncodeTiled_v12000 f = g_encode.load(std::memory_order_acquire);
    if (f) return f;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return nullptr;
    f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    g_encode.store(f, std::memory_order_release);
    return f;
}

bi_status device_init(int dev);

// The code in this library is built for sm_103a only.  The first call on a
// device also initialises everything later calls need on it (see device_init),
// so that no later call makes a non-stream CUDA call.  Concurrent first calls
// from several host threads are serialised; later calls take no lock.
bi_status check_device() {
    const int dev = current_device();
    if (dev < 0) return BI_ERR_CUDA;
    if (g_ready[dev].load(std::memory_order_acquire)) return BI_OK;
    std::lock_guard<std::mutex> lock(g_init_mutex);
    if (g_ready[dev].load(std::memory_order_relaxed)) return BI_OK;
    if (g_arch_ok[dev].load(std::memory_order_relaxed) == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return BI_ERR_CUDA;
        g_arch_ok[dev].store((major == 10 && minor == 3) ? 1 : -1, std::memory_order_relaxed);
    }
    if (g_arch_ok[dev].load(std::memory_order_relaxed) != 1) return BI_ERR_UNSUPPORTED;
    bi_status st = device_init(dev);
    if (st != BI_OK) return st;
    g_ready[dev].store(1, std::memory_order_release);
    return BI_OK;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool valid_dtype(bi_dtype dt) { return dt == BI_F32 || dt == BI_F16 || dt == BI_BF16; }
// Element alignment of a pointer that kernels read or write one element at a time
// (2 bytes for the 16-bit dtypes, 4 for fp32); null passes.
inline bool elem_aligned(const void *p, bi_dtype dt) {
    return (reinterpret_cast<uintptr_t>(p) & (dt == BI_F32 ? 3u : 1u)) == 0;
}

// Common validation of the GEMM family.  Returns BI_OK to proceed.
bi_status check_gemm(const void *a, int64_t lda, const void *b, int64_t ldb, void *y, int64_t ldy,
                     int64_t M, int64_t N, int64_t K, bi_dtype dt, bool b_nk) {
    if (!valid_dtype(dt)) return BI_ERR_UNSUPPORTED;
    if (M < 0 || N <= 0 || K <= 0) return BI_ERR_INVALID_ARG;
    if (!a || !b || !y) return BI_ERR_INVALID_ARG;
    if (lda < K || ldy < N || (b_nk ? ldb < K : ldb < N)) return BI_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) || N > (int64_t(1) << 31) || K > (int64_t(1) << 31))
        return BI_ERR_UNSUPPORTED;
    if (dt != BI_F32) {
        if (!aligned16(a) || !aligned16(b) || !aligned16(y)) return BI_ERR_ALIGNMENT;
        if (lda % 8 || ldb % 8 || ldy % 8) return BI_ERR_ALIGNMENT;
    } else {
        if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
             reinterpret_cast<uintptr_t>(y)) & 3u)
            return BI_ERR_ALIGNMENT;
    }
    return BI_OK;
}

bi_status run_gemm(const void *a, int64_t lda, const void *b, int64_t ldb, bool b_nk,
                   GemmArgs &args, bi_dtype dt, cudaStream_t s);

}  // namespace

uint32_t *device_error_word();
int device_sm_count();

namespace {

// Everything a call may need on this device, done once: the shared-memory
// attribute of every kernel, the device error word's address, the SM count and
// the tensor-map encoder.
bi_status device_init(int dev) {
    (void)dev;
    bi_status st;
    if ((st = init_gemm_tc_bf16()) != BI_OK) return st;
    if ((st = init_gemm_tc_f16()) != BI_OK) return st;
    if ((st = init_sdpa()) != BI_OK) return st;
    if ((st = init_qgemm()) != BI_OK) return st;
    if (!device_error_word()) return BI_ERR_CUDA;
    device_sm_count();
    if (!load_encode()) return BI_ERR_CUDA;
    return BI_OK;
}

}  // namespace

// ------------------------------------------------------------------ helpers

bi_status cuda_status(cudaError_t e) { return e == cudaSuccess ? BI_OK : BI_ERR_CUDA; }

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

uint32_t *device_error_word() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    uint32_t *w = g_err_ptr[dev].load(std::memory_order_acquire);
    if (!w) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
        w = static_cast<uint32_t *>(p);
        g_err_ptr[dev].store(w, std::memory_order_release);
    }
    return w;
}

int device_sm_count() {
    const int dev = current_device();
    if (dev < 0) return 1;
    int n = g_sm_count[dev].load(std::memory_order_acquire);
    if (!n) {
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        n = n > 0 ? n : 1;
        g_sm_count[dev].store(n, std::memory_order_release);
    }
    return n;
}

bi_status encode_tmap(CUtensorMap *map, bi_dtype dt, int rank, void *base, const uint64_t *dims,
                      const uint64_t *strides_bytes, const uint32_t *box, bool swizzle128) {
    const PFN_cuTensorMapEncodeTiled_v12000 encode = load_encode();
    if (!encode) return BI_ERR_CUDA;
    const CUtensorMapDataType t = dt == BI_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                  : dt == BI_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    cuuint64_t gdim[5], gstr[4];
    cuuint32_t bdim[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estr[i] = 1;
    }
    for (int i = 0; i + 1 < rank; ++i) gstr[i] = strides_bytes[i];
    const CUresult r = encode(map, t, static_cast<cuuint32_t>(rank), base, gdim, gstr, bdim, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BI_OK : BI_ERR_INVALID_ARG;
}

// Packed 32-bit words (quantized weights); with swizzle128 the box's 128-byte
// rows are stored with the 128-byte swizzle (16-byte chunk c of row r at c ^ (r % 8)).
bi_status encode_tmap_u32(CUtensorMap *map, int rank, void *base, const uint64_t *dims,
                          const uint64_t *strides_bytes, const uint32_t *box, bool swizzle128) {
    const PFN_cuTensorMapEncodeTiled_v12000 encode = load_encode();
    if (!encode) return BI_ERR_CUDA;
    cuuint64_t gdim[5], gstr[4];
    cuuint32_t bdim[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estr[i] = 1;
    }
    for (int i = 0; i + 1 < rank; ++i) gstr[i] = strides_bytes[i];
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, static_cast<cuuint32_t>(rank),
                                base, gdim, gstr, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BI_OK : BI_ERR_INVALID_ARG;
}

// Tile form of the tensor-core GEMM for (N, K, dtype, layout).  M is not an
// input, and neither is anything else about the call.  Measured on GB300
// (bf16, weights streamed from HBM):
//   * K = 4096: a 128 x 128 tile on one CTA is within a few percent of the best
//     width for every M from 1 to 512 (it keeps N/128 blocks streaming weights
//     for decode-shaped calls).  The 256 x 256 pair tile is slower there: each
//     SM then runs the K loop of a 128 x 256 output, 25 us instead of 20.5 us
//     at N = 11008, M = 1, and 614 us instead of 589 us over the M = 1..512 sweep.
//     Wider tiles on one CTA trade the same way: 192 columns take N = 11008,
//     M = 256 from 37 to 28 us but M = 1 from 20.6 to 23.6 us, and the eleven
//     batch sizes at N = 11008 and 14336 sum to 602 us (256 columns: 690 us)
//     against 585 us for 128.
//     256 x 128 pair tiles (half the weight rows per SM) need twice the CTAs,
//     so decode-shaped calls run two waves: 42 us instead of 21 at N = 11008,
//     and the sweep over N = 4096, 11008 and 14336 takes 1231 us against 791.
//   * K = 8192: 256 columns win both for decode-shaped calls and at M = 8192,
//     and on a CTA pair (256 x 256, a third fewer bytes into each SM) the 8192^3
//     product runs at 1.81 PFLOP/s, against 1.67 for 128 x 256 on one CTA and
//     1.1 for 128 x 128.
// Hence: 256 x 256 pair tiles from K = 8192 up, 128 x 128 below, for both
// weight layouts.
TcConfig tc_config(int64_t N, int64_t K, bi_dtype dt, bool b_mn_major) {
    (void)N;
    (void)dt;
    (void)b_mn_major;
    TcConfig c;
    c.block_n = K >= 8192 ? 256 : 128;
    c.stages = c.block_n == 256 ? 4 : 3;    // ring depth (stages of 1 or 2 K panels)
    c.pair = c.block_n == 256;
    return c;
}

bi_status launch_gemm_tc_bf16(const void *a, int64_t lda, const void *b, int64_t ldb, bool b_nk,
                              const GemmArgs &args, const TcConfig &cfg, cudaStream_t s);
bi_status launch_gemm_tc_f16(const void *a, int64_t lda, const void *b, int64_t ldb, bool b_nk,
                             const GemmArgs &args, const TcConfig &cfg, cudaStream_t s);

bi_status launch_gemm_tc(const void *a, int64_t lda, const void *b, int64_t ldb, bool b_nk,
                         const GemmArgs &args, bi_dtype dt, const TcConfig &cfg, cudaStream_t s) {
    if (dt == BI_BF16) return launch_gemm_tc_bf16(a, lda, b, ldb, b_nk, args, cfg, s);
    if (dt == BI_F16) return launch_gemm_tc_f16(a, lda, b, ldb, b_nk, args, cfg, s);
    return BI_ERR_UNSUPPORTED;
}

namespace {

bi_status run_gemm(const void *a, int64_t lda, const void *b, int64_t ldb, bool b_nk,
                   GemmArgs &args, bi_dtype dt, cudaStream_t s) {
    if (args.M == 0) return BI_OK;
    bi_status st = check_device();
    if (st != BI_OK) return st;
    args.err = device_error_word();
    if (!args.err) return BI_ERR_CUDA;
    if (dt == BI_F32)
        return launch_gemm_f32(static_cast<const float *>(a), lda, static_cast<const float *>(b),
                               ldb, b_nk, args, s);
    const TcConfig cfg = tc_config(args.N, args.K, dt, !b_nk);
    // Rows of the A tile each copy moves.  The kernel, its tile and every stored
    // row's arithmetic are the same for every M; this only spares the copy engine
    // rows that do not exist (small batches ran 1.7x slower with a 128-row box
    // holding fewer than 16 real rows).
    args.a_rows = static_cast<int>(args.M >= 128 ? 128 : ((args.M + 15) / 16) * 16);
    return launch_gemm_tc(a, lda, b, ldb, b_nk, args, dt, cfg, s);
}

}  // namespace

}  // namespace bi

using namespace bi;

extern "C" {

bi_status bi_linear(const void *x, int64_t ldx, const void *w, int64_t ldw, const void *bias,
                    void *y, int64_t ldy, int64_t M, int64_t N, int64_t K, bi_dtype dtype,
                    bi_stream_t stream) {
    bi_status st = check_gemm(x, ldx, w, ldw, y, ldy, M, N, K, dtype, true);
    if (st != BI_OK) return st;
    if (!elem_aligned(bias, dtype)) return BI_ERR_ALIGNMENT;   // read one element at a time
    GemmArgs args{};
    args.M = M; args.N = N; args.K = K; args.y = y; args.ldy = ldy; args.batch = 1;
    args.bias = bias;
    args.epi = bias ? EPI_BIAS : EPI_NONE;
    return run_gemm(x, ldx, w, ldw, true, args, dtype, reinterpret_cast<cudaStream_t>(stream));
}

bi_status bi_matmul(const void *a, int64_t lda, const void *b, int64_t ldb, void *y, int64_t ldy,
                    int64_t M, int64_t N, int64_t K, bi_dtype dtype, bi_stream_t stream) {
    bi_status st = check_gemm(a, lda, b, ldb, y, ldy, M, N, K, dtype, false);
    if (st != BI_OK) return st;
    GemmArgs args{};
    args.M = M; args.N = N; args.K = K; args.y = y; args.ldy = ldy; args.batch = 1;
    args.epi = EPI_NONE;
    return run_gemm(a, lda, b, ldb, false, args, dtype, reinterpret_cast<cudaStream_t>(stream));
}

bi_status bi_matmul_batched(const void *a, int64_t lda, int64_t sa, const void *b, int64_t ldb,
                            int64_t sb, int b_layout, void *y, int64_t ldy, int64_t sy,
                            int64_t batch, int64_t M, int64_t N, int64_t K, bi_dtype dtype,
                            bi_stream_t stream) {
    if (b_layout != 0 && b_layout != 1) return BI_ERR_INVALID_ARG;
    const bool b_nk = b_layout == 0;
    bi_status st = check_gemm(a, lda, b, ldb, y, ldy, M, N, K, dtype, b_nk);
    if (st != BI_OK) return st;
    if (batch < 0 || sa < 0 || sb < 0 || sy < 0) return BI_ERR_INVALID_ARG;
    if (batch == 0 || M == 0) return BI_OK;
    // Entries of y must not overlap (each is written by its own tiles).
    if (batch > 1 && sy < (M - 1) * ldy + N) return BI_ERR_INVALID_ARG;
    if (batch > 65535) return BI_ERR_UNSUPPORTED;
    if (dtype != BI_F32 && (sa % 8 || sb % 8 || sy % 8)) return BI_ERR_ALIGNMENT;
    GemmArgs args{};
    args.M = M; args.N = N; args.K = K; args.y = y; args.ldy = ldy;
    args.batch = batch; args.sa = sa; args.sb = sb; args.sy = sy;
    args.epi = EPI_NONE;
    return run_gemm(a, lda, b, ldb, b_nk, args, dtype, reinterpret_cast<cudaStream_t>(stream));
}

bi_status bi_qlinear(const void *x, int64_t ldx, const uint32_t *wq, int64_t ldq,
                     const void *scales, const void *biases, int64_t ldsb, const void *bias,
                     void *y, int64_t ldy, int64_t M, int64_t N, int64_t K, int bits,
                     int group_size, bi_dtype dtype, bi_stream_t stream) {
    if (dtype != BI_BF16 && dtype != BI_F16) return BI_ERR_UNSUPPORTED;
    if (bits != 2 && bits != 4 && bits != 8) return BI_ERR_UNSUPPORTED;
    if (group_size != 32 && group_size != 64 && group_size != 128) return BI_ERR_UNSUPPORTED;
    if (!x || !wq || !scales || !biases || !y) return BI_ERR_INVALID_ARG;
    if (M < 0 || N <= 0 || K <= 0) return BI_ERR_INVALID_ARG;
    if (K % group_size) return BI_ERR_INVALID_ARG;
    if (K % 64) return BI_ERR_UNSUPPORTED;                  // whole 64-wide panels
    if (ldx < K || ldy < N || ldq < K / 32 * bits || ldsb < K / group_size)
        return BI_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) || N > (int64_t(1) << 31) || K > (int64_t(1) << 31))
        return BI_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(wq) || ldx % 8 || ldq % 4) return BI_ERR_ALIGNMENT;
    if (!aligned16(scales) || !aligned16(biases) || ldsb % 8) return BI_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(bias) | reinterpret_cast<uintptr_t>(y)) & 1u)
        return BI_ERR_ALIGNMENT;
    if (M == 0) return BI_OK;
    bi_status st = check_device();
    if (st != BI_OK) return st;
    QGemmArgs a{};
    a.M = M; a.N = N; a.K = K;
    a.scales = scales; a.biases = biases; a.ldsb = ldsb; a.group_size = group_size;
    a.bias = bias; a.y = y; a.ldy = ldy;
    a.err = device_error_word();
    if (!a.err) return BI_ERR_CUDA;
    // Token rows each x copy moves; the MMA always spans 64 token columns.
    a.x_rows = static_cast<int>(M >= 64 ? 64 : ((M + 15) / 16) * 16);
    return launch_qgemm(x, ldx, wq, ldq, bits, a, dtype, reinterpret_cast<cudaStream_t>(stream));
}

bi_status bi_addmm(const void *c, int64_t ldc, const void *a, int64_t lda, const void *b,
                   int64_t ldb, void *y, int64_t ldy, int64_t M, int64_t N, int64_t K, float alpha,
                   float beta, bi_dtype dtype, bi_stream_t stream) {
    bi_status st = check_gemm(a, lda, b, ldb, y, ldy, M, N, K, dtype, false);
    if (st != BI_OK) return st;
    if (!c || ldc < 0 || (ldc > 0 && ldc < N)) return BI_ERR_INVALID_ARG;
    if (!std::isfinite(alpha) || !std::isfinite(beta)) return BI_ERR_INVALID_ARG;
    if (!elem_aligned(c, dtype)) return BI_ERR_ALIGNMENT;      // read one element at a time
    GemmArgs args{};
    args.M = M; args.N = N; args.K = K; args.y = y; args.ldy = ldy; args.batch = 1;
    args.c = c; args.ldc = ldc; args.alpha = alpha; args.beta = beta;
    args.epi = EPI_ADDMM;
    return run_gemm(a, lda, b, ldb, false, args, dtype, reinterpret_cast<cudaStream_t>(stream));
}

bi_status bi_gemm_config(int64_t N, int64_t K, bi_dtype dtype, int b_layout, int *block_n,
                         int *stages) {
    if (N <= 0 || K <= 0 || (b_layout != 0 && b_layout != 1)) return BI_ERR_INVALID_ARG;
    if (dtype != BI_F16 && dtype != BI_BF16) {
        if (dtype != BI_F32) return BI_ERR_UNSUPPORTED;
        if (block_n) *block_n = 64;   // SIMT path: fixed 64 x 64 block tiles
        if (stages) *stages = 1;
        return BI_OK;
    }
    const TcConfig c = tc_config(N, K, dtype, b_layout == 1);
    if (block_n) *block_n = c.block_n;
    if (stages) *stages = c.stages;
    return BI_OK;
}

bi_status bi_sdpa_ex(const void *q, const int64_t qs[4], const void *k, const int64_t ks[4],
                     const void *v, const int64_t vs[4], void *o, const int64_t os[4], int64_t B,
                     int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D, float scale,
                     bi_mask mask, int64_t q_offset, const float *sinks, const uint8_t *mask_array,
                     const int64_t ms[4], bi_dtype dtype, bi_stream_t stream) {
    if (dtype != BI_BF16 && dtype != BI_F16) return BI_ERR_UNSUPPORTED;
    if (!q || !k || !v || !o || !qs || !ks || !vs || !os) return BI_ERR_INVALID_ARG;
    if (B < 0 || H <= 0 || Hkv <= 0 || Lq < 0 || Lkv < 0 || D <= 0) return BI_ERR_INVALID_ARG;
    if (H % Hkv) return BI_ERR_INVALID_ARG;
    if (mask != BI_MASK_CAUSAL && mask != BI_MASK_NONE && mask != BI_MASK_ARRAY)
        return BI_ERR_UNSUPPORTED;
    if (mask == BI_MASK_ARRAY) {
        if (!mask_array || !ms || ms[3] != 1) return BI_ERR_INVALID_ARG;
        for (int i = 0; i < 3; ++i)
            if (ms[i] < 0) return BI_ERR_INVALID_ARG;
    } else if (mask_array) {
        return BI_ERR_INVALID_ARG;
    }
    // Causal: query i at position q_offset + i must see key 0 and no key past the
    // cache (q_offset + Lq <= Lkv).  The other forms only use the positions to
    // align the query tiles; their default is max(Lkv - Lq, 0).
    if (q_offset < 0)
        q_offset = mask == BI_MASK_CAUSAL ? Lkv - Lq : (Lkv > Lq ? Lkv - Lq : 0);
    if (q_offset < 0 || (mask == BI_MASK_CAUSAL && q_offset + Lq > Lkv)) return BI_ERR_INVALID_ARG;
    if (Lq == 0 || B == 0) return BI_OK;
    if (Lkv == 0) return BI_ERR_INVALID_ARG;   // no key at all
    if (D != 64 && D != 96 && D != 128 && D != 160 && D != 192 && D != 224 && D != 256)
        return BI_ERR_UNSUPPORTED;
    const int64_t G = H / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return BI_ERR_UNSUPPORTED;
    if (qs[3] != 1 || ks[3] != 1 || vs[3] != 1 || os[3] != 1) return BI_ERR_INVALID_ARG;
    for (int i = 0; i < 3; ++i)
        if (qs[i] < 0 || ks[i] < 0 || vs[i] < 0 || os[i] < 0) return BI_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return BI_ERR_ALIGNMENT;
    for (int i = 0; i < 3; ++i)
        if (qs[i] % 8 || ks[i] % 8 || vs[i] % 8 || os[i] % 8) return BI_ERR_ALIGNMENT;
    if (sinks && (reinterpret_cast<uintptr_t>(sinks) & 3u)) return BI_ERR_ALIGNMENT;
    if (Lkv > (int64_t(1) << 31) || q_offset + Lq > (int64_t(1) << 31)) return BI_ERR_UNSUPPORTED;
    bi_status st = check_device();
    if (st != BI_OK) return st;

    SdpaArgs a{};
    a.B = B; a.H = H; a.Hkv = Hkv; a.Lq = Lq; a.Lkv = Lkv; a.q_offset = q_offset;
    a.group = static_cast<int>(G);
    a.qt = static_cast<int>(128 / G);
    a.D = static_cast<int>(D);
    a.dp = D <= 64 ? 64 : D <= 128 ? 128 : 256;
    a.chunk = a.dp == 256 ? 64 : 128;
    a.mode = mask == BI_MASK_CAUSAL ? 1 : mask == BI_MASK_ARRAY ? 2 : 0;
    const double sc = scale > 0.0f ? static_cast<double>(scale) : 1.0 / std::sqrt(static_cast<double>(D));
    a.scale_log2 = static_cast<float>(sc * 1.4426950408889634);   // scale * log2(e)
    a.o = o;
    for (int i = 0; i < 4; ++i) a.os[i] = os[i];
    a.err = device_error_word();
    if (!a.err) return BI_ERR_CUDA;
    a.sinks = sinks;
    a.mask = mask_array;
    if (mask == BI_MASK_ARRAY)
        for (int i = 0; i < 4; ++i) a.ms[i] = ms[i];

    CUtensorMap tq, tk, tv;
    {
        const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(H),
                                  static_cast<uint64_t>(Lq), static_cast<uint64_t>(B)};
        const uint64_t str[3] = {static_cast<uint64_t>(qs[1]) * 2, static_cast<uint64_t>(qs[2]) * 2,
                                 static_cast<uint64_t>(qs[0]) * 2};
        const uint32_t box[4] = {64, static_cast<uint32_t>(G), static_cast<uint32_t>(128 / G), 1};
        st = encode_tmap(&tq, dtype, 4, const_cast<void *>(q), dims, str, box, true);
        if (st != BI_OK) return st;
    }
    {
        const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Lkv),
                                  static_cast<uint64_t>(Hkv), static_cast<uint64_t>(B)};
        // key chunks of 128 (head dims up to 128) or 64 (the 256-column kernel)
        const uint32_t box[4] = {64, static_cast<uint32_t>(a.chunk), 1, 1};
        const uint64_t sk[3] = {static_cast<uint64_t>(ks[2]) * 2, static_cast<uint64_t>(ks[1]) * 2,
                                static_cast<uint64_t>(ks[0]) * 2};
        st = encode_tmap(&tk, dtype, 4, const_cast<void *>(k), dims, sk, box, true);
        if (st != BI_OK) return st;
        const uint64_t sv[3] = {static_cast<uint64_t>(vs[2]) * 2, static_cast<uint64_t>(vs[1]) * 2,
                                static_cast<uint64_t>(vs[0]) * 2};
        st = encode_tmap(&tv, dtype, 4, const_cast<void *>(v), dims, sv, box, true);
        if (st != BI_OK) return st;
    }
    return launch_sdpa(tq, tk, tv, a, dtype, reinterpret_cast<cudaStream_t>(stream));
}

bi_status bi_sdpa(const void *q, const int64_t qs[4], const void *k, const int64_t ks[4],
                  const void *v, const int64_t vs[4], void *o, const int64_t os[4], int64_t B,
                  int64_t H, int64_t Hkv, int64_t Lq, int64_t Lkv, int64_t D, float scale,
                  bi_mask mask, int64_t q_offset, bi_dtype dtype, bi_stream_t stream) {
    if (mask == BI_MASK_ARRAY) return BI_ERR_INVALID_ARG;   // needs the mask: bi_sdpa_ex
    return bi_sdpa_ex(q, qs, k, ks, v, vs, o, os, B, H, Hkv, Lq, Lkv, D, scale, mask, q_offset,
                      nullptr, nullptr, nullptr, dtype, stream);
}

bi_status bi_rmsnorm(const void *x, int64_t ldx, const void *w, void *y, int64_t ldy, int64_t M,
                     int64_t N, float eps, bi_dtype dtype, bi_stream_t stream) {
    if (!valid_dtype(dtype)) return BI_ERR_UNSUPPORTED;
    if (!x || !w || !y || M < 0 || N <= 0 || ldx < N || ldy < N) return BI_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return BI_ERR_INVALID_ARG;
    if (!elem_aligned(x, dtype) || !elem_aligned(w, dtype) || !elem_aligned(y, dtype))
        return BI_ERR_ALIGNMENT;
    if (M == 0) return BI_OK;
    bi_status st = check_device();
    if (st != BI_OK) return st;
    return launch_rmsnorm(x, ldx, w, y, ldy, M, N, eps, dtype, reinterpret_cast<cudaStream_t>(stream));
}

bi_status bi_rope(const void *x, const int64_t xs[4], void *y, const int64_t ys[4], int64_t B,
                  int64_t L, int64_t nh, int64_t D, int64_t pos0, float base, bi_dtype dtype,
                  bi_stream_t stream) {
    if (dtype != BI_BF16 && dtype != BI_F16) return BI_ERR_UNSUPPORTED;
    if (!x || !y || !xs || !ys || B < 0 || L < 0 || nh <= 0 || D <= 0 || (D & 1) || pos0 < 0)
        return BI_ERR_INVALID_ARG;
    if (!(base > 1.0f) || !std::isfinite(base)) return BI_ERR_INVALID_ARG;
    if (xs[3] != 1 || ys[3] != 1) return BI_ERR_INVALID_ARG;
    if (!elem_aligned(x, dtype) || !elem_aligned(y, dtype)) return BI_ERR_ALIGNMENT;
    if (B == 0 || L == 0) return BI_OK;
    bi_status st = check_device();
    if (st != BI_OK) return st;
    return launch_rope(x, xs, y, ys, B, L, nh, D, pos0, base, dtype,
                       reinterpret_cast<cudaStream_t>(stream));
}

bi_status bi_swiglu(const void *gu, int64_t ldgu, void *y, int64_t ldy, int64_t M, int64_t I,
                    bi_dtype dtype, bi_stream_t stream) {
    if (!valid_dtype(dtype)) return BI_ERR_UNSUPPORTED;
    if (!gu || !y || M < 0 || I <= 0 || ldgu < 2 * I || ldy < I) return BI_ERR_INVALID_ARG;
    if (!elem_aligned(gu, dtype) || !elem_aligned(y, dtype)) return BI_ERR_ALIGNMENT;
    if (M == 0) return BI_OK;
    bi_status st = check_device();
    if (st != BI_OK) return st;
    return launch_swiglu(gu, ldgu, y, ldy, M, I, dtype, reinterpret_cast<cudaStream_t>(stream));
}

bi_status bi_add(const void *a, const void *b, void *y, int64_t n, bi_dtype dtype,
                 bi_stream_t stream) {
    if (!valid_dtype(dtype)) return BI_ERR_UNSUPPORTED;
    if (!a || !b || !y || n < 0) return BI_ERR_INVALID_ARG;
    if (!elem_aligned(a, dtype) || !elem_aligned(b, dtype) || !elem_aligned(y, dtype))
        return BI_ERR_ALIGNMENT;
    if (n == 0) return BI_OK;
    bi_status st = check_device();
    if (st != BI_OK) return st;
    return launch_add(a, b, y, n, dtype, reinterpret_cast<cudaStream_t>(stream));
}

bi_status bi_embedding(const int64_t *ids, int64_t n_ids, const void *table, int64_t ldt,
                       int64_t vocab, void *y, int64_t ldy, int64_t dim, bi_dtype dtype,
                       bi_stream_t stream) {
    if (!valid_dtype(dtype)) return BI_ERR_UNSUPPORTED;
    if (!ids || !table || !y || n_ids < 0 || vocab <= 0 || dim <= 0 || ldt < dim || ldy < dim)
        return BI_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ids) & 7u) return BI_ERR_ALIGNMENT;   // read as int64
    if (n_ids > 0x7fffffff) return BI_ERR_UNSUPPORTED;                     // one block per id
    if (n_ids == 0) return BI_OK;
    bi_status st = check_device();
    if (st != BI_OK) return st;
    if (!device_error_word()) return BI_ERR_CUDA;
    return launch_embedding(ids, n_ids, table, ldt, vocab, y, ldy, dim, dtype,
                            reinterpret_cast<cudaStream_t>(stream));
}

bi_status bi_copy4d(const void *src, const int64_t ss[4], void *dst, const int64_t ds[4],
                    const int64_t n[4], bi_dtype dtype, bi_stream_t stream) {
    if (!valid_dtype(dtype)) return BI_ERR_UNSUPPORTED;
    if (!src || !dst || !ss || !ds || !n) return BI_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i)
        if (n[i] < 0 || ss[i] < 0 || ds[i] < 0) return BI_ERR_INVALID_ARG;
    if (ss[3] != 1 || ds[3] != 1) return BI_ERR_INVALID_ARG;
    if (!elem_aligned(src, dtype) || !elem_aligned(dst, dtype)) return BI_ERR_ALIGNMENT;
    if (n[0] * n[1] * n[2] * n[3] == 0) return BI_OK;
    bi_status st = check_device();
    if (st != BI_OK) return st;
    return launch_copy4d(src, ss, dst, ds, n, dtype, reinterpret_cast<cudaStream_t>(stream));
}

const char *bi_status_string(bi_status status) {
    switch (status) {
        case BI_OK: return "BI_OK";
        case BI_ERR_INVALID_ARG: return "BI_ERR_INVALID_ARG: invalid argument";
        case BI_ERR_UNSUPPORTED: return "BI_ERR_UNSUPPORTED: configuration not built";
        case BI_ERR_ALIGNMENT: return "BI_ERR_ALIGNMENT: pointer or stride not 16-byte aligned";
        case BI_ERR_CUDA: return "BI_ERR_CUDA: CUDA runtime or driver error";
        case BI_ERR_TIMEOUT: return "BI_ERR_TIMEOUT: a device-side bounded wait ran out";
        default: return "unknown bi_status";
    }
}

int bi_version(void) { return 100; }   // 0.1.0

bi_status bi_last_device_error(bi_stream_t stream, uint32_t *code) {
    uint32_t *p = device_error_word();
    if (!p) return BI_ERR_CUDA;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return BI_ERR_CUDA;
    uint32_t w = 0;
    if (cudaMemcpy(&w, p, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return BI_ERR_CUDA;
    const uint32_t zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return BI_ERR_CUDA;
    if (code) *code = w;
    if (w & ERR_TIMEOUT) return BI_ERR_TIMEOUT;
    if (w & ERR_BAD_INDEX) return BI_ERR_INVALID_ARG;
    return w ? BI_ERR_CUDA : BI_OK;
}

int64_t bi_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

bi_status bi_debug_wait_probe(int64_t limit_us, bi_stream_t stream) {
    if (limit_us < 1 || limit_us > 2000000) return BI_ERR_INVALID_ARG;
    bi_status st = check_device();
    if (st != BI_OK) return st;
    if (!device_error_word()) return BI_ERR_CUDA;
    return launch_wait_probe(limit_us, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
