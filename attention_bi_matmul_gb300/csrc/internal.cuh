// internal.cuh -- declarations shared by the library's translation units.
// Not part of the public ABI (that is include/bi.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bi.h"

namespace bi {

// Epilogue kinds of the GEMM kernels.
enum Epilogue : int { EPI_NONE = 0, EPI_BIAS = 1, EPI_ADDMM = 2 };

struct GemmArgs {
    int64_t M, N, K;
    void *y;
    int64_t ldy;
    const void *bias;  // EPI_BIAS
    const void *c;     // EPI_ADDMM
    int64_t ldc;       // 0: c is one row [N]
    float alpha, beta; // EPI_ADDMM
    int epi;
    uint32_t *err;     // device error word
    int a_rows;        // rows of A each copy moves: min(128, M rounded up to 16)
    // Batched calls: `batch` independent problems of the same shape (1 otherwise).
    // Entry e reads a + e*sa and b + e*sb and writes y + e*sy (elements); a stride
    // of 0 shares that operand across the batch.
    int64_t batch;
    int64_t sa, sb, sy;
};

// Tile configuration of the tensor-core GEMM for one (N, K, dtype, layout).
struct TcConfig {
    int block_n;
    int stages;
    bool pair;      // 256-row tiles on a CTA pair (cta_group::2)
};

// ---- host helpers (api.cu)
uint32_t *device_error_word();                   // per current device, cached
int device_sm_count();                           // per current device, cached
void count_launch();                             // launch counter
bi_status encode_tmap(CUtensorMap *map, bi_dtype dt, int rank, void *base,
                      const uint64_t *dims, const uint64_t *strides_bytes,
                      const uint32_t *box, bool swizzle128);
bi_status encode_tmap_u32(CUtensorMap *map, int rank, void *base, const uint64_t *dims,
                          const uint64_t *strides_bytes, const uint32_t *box, bool swizzle128);
TcConfig tc_config(int64_t N, int64_t K, bi_dtype dt, bool b_mn_major);
bi_status cuda_status(cudaError_t e);

// ---- per-device initialisation of each translation unit (kernel attributes)
bi_status init_gemm_tc_bf16();
bi_status init_gemm_tc_f16();
bi_status init_sdpa();
bi_status init_qgemm();

// ---- launchers
bi_status launch_gemm_f32(const float *a, int64_t lda, const float *b, int64_t ldb, bool b_nk,
                          const GemmArgs &args, cudaStream_t s);
bi_status launch_gemm_tc(const void *a, int64_t lda, const void *b, int64_t ldb, bool b_nk,
                         const GemmArgs &args, bi_dtype dt, const TcConfig &cfg, cudaStream_t s);

// Group-wise affine quantized linear: y[M,N] = x[M,K] . w^T (+ bias), with
// w[n,k] = rnd(scales[n,g] * q[n,k] + biases[n,g]), g = k / group_size.
struct QGemmArgs {
    int64_t M, N, K;
    const void *scales, *biases;  // [N, ldsb] in the activation dtype
    int64_t ldsb;
    int group_size;               // 32, 64 or 128
    const void *bias;             // [N] or null
    void *y;
    int64_t ldy;
    uint32_t *err;
    int x_rows;                   // token rows each x copy moves: min(64, M rounded up to 16)
};
bi_status launch_qgemm(const void *x, int64_t ldx, const uint32_t *wq, int64_t ldq, int bits,
                       const QGemmArgs &args, bi_dtype dt, cudaStream_t s);

struct SdpaArgs {
    int64_t B, H, Hkv, Lq, Lkv, q_offset;
    int group;         // H / Hkv
    int qt;            // query positions per tile = 128 / group
    int D;             // head dim (64, 96, 128, 160, 192, 224 or 256)
    int dp;            // padded head dim of the kernel: 64, 128 or 256
    int chunk;         // keys per chunk: 128 up to head dim 128, 64 above
    int mode;          // 0: no mask, 1: causal, 2: boolean array mask
    float scale_log2;  // scale * log2(e)
    void *o;
    int64_t os[4];
    uint32_t *err;
    const float *sinks;     // [H] sink logits (units of the scaled scores), or null
    const uint8_t *mask;    // mode 2: mask[b*ms[0] + h*ms[1] + i*ms[2] + j], nonzero = visible
    int64_t ms[4];
};
bi_status launch_sdpa(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                      const SdpaArgs &args, bi_dtype dt, cudaStream_t s);

bi_status launch_rmsnorm(const void *x, int64_t ldx, const void *w, void *y, int64_t ldy,
                         int64_t M, int64_t N, float eps, bi_dtype dt, cudaStream_t s);
bi_status launch_rope(const void *x, const int64_t xs[4], void *y, const int64_t ys[4],
                      int64_t B, int64_t L, int64_t nh, int64_t D, int64_t pos0, float base,
                      bi_dtype dt, cudaStream_t s);
bi_status launch_swiglu(const void *gu, int64_t ldgu, void *y, int64_t ldy, int64_t M, int64_t I,
                        bi_dtype dt, cudaStream_t s);
bi_status launch_add(const void *a, const void *b, void *y, int64_t n, bi_dtype dt,
                     cudaStream_t s);
bi_status launch_embedding(const int64_t *ids, int64_t n_ids, const void *table, int64_t ldt,
                           int64_t vocab, void *y, int64_t ldy, int64_t dim, bi_dtype dt,
                           cudaStream_t s);
bi_status launch_copy4d(const void *src, const int64_t ss[4], void *dst, const int64_t ds[4],
                        const int64_t n[4], bi_dtype dt, cudaStream_t s);
bi_status launch_wait_probe(int64_t limit_us, cudaStream_t s);

}  // namespace bi
