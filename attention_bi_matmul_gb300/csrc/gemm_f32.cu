// gemm_f32.cu -- batch-invariant fp32 GEMM on the CUDA cores.
//
// "mlx-batch-invariant" README, "How the kernels work" / GEMM and "Accuracy":
// one sequential pass over K per output element (the README accepts that this
// costs some accuracy against a pairwise/split-K sum; it is what fixes the
// order).  Every output is acc = fma(a[m,k], b[k,n], acc) for k = 0, 1, ..., K-1
// starting from acc = 0, so its bits depend on row m of a and column n of b
// only -- never on M, the tile, or the grid.
//
// Register tiling: a 64x64 block tile, 256 threads, 4x4 outputs per thread,
// K staged through shared memory 16 at a time.
#include "internal.cuh"
#include "ptx.cuh"

namespace bi {

namespace {

constexpr int F_BM = 64, F_BN = 64, F_BK = 16, F_TM = 4, F_TN = 4;

// B_NK: b is w[N,K] (linear layout); otherwise b is [K,N].
template <bool B_NK>
__global__ void __launch_bounds__(256) gemm_f32_kernel(const float *__restrict__ a, int64_t lda,
                                                       const float *__restrict__ b, int64_t ldb,
                                                       const GemmArgs args) {
    __shared__ float As[F_BK][F_BM + 4];
    __shared__ float Bs[F_BK][F_BN + 4];
    const int64_t M = args.M, N = args.N, K = args.K;
    const int64_t e = blockIdx.z;                  // batch entry
    a += e * args.sa;
    b += e * args.sb;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * F_BM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * F_BN;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;

    float acc[F_TM][F_TN];
#pragma unroll
    for (int i = 0; i < F_TM; ++i)
#pragma unroll
        for (int j = 0; j < F_TN; ++j) acc[i][j] = 0.0f;

    for (int64_t k0 = 0; k0 < K; k0 += F_BK) {
        // Stage a[m0:m0+64, k0:k0+16] and b's matching 16 x 64 block (zero outside).
        for (int idx = threadIdx.x; idx < F_BK * F_BM; idx += 256) {
            const int kk = idx % F_BK, mm = idx / F_BK;
            const int64_t m = m0 + mm, k = k0 + kk;
            As[kk][mm] = (m < M && k < K) ? a[m * lda + k] : 0.0f;
        }
        for (int idx = threadIdx.x; idx < F_BK * F_BN; idx += 256) {
            int kk, nn;
            if (B_NK) { kk = idx % F_BK; nn = idx / F_BK; }
            else { nn = idx % F_BN; kk = idx / F_BN; }
            const int64_t n = n0 + nn, k = k0 + kk;
            float val = 0.0f;
            if (n < N && k < K) val = B_NK ? b[n * ldb + k] : b[k * ldb + n];
            Bs[kk][nn] = val;
        }
        __syncthreads();
        // Only the real k < K steps are applied, so the chain is exactly K long.
        const int kend = (K - k0) < F_BK ? static_cast<int>(K - k0) : F_BK;
        for (int kk = 0; kk < kend; ++kk) {
            float av[F_TM], bv[F_TN];
#pragma unroll
            for (int i = 0; i < F_TM; ++i) av[i] = As[kk][ty * F_TM + i];
#pragma unroll
            for (int j = 0; j < F_TN; ++j) bv[j] = Bs[kk][tx * F_TN + j];
#pragma unroll
            for (int i = 0; i < F_TM; ++i)
#pragma unroll
                for (int j = 0; j < F_TN; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }

    // Epilogue, fixed order in fp32 (same rule as the tensor-core path):
    //   bias:  y = acc + bias[n];   addmm: y = (alpha * acc) + (beta * c).
    float *y = static_cast<float *>(args.y) + e * args.sy;
#pragma unroll
    for (int i = 0; i < F_TM; ++i) {
        const int64_t m = m0 + ty * F_TM + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < F_TN; ++j) {
            const int64_t n = n0 + tx * F_TN + j;
            if (n >= N) continue;
            float v = acc[i][j];
            if (args.epi == EPI_BIAS) {
                v = __fadd_rn(v, static_cast<const float *>(args.bias)[n]);
            } else if (args.epi == EPI_ADDMM) {
                const float *c = static_cast<const float *>(args.c);
                const float cv = args.ldc ? c[m * args.ldc + n] : c[n];
                v = __fadd_rn(__fmul_rn(args.alpha, v), __fmul_rn(args.beta, cv));
            }
            y[m * args.ldy + n] = v;
        }
    }
}

}  // namespace

bi_status launch_gemm_f32(const float *a, int64_t lda, const float *b, int64_t ldb, bool b_nk,
                          const GemmArgs &args, cudaStream_t s) {
    const int64_t gx = (args.N + F_BN - 1) / F_BN;
    const int64_t gy = (args.M + F_BM - 1) / F_BM;
    if (gx > 0x7fffffff || gy > 65535 || args.batch > 65535) return BI_ERR_UNSUPPORTED;
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy),
              static_cast<unsigned>(args.batch));
    if (b_nk)
        gemm_f32_kernel<true><<<grid, 256, 0, s>>>(a, lda, b, ldb, args);
    else
        gemm_f32_kernel<false><<<grid, 256, 0, s>>>(a, lda, b, ldb, args);
    count_launch();
    return cuda_status(cudaGetLastError());
}

}  // namespace bi
