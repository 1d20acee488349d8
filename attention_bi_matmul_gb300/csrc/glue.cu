// glue.cu -- row-local decoder ops with a reduction order fixed by construction:
// RMSNorm, rotary embedding, SwiGLU, residual add, embedding gather, a strided
// copy for KV-cache writes, and the bounded-wait test probe.
//
// "mlx-batch-invariant" README, "Why MLX is not invariant" (last paragraph):
// normalisation and elementwise ops are batch-invariant in MLX already.  On
// CUDA that is a property of each kernel's launch shape, so these kernels make
// it structural: every output element depends only on its own row (RMSNorm:
// one block per row, a fixed reduction tree over a fixed thread count) or only
// on its own inputs (the elementwise ops).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_tc.cuh"  // to_f32 / from_f32
#include "internal.cuh"
#include "ptx.cuh"

namespace bi {

namespace {

template <typename T> __device__ __forceinline__ float ld_f32(const T *p) { return to_f32<T>(*p); }
template <> __device__ __forceinline__ float ld_f32<float>(const float *p) { return *p; }
template <typename T> __device__ __forceinline__ void st_f32(T *p, float v) { *p = from_f32<T>(v); }
template <> __device__ __forceinline__ void st_f32<float>(float *p, float v) { *p = v; }

// ---------------------------------------------------------------- RMSNorm
constexpr int RMS_THREADS = 256;

template <typename T>
__global__ void __launch_bounds__(RMS_THREADS) rmsnorm_kernel(const T *__restrict__ x, int64_t ldx,
                                                              const T *__restrict__ w, T *y,
                                                              int64_t ldy, int64_t N, float eps) {
    __shared__ float partial[RMS_THREADS / 32];
    const int64_t m = blockIdx.x;
    const T *xr = x + m * ldx;
    // Thread t sums squares of elements t, t+256, t+512, ... in that order.
    float ss = 0.0f;
    for (int64_t n = threadIdx.x; n < N; n += RMS_THREADS) {
        const float v = ld_f32<T>(xr + n);
        ss = __fmaf_rn(v, v, ss);
    }
    // Fixed butterfly within the warp, then warps 0..7 summed in order.
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    if ((threadIdx.x & 31) == 0) partial[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int i = 0; i < RMS_THREADS / 32; ++i) tot = __fadd_rn(tot, partial[i]);
    const float r = __frsqrt_rn(__fadd_rn(__fdiv_rn(tot, static_cast<float>(N)), eps));
    T *yr = y + m * ldy;
    for (int64_t n = threadIdx.x; n < N; n += RMS_THREADS)
        st_f32<T>(yr + n, __fmul_rn(__fmul_rn(ld_f32<T>(xr + n), r), ld_f32<T>(w + n)));
}

// ---------------------------------------------------------------- RoPE
// Grid: position l x groups of (b, head) pairs.  Each block first forms cos/sin
// of the position's D/2 angles (the angle kept in fp64 so that it keeps its
// precision at long positions), then rotates its (b, head) pairs in fp32 in a
// fixed order.  An output element depends only on its input pair and its
// absolute position.
constexpr int ROPE_MAX_HALF = 256;
constexpr int ROPE_PAIRS_PER_BLOCK = 16;   // (b, head) pairs rotated by one block

// The angle of pair i is theta = pos * r^i with r = base^(-2/D) (r passed in).
// In fp64: r^i by repeated squaring (at most 8 multiplications, relative error
// a few 1e-16), u = theta / pi, and u reduced modulo 2 -- u - 2*rint(u/2) is
// exact.  cos/sin of pi*u then come from the fp32 sincospif of the reduced
// value in [-1, 1].
template <typename T>
__global__ void rope_kernel(const T *x, int64_t xs0, int64_t xs1, int64_t xs2, T *y, int64_t ys0,
                            int64_t ys1, int64_t ys2, int64_t B, int64_t nh, int64_t D,
                            int64_t pos0, double ratio) {
    __shared__ float cs[ROPE_MAX_HALF], sn[ROPE_MAX_HALF];
    const int64_t l = blockIdx.x;
    const int64_t half = D / 2;
    constexpr double INV_PI = 0.31830988618379067154;
    for (int64_t i = threadIdx.x; i < half; i += blockDim.x) {
        double pw = 1.0, bsq = ratio;
        for (int64_t e = i; e; e >>= 1) {
            if (e & 1) pw *= bsq;
            bsq *= bsq;
        }
        const double u = static_cast<double>(pos0 + l) * pw * INV_PI;
        const double ur = u - 2.0 * rint(0.5 * u);
        float sf, cf;
        sincospif(static_cast<float>(ur), &sf, &cf);
        cs[i] = cf;
        sn[i] = sf;
    }
    __syncthreads();
    // this block's share of the position's (b, head) pairs
    const int64_t bh0 = static_cast<int64_t>(blockIdx.y) * ROPE_PAIRS_PER_BLOCK;
    const int64_t nbh = (B * nh - bh0) < ROPE_PAIRS_PER_BLOCK ? (B * nh - bh0) : ROPE_PAIRS_PER_BLOCK;
    const int64_t total = nbh * half;
    for (int64_t idx = threadIdx.x; idx < total; idx += blockDim.x) {
        const int64_t i = idx % half;
        const int64_t bh = bh0 + idx / half;
        const int64_t h = bh % nh, b = bh / nh;
        const T *xp = x + b * xs0 + l * xs1 + h * xs2;
        T *yp = y + b * ys0 + l * ys1 + h * ys2;
        const float c = cs[i], sv = sn[i];
        const float x0 = to_f32<T>(xp[i]), x1 = to_f32<T>(xp[i + half]);
        const float y0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, sv));
        const float y1 = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, sv));
        yp[i] = from_f32<T>(y0);
        yp[i + half] = from_f32<T>(y1);
    }
}

// ---------------------------------------------------------------- SwiGLU
template <typename T>
__device__ __forceinline__ float swiglu1(float g, float u) {
    const float silu = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
    return __fmul_rn(silu, u);
}

template <typename T>
__global__ void swiglu_kernel(const T *gu, int64_t ldgu, T *y, int64_t ldy, int64_t M, int64_t I) {
    const int64_t total = M * I;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = idx / I, i = idx - (idx / I) * I;
        const float g = ld_f32<T>(gu + m * ldgu + i);
        const float u = ld_f32<T>(gu + m * ldgu + I + i);
        st_f32<T>(y + m * ldy + i, swiglu1<T>(g, u));
    }
}

// 8 consecutive outputs per thread (16-byte loads/stores); same per-element arithmetic.
template <typename T>
__global__ void swiglu_vec8_kernel(const T *gu, int64_t ldgu, T *y, int64_t ldy, int64_t M,
                                   int64_t I) {
    const int64_t per_row = I / 8;
    const int64_t total = M * per_row;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = idx / per_row, i = (idx - m * per_row) * 8;
        union V { uint4 u; T h[8]; } g, u, o;
        g.u = *reinterpret_cast<const uint4 *>(gu + m * ldgu + i);
        u.u = *reinterpret_cast<const uint4 *>(gu + m * ldgu + I + i);
#pragma unroll
        for (int e = 0; e < 8; ++e)
            o.h[e] = from_f32<T>(swiglu1<T>(to_f32<T>(g.h[e]), to_f32<T>(u.h[e])));
        *reinterpret_cast<uint4 *>(y + m * ldy + i) = o.u;
    }
}

// ---------------------------------------------------------------- add
template <typename T>
__global__ void add_kernel(const T *a, const T *b, T *y, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        st_f32<T>(y + i, __fadd_rn(ld_f32<T>(a + i), ld_f32<T>(b + i)));
}

template <typename T>
__global__ void add_vec8_kernel(const T *a, const T *b, T *y, int64_t n8) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8;
         i += (int64_t)gridDim.x * blockDim.x) {
        union V { uint4 u; T h[8]; } x, z, o;
        x.u = reinterpret_cast<const uint4 *>(a)[i];
        z.u = reinterpret_cast<const uint4 *>(b)[i];
#pragma unroll
        for (int e = 0; e < 8; ++e) o.h[e] = from_f32<T>(__fadd_rn(to_f32<T>(x.h[e]), to_f32<T>(z.h[e])));
        reinterpret_cast<uint4 *>(y)[i] = o.u;
    }
}

// ---------------------------------------------------------------- embedding / copy (bytes)
__global__ void embedding_kernel(const int64_t *ids, int64_t n_ids, const uint8_t *table,
                                 int64_t ldt_bytes, int64_t vocab, uint8_t *y, int64_t ldy_bytes,
                                 int64_t row_bytes, uint32_t *err) {
    const int64_t t = blockIdx.x;
    if (t >= n_ids) return;
    const int64_t id = ids[t];
    const bool ok = id >= 0 && id < vocab;
    if (!ok && threadIdx.x == 0) atomicOr(err, ERR_BAD_INDEX);
    uint8_t *dst = y + t * ldy_bytes;
    const uint8_t *src = table + (ok ? id : 0) * ldt_bytes;
    if (((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | row_bytes) & 15) == 0) {
        const uint4 zero = make_uint4(0, 0, 0, 0);
        for (int64_t i = threadIdx.x; i < row_bytes / 16; i += blockDim.x)
            reinterpret_cast<uint4 *>(dst)[i] = ok ? reinterpret_cast<const uint4 *>(src)[i] : zero;
    } else {
        for (int64_t i = threadIdx.x; i < row_bytes; i += blockDim.x) dst[i] = ok ? src[i] : 0;
    }
}

template <typename T>
__global__ void copy4d_kernel(const T *src, int64_t s0, int64_t s1, int64_t s2, T *dst, int64_t d0,
                              int64_t d1, int64_t d2, int64_t n0, int64_t n1, int64_t n2,
                              int64_t n3) {
    const int64_t total = n0 * n1 * n2 * n3;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i3 = idx % n3;
        int64_t r = idx / n3;
        const int64_t i2 = r % n2;
        r /= n2;
        const int64_t i1 = r % n1;
        const int64_t i0 = r / n1;
        dst[i0 * d0 + i1 * d1 + i2 * d2 + i3] = src[i0 * s0 + i1 * s1 + i2 * s2 + i3];
    }
}

// ---------------------------------------------------------------- bounded-wait probe
__global__ void wait_probe_kernel(uint64_t limit_ns, uint32_t *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        // Nothing ever arrives on `bar`: the wait must run out.
        if (!mbar_wait_limited(&bar, 0, limit_ns)) atomicOr(err, ERR_TIMEOUT);
    }
}

int grid_for(int64_t total, int threads) {
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

}  // namespace

#define BI_DISPATCH_T(dt, ...)                                                   \
    do {                                                                         \
        if ((dt) == BI_BF16) { using T = __nv_bfloat16; __VA_ARGS__; }           \
        else if ((dt) == BI_F16) { using T = __half; __VA_ARGS__; }              \
        else if ((dt) == BI_F32) { using T = float; __VA_ARGS__; }               \
        else return BI_ERR_UNSUPPORTED;                                          \
    } while (0)

bi_status launch_rmsnorm(const void *x, int64_t ldx, const void *w, void *y, int64_t ldy,
                         int64_t M, int64_t N, float eps, bi_dtype dt, cudaStream_t s) {
    if (M > 0x7fffffff) return BI_ERR_UNSUPPORTED;
    BI_DISPATCH_T(dt, rmsnorm_kernel<T><<<static_cast<unsigned>(M), RMS_THREADS, 0, s>>>(
                          static_cast<const T *>(x), ldx, static_cast<const T *>(w),
                          static_cast<T *>(y), ldy, N, eps));
    count_launch();
    return cuda_status(cudaGetLastError());
}

bi_status launch_rope(const void *x, const int64_t xs[4], void *y, const int64_t ys[4], int64_t B,
                      int64_t L, int64_t nh, int64_t D, int64_t pos0, float base, bi_dtype dt,
                      cudaStream_t s) {
    const double ratio = pow(static_cast<double>(base), -2.0 / static_cast<double>(D));
    if (dt == BI_F32) return BI_ERR_UNSUPPORTED;
    if (D / 2 > ROPE_MAX_HALF || L > 0x7fffffff) return BI_ERR_UNSUPPORTED;
    const int64_t bh_blocks = (B * nh + ROPE_PAIRS_PER_BLOCK - 1) / ROPE_PAIRS_PER_BLOCK;
    if (bh_blocks > 65535) return BI_ERR_UNSUPPORTED;
    if (dt == BI_BF16) {
        using T = __nv_bfloat16;
        rope_kernel<T><<<dim3(static_cast<unsigned>(L), static_cast<unsigned>(bh_blocks)), 256, 0, s>>>(
            static_cast<const T *>(x), xs[0], xs[1], xs[2], static_cast<T *>(y), ys[0], ys[1],
            ys[2], B, nh, D, pos0, ratio);
    } else {
        using T = __half;
        rope_kernel<T><<<dim3(static_cast<unsigned>(L), static_cast<unsigned>(bh_blocks)), 256, 0, s>>>(
            static_cast<const T *>(x), xs[0], xs[1], xs[2], static_cast<T *>(y), ys[0], ys[1],
            ys[2], B, nh, D, pos0, ratio);
    }
    count_launch();
    return cuda_status(cudaGetLastError());
}

bi_status launch_swiglu(const void *gu, int64_t ldgu, void *y, int64_t ldy, int64_t M, int64_t I,
                        bi_dtype dt, cudaStream_t s) {
    const bool vec = dt != BI_F32 && I % 8 == 0 && ldgu % 8 == 0 && ldy % 8 == 0 &&
                     ((reinterpret_cast<uintptr_t>(gu) | reinterpret_cast<uintptr_t>(y)) & 15) == 0;
    if (vec) {
        BI_DISPATCH_T(dt, swiglu_vec8_kernel<T><<<grid_for(M * I / 8, 256), 256, 0, s>>>(
                              static_cast<const T *>(gu), ldgu, static_cast<T *>(y), ldy, M, I));
    } else {
        BI_DISPATCH_T(dt, swiglu_kernel<T><<<grid_for(M * I, 256), 256, 0, s>>>(
                              static_cast<const T *>(gu), ldgu, static_cast<T *>(y), ldy, M, I));
    }
    count_launch();
    return cuda_status(cudaGetLastError());
}

bi_status launch_add(const void *a, const void *b, void *y, int64_t n, bi_dtype dt,
                     cudaStream_t s) {
    const bool vec = dt != BI_F32 && n % 8 == 0 &&
                     ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
                       reinterpret_cast<uintptr_t>(y)) & 15) == 0;
    if (vec) {
        BI_DISPATCH_T(dt, add_vec8_kernel<T><<<grid_for(n / 8, 256), 256, 0, s>>>(
                              static_cast<const T *>(a), static_cast<const T *>(b),
                              static_cast<T *>(y), n / 8));
    } else {
        BI_DISPATCH_T(dt, add_kernel<T><<<grid_for(n, 256), 256, 0, s>>>(
                              static_cast<const T *>(a), static_cast<const T *>(b),
                              static_cast<T *>(y), n));
    }
    count_launch();
    return cuda_status(cudaGetLastError());
}

bi_status launch_embedding(const int64_t *ids, int64_t n_ids, const void *table, int64_t ldt,
                           int64_t vocab, void *y, int64_t ldy, int64_t dim, bi_dtype dt,
                           cudaStream_t s) {
    const int64_t es = dt == BI_F32 ? 4 : 2;
    if (n_ids > 0x7fffffff) return BI_ERR_UNSUPPORTED;
    embedding_kernel<<<static_cast<unsigned>(n_ids), 256, 0, s>>>(
        ids, n_ids, static_cast<const uint8_t *>(table), ldt * es, vocab,
        static_cast<uint8_t *>(y), ldy * es, dim * es, device_error_word());
    count_launch();
    return cuda_status(cudaGetLastError());
}

bi_status launch_copy4d(const void *src, const int64_t ss[4], void *dst, const int64_t ds[4],
                        const int64_t n[4], bi_dtype dt, cudaStream_t s) {
    const int64_t total = n[0] * n[1] * n[2] * n[3];
    if (dt == BI_F32) {
        copy4d_kernel<float><<<grid_for(total, 256), 256, 0, s>>>(
            static_cast<const float *>(src), ss[0], ss[1], ss[2], static_cast<float *>(dst),
            ds[0], ds[1], ds[2], n[0], n[1], n[2], n[3]);
    } else {
        copy4d_kernel<uint16_t><<<grid_for(total, 256), 256, 0, s>>>(
            static_cast<const uint16_t *>(src), ss[0], ss[1], ss[2], static_cast<uint16_t *>(dst),
            ds[0], ds[1], ds[2], n[0], n[1], n[2], n[3]);
    }
    count_launch();
    return cuda_status(cudaGetLastError());
}

bi_status launch_wait_probe(int64_t limit_us, cudaStream_t s) {
    wait_probe_kernel<<<1, 32, 0, s>>>(static_cast<uint64_t>(limit_us) * 1000ull,
                                       device_error_word());
    count_launch();
    return cuda_status(cudaGetLastError());
}

}  // namespace bi
