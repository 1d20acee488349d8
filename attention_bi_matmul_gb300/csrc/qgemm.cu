// qgemm.cu -- batch-invariant group-wise affine quantized linear on the tensor cores.
//
// "mlx-batch-invariant" README, "Quantized models": 2, 4 and 8-bit affine
// weights are unpacked inside the K loop of one fused invariant kernel, so a
// quantized layer keeps the GEMM's rule -- every output is one reduction over K
// in an order fixed by K alone, whatever the number of tokens.  Format (the
// plain affine reading): per group of `group_size` consecutive k of weight row
// n, w[n,k] = scales[n,g] * q[n,k] + biases[n,g], with q the unsigned `bits`-wide
// field (k mod 32/bits) of 32-bit word k / (32/bits) of row n, fields counted
// from the least significant bit.
//
// The GB300 form:
//   * the weight rows fill the MMA's 128-row M side and the tokens its fixed
//     64-wide N side: D[n, m] = sum_k w[n,k] x[m,k] (y = D^T).  A decode step
//     therefore pays for 64 token columns, not 128 rows; a token's output
//     depends only on its own x row, as in the plain GEMM;
//   * the dequantised weight of an element is rnd(s * q + b) with ONE rounding
//     to the activation dtype: a packed 16-bit fused multiply-add with q exact
//     in that type.  It depends on (q, s, b) only, never on M or the tile;
//   * K is visited in ascending 64-wide panels, each as four K = 16 MMAs from a
//     zero accumulator -- for every M.  No split-K, no atomics;
//   * epilogue: + bias in fp32, one rounding, y[m, n] stored (32 consecutive n
//     per warp and token: 64-byte segments).
//
// Roles (320 threads, persistent over (n block, token block) tiles):
//   warp 0 lane 0   TMA producer: per panel the x panel (64 tokens x 64 k,
//                   128-byte swizzle) and the packed weight panel (128 rows x
//                   8*bits bytes) into one ring stage; L2 prefetch of the
//                   weight panels one ring further on
//   warp 1          TMEM allocation (128 columns: two 64-column accumulators);
//                   lane 0 issues the MMAs
//   warps 2..9      dequantisers: warp w owns weight rows 32*(w%4)..+31 and
//                   half (w-2)/4 of each panel's 64 k; they write the 16-bit
//                   weight panel in the tensor cores' swizzled K-major layout.
//                   After a tile's last panel they run its epilogue (the warp's
//                   TMEM lane quarter, token columns 32*half..+31).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_tc.cuh"  // IsBf16 / to_f32 / from_f32
#include "internal.cuh"
#include "ptx.cuh"

namespace bi {

namespace {

constexpr int QG_N = 128;      // weight rows per tile (MMA M)
constexpr int QG_T = 64;       // tokens per tile (MMA N)
constexpr int QG_K = 64;       // k per panel
constexpr int QG_THREADS = 320;
constexpr int QG_DS = 4;       // dequantised weight panels in flight
constexpr uint32_t QG_XP = QG_T * QG_K * 2;     // 8 KB x panel
constexpr uint32_t QG_AP = QG_N * QG_K * 2;     // 16 KB dequantised weight panel
constexpr uint32_t QG_TMEM_COLS = 2 * QG_T;     // 128

// Raw ring depth by width: enough packed weight bytes in flight per SM.
template <int BITS> __host__ __device__ constexpr int qg_rs() {
    return BITS == 2 ? 10 : BITS == 4 ? 8 : 6;
}
template <int BITS> __host__ __device__ constexpr uint32_t qg_wraw() {
    return QG_N * QG_K * BITS / 8;   // packed bytes of one weight panel
}

template <int BITS>
struct QgSmem {
    static constexpr uint32_t RS = qg_rs<BITS>();
    // byte offsets from the 1024-aligned base
    static constexpr uint32_t X = 0;                                // [RS] x panels
    static constexpr uint32_t A = X + RS * QG_XP;                   // [DS] weight panels
    static constexpr uint32_t W = A + QG_DS * QG_AP;                // [RS] packed panels
    static constexpr uint32_t BARS = W + RS * qg_wraw<BITS>();
    // raw_full[RS] raw_empty[RS] a_full[DS] a_empty[DS] tfull[2] tempty[2] mma_done
    static constexpr uint32_t NBARS = 2 * RS + 2 * QG_DS + 4 + 1;
    static constexpr uint32_t MISC = BARS + NBARS * 8;               // tmem slot, abort flag
    static constexpr uint32_t END = MISC + 16;
    static constexpr size_t BYTES = 1024 + END;
};

// Fields 2j and 2j+1 (bit offsets OA and OA + BITS) of w in the two 16-bit halves.
template <int BITS, int OA>
__device__ __forceinline__ uint32_t field_pair(uint32_t w) {
    constexpr uint32_t MASK = (1u << BITS) - 1u;
    constexpr int OB = OA + BITS;
    const uint32_t lo = w >> OA;
    const uint32_t hi = OB >= 16 ? (w >> (OB - 16)) : (w << (16 - OB));
    return (lo & MASK) | (hi & (MASK << 16));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

template <typename T> struct Pair;
template <> struct Pair<__nv_bfloat16> { using t = __nv_bfloat162; };
template <> struct Pair<__half> { using t = __half2; };

template <typename P> __device__ __forceinline__ P as_pair(uint32_t u) {
    return *reinterpret_cast<P *>(&u);
}
template <typename P> __device__ __forceinline__ uint32_t as_u32(P p) {
    return *reinterpret_cast<uint32_t *>(&p);
}

// q pair (exact small integers in the 16-bit type) from two fields in 16-bit halves:
// the field becomes the low mantissa bits of a constant whose unit in the last
// place is 1 (bf16 128 + q for q < 128, fp16 1024 + q for q < 1024), then the
// constant is subtracted exactly.
template <typename T> __device__ __forceinline__ uint32_t q_pair(uint32_t halves);
template <> __device__ __forceinline__ uint32_t q_pair<__nv_bfloat16>(uint32_t halves) {
    const __nv_bfloat162 v = as_pair<__nv_bfloat162>(halves | 0x43004300u);   // 128 + q
    return as_u32(__hsub2(v, as_pair<__nv_bfloat162>(0x43004300u)));
}
template <> __device__ __forceinline__ uint32_t q_pair<__half>(uint32_t halves) {
    const __half2 v = as_pair<__half2>(halves | 0x64006400u);                 // 1024 + q
    return as_u32(__hsub2(v, as_pair<__half2>(0x64006400u)));
}

// rnd(s * q + b) for a pair: one fused multiply-add, one rounding.
template <typename T>
__device__ __forceinline__ uint32_t deq_pair(uint32_t q2, uint32_t s2, uint32_t b2) {
    using P = typename Pair<T>::t;
    return as_u32(__hfma2(as_pair<P>(q2), as_pair<P>(s2), as_pair<P>(b2)));
}

// Eight consecutive weights (one 16-byte chunk of a panel row) from the packed
// words that hold them: BITS = 4 one word, 8 two words, 2 the low or high half
// of a word (`sub` = 0 / 1).
template <typename T, int BITS>
__device__ __forceinline__ uint4 deq8(const uint32_t *w, int sub, uint32_t s2, uint32_t b2) {
    uint32_t q[4];
    if constexpr (BITS == 4) {
        q[0] = q_pair<T>(field_pair<4, 0>(w[0]));
        q[1] = q_pair<T>(field_pair<4, 8>(w[0]));
        q[2] = q_pair<T>(field_pair<4, 16>(w[0]));
        q[3] = q_pair<T>(field_pair<4, 24>(w[0]));
    } else if constexpr (BITS == 2) {
        const uint32_t v = sub ? (w[0] >> 16) : w[0];
        q[0] = q_pair<T>(field_pair<2, 0>(v));
        q[1] = q_pair<T>(field_pair<2, 4>(v));
        q[2] = q_pair<T>(field_pair<2, 8>(v));
        q[3] = q_pair<T>(field_pair<2, 12>(v));
    } else {   // BITS == 8
        if constexpr (IsBf16<T>::value) {
            // q up to 255 needs 8 significant bits: form it exactly in fp32
            // (2^23 + q, minus 2^23) and convert the pair exactly to bf16.
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t wd = w[i >> 1];
                const uint32_t j = (i & 1) * 2;
                const float fa = __uint_as_float(prmt(wd, 0x4B000000u, 0x7650u + j)) - 8388608.0f;
                const float fb = __uint_as_float(prmt(wd, 0x4B000000u, 0x7651u + j)) - 8388608.0f;
                q[i] = as_u32(__floats2bfloat162_rn(fa, fb));
            }
        } else {
            // bytes (2i, 2i+1) of the two words straight into the fp16 halves
            q[0] = q_pair<T>(prmt(w[0], 0u, 0x7170u) & 0x00FF00FFu);
            q[1] = q_pair<T>(prmt(w[0], 0u, 0x7372u) & 0x00FF00FFu);
            q[2] = q_pair<T>(prmt(w[1], 0u, 0x7170u) & 0x00FF00FFu);
            q[3] = q_pair<T>(prmt(w[1], 0u, 0x7372u) & 0x00FF00FFu);
        }
    }
    return make_uint4(deq_pair<T>(q[0], s2, b2), deq_pair<T>(q[1], s2, b2),
                      deq_pair<T>(q[2], s2, b2), deq_pair<T>(q[3], s2, b2));
}

__device__ __forceinline__ uint32_t ld_u16_nc(const void *p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

template <typename T, int BITS>
__global__ void __launch_bounds__(QG_THREADS, 1)
    qgemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 const QGemmArgs args) {
    using S = QgSmem<BITS>;
    constexpr int RS = S::RS;
    constexpr uint32_t WRAW = qg_wraw<BITS>();
    constexpr uint32_t WROW = QG_K * BITS / 8;          // packed bytes of one row's panel
    constexpr int WPP = QG_K * BITS / 32;               // packed words of one row's panel
    constexpr uint32_t IDESC = mma_idesc(IsBf16<T>::value, QG_N, QG_T, false);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sX = smem + S::X;
    uint8_t *sA = smem + S::A;
    uint8_t *sW = smem + S::W;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::BARS);
    uint64_t *raw_full = bars;
    uint64_t *raw_empty = raw_full + RS;
    uint64_t *a_full = raw_empty + RS;
    uint64_t *a_empty = a_full + QG_DS;
    uint64_t *tfull = a_empty + QG_DS;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int64_t M = args.M, N = args.N, K = args.K;
    const int64_t num_n = (N + QG_N - 1) / QG_N;
    const int64_t num_t = (M + QG_T - 1) / QG_T;
    const int64_t total = num_n * num_t;
    const int KP = static_cast<int>(K / QG_K);          // panels per tile (K % 64 == 0)

    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], 1 + 8);   // the MMA's commit (x) + 8 dequantisers (w)
        }
        for (int d = 0; d < QG_DS; ++d) {
            mbar_init(&a_full[d], 8);
            mbar_init(&a_empty[d], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 8);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, QG_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            prefetch_tmap(&tmX);
            prefetch_tmap(&tmW);
            const uint32_t tx = static_cast<uint32_t>(args.x_rows) * QG_K * 2 + WRAW;
            uint32_t it = 0, s = 0, ph = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; ok && t < total; t += gridDim.x) {
                const int64_t nb = t % num_n, tb = t / num_n;
                const int32_t wrow = static_cast<int32_t>(nb * QG_N);
                for (int p = 0; p < RS && p < KP; ++p)
                    tma_prefetch_2d(&tmW, p * WPP, wrow);
                for (int p = 0; p < KP; ++p, ++it) {
                    if (!mbar_wait(&raw_empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&raw_full[s], tx);
                    tma_load_2d(sX + s * QG_XP, &tmX, &raw_full[s], p * QG_K,
                                static_cast<int32_t>(tb * QG_T));
                    tma_load_2d(sW + s * WRAW, &tmW, &raw_full[s], p * WPP, wrow);
                    if (p + RS < KP) tma_prefetch_2d(&tmW, (p + RS) * WPP, wrow);
                    if (++s == RS) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // Let every copy already issued land before the block can exit.
                const uint32_t first = it > static_cast<uint32_t>(RS) ? it - RS : 0;
                for (uint32_t i = first; i < it; ++i)
                    mbar_wait_limited(&raw_full[i % RS], (i / RS) & 1u, WAIT_LIMIT_NS);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            const uint64_t a_desc0 = smem_desc(smem_u32(sA), 16, 1024);
            const uint64_t x_desc0 = smem_desc(smem_u32(sX), 16, 1024);
            uint32_t tc = 0, s = 0, ph = 0, d = 0, dph = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; ok && t < total; t += gridDim.x, ++tc) {
                const uint32_t acc = tc & 1u;
                if (!mbar_wait(&tempty[acc], ((tc >> 1) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * QG_T;
                for (int p = 0; p < KP; ++p) {
                    if (!mbar_wait(&a_full[d], dph, abort_flag)) { ok = false; break; }
                    if (!mbar_wait(&raw_full[s], ph, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = a_desc0 + ((d * QG_AP) >> 4);
                    const uint64_t xd = x_desc0 + ((s * QG_XP) >> 4);
#pragma unroll
                    for (int j = 0; j < QG_K / 16; ++j)
                        mma_f16_ss(d_tmem, ad + j * (32 >> 4), xd + j * (32 >> 4), IDESC,
                                   (p | j) != 0 ? 1u : 0u);
                    mma_commit(&a_empty[d]);
                    mma_commit(&raw_empty[s]);
                    if (++d == QG_DS) { d = 0; dph ^= 1u; }
                    if (++s == RS) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
            }
            // All issued MMAs must be complete before TMEM is released.
            mma_commit(mma_done);
            mbar_wait_limited(mma_done, 0, WAIT_LIMIT_NS);
        }
    } else {
        // ------------------------------------------------ dequantisers + epilogue (2..9)
        using Tv = T;
        const uint32_t quarter = static_cast<uint32_t>(warp & 3);
        const int half = (warp - 2) >> 2;
        const int r = static_cast<int>(quarter) * 32 + lane;     // weight row in the tile
        const int gs = args.group_size;
        const Tv *scales = static_cast<const Tv *>(args.scales);
        const Tv *biases = static_cast<const Tv *>(args.biases);
        uint32_t tc = 0, s = 0, ph = 0, d = 0, dph = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; ok && t < total; t += gridDim.x, ++tc) {
            const int64_t nb = t % num_n, tb = t / num_n;
            const int64_t n = nb * QG_N + r;
            const bool nvalid = n < N;
            const int64_t sb_row = (nvalid ? n : 0) * args.ldsb;
            for (int p = 0; p < KP; ++p) {
                // this thread's group: k0 = 64 p + 32 half lies in one group (gs >= 32)
                const int64_t g = (static_cast<int64_t>(p) * QG_K + half * 32) / gs;
                uint32_t sv = 0, bv = 0;
                if (nvalid) {
                    sv = ld_u16_nc(scales + sb_row + g);
                    bv = ld_u16_nc(biases + sb_row + g);
                }
                const uint32_t s2 = sv | (sv << 16), b2 = bv | (bv << 16);
                if (!warp_wait(&raw_full[s], ph, abort_flag)) { ok = false; break; }
                // this row's packed words for k in [32 half, 32 half + 32)
                uint32_t wv[WPP / 2];
                const uint8_t *src = sW + s * WRAW + r * WROW + half * (WROW / 2);
                if constexpr (WPP / 2 == 1) {
                    wv[0] = *reinterpret_cast<const uint32_t *>(src);
                } else if constexpr (WPP / 2 == 2) {
                    const uint2 u = *reinterpret_cast<const uint2 *>(src);
                    wv[0] = u.x; wv[1] = u.y;
                } else {
#pragma unroll
                    for (int i = 0; i < WPP / 2; i += 4) {
                        const uint4 u = *reinterpret_cast<const uint4 *>(src + 4 * i);
                        wv[i] = u.x; wv[i + 1] = u.y; wv[i + 2] = u.z; wv[i + 3] = u.w;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&raw_empty[s]);
                if (!warp_wait(&a_empty[d], dph ^ 1u, abort_flag)) { ok = false; break; }
                uint8_t *dst = sA + d * QG_AP + r * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int chunk = half * 4 + c;                    // 8 weights each
                    uint4 v;
                    if constexpr (BITS == 4) v = deq8<T, 4>(&wv[c], 0, s2, b2);
                    else if constexpr (BITS == 8) v = deq8<T, 8>(&wv[2 * c], 0, s2, b2);
                    else v = deq8<T, 2>(&wv[c >> 1], c & 1, s2, b2);
                    *reinterpret_cast<uint4 *>(dst + ((chunk ^ (r & 7)) << 4)) = v;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[d]);
                if (++d == QG_DS) { d = 0; dph ^= 1u; }
                if (++s == RS) { s = 0; ph ^= 1u; }
            }
            if (!ok) break;
            // ---------------- epilogue of this tile: rows r, token columns 32 half..+31
            const uint32_t acc = tc & 1u;
            if (!warp_wait(&tfull[acc], (tc >> 1) & 1u, abort_flag)) break;
            tc_fence_after();
            uint32_t v[32];
            tmem_ld32(tmem_base + ((quarter * 32u) << 16) + acc * QG_T + half * 32, v);
            tmem_wait_ld(v);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            if (nvalid) {
                const float bn = args.bias ? to_f32<T>(static_cast<const T *>(args.bias)[n]) : 0.0f;
                T *ycol = static_cast<T *>(args.y) + n;
                const int64_t m0 = tb * QG_T + half * 32;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int64_t m = m0 + i;
                    if (m < M) {
                        float a = __uint_as_float(v[i]);
                        if (args.bias) a = __fadd_rn(a, bn);
                        ycol[m * args.ldy] = from_f32<T>(a);
                    }
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, QG_TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(args.err, ERR_TIMEOUT);
}

template <typename T, int BITS>
bi_status qgemm_attr() {
    return cuda_status(cudaFuncSetAttribute(qgemm_kernel<T, BITS>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(QgSmem<BITS>::BYTES)));
}

template <typename T, int BITS>
bi_status qgemm_launch(const CUtensorMap &tx, const CUtensorMap &tw, const QGemmArgs &args,
                       cudaStream_t s) {
    const int64_t tiles = ((args.N + QG_N - 1) / QG_N) * ((args.M + QG_T - 1) / QG_T);
    const int sms = device_sm_count();
    const int grid = static_cast<int>(tiles < sms ? tiles : sms);
    qgemm_kernel<T, BITS><<<grid, QG_THREADS, QgSmem<BITS>::BYTES, s>>>(tx, tw, args);
    count_launch();
    return cuda_status(cudaGetLastError());
}

template <typename T>
bi_status qgemm_bits(int bits, const CUtensorMap &tx, const CUtensorMap &tw,
                     const QGemmArgs &args, cudaStream_t s) {
    switch (bits) {
        case 2: return qgemm_launch<T, 2>(tx, tw, args, s);
        case 4: return qgemm_launch<T, 4>(tx, tw, args, s);
        case 8: return qgemm_launch<T, 8>(tx, tw, args, s);
        default: return BI_ERR_UNSUPPORTED;
    }
}

}  // namespace

bi_status init_qgemm() {
    bi_status (*const fns[])() = {qgemm_attr<__nv_bfloat16, 2>, qgemm_attr<__nv_bfloat16, 4>,
                                  qgemm_attr<__nv_bfloat16, 8>, qgemm_attr<__half, 2>,
                                  qgemm_attr<__half, 4>,        qgemm_attr<__half, 8>};
    for (auto f : fns) {
        const bi_status st = f();
        if (st != BI_OK) return st;
    }
    return BI_OK;
}

bi_status launch_qgemm(const void *x, int64_t ldx, const uint32_t *wq, int64_t ldq, int bits,
                       const QGemmArgs &args, bi_dtype dt, cudaStream_t s) {
    CUtensorMap tx, tw;
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(args.K), static_cast<uint64_t>(args.M)};
        const uint64_t strides[1] = {static_cast<uint64_t>(ldx) * 2};
        const uint32_t box[2] = {QG_K, static_cast<uint32_t>(args.x_rows)};
        bi_status st = encode_tmap(&tx, dt, 2, const_cast<void *>(x), dims, strides, box, true);
        if (st != BI_OK) return st;
    }
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(args.K * bits / 32),
                                  static_cast<uint64_t>(args.N)};
        const uint64_t strides[1] = {static_cast<uint64_t>(ldq) * 4};
        const uint32_t box[2] = {static_cast<uint32_t>(QG_K * bits / 32), QG_N};
        bi_status st = encode_tmap_u32(&tw, 2, const_cast<uint32_t *>(wq), dims, strides, box);
        if (st != BI_OK) return st;
    }
    if (dt == BI_BF16) return qgemm_bits<__nv_bfloat16>(bits, tx, tw, args, s);
    if (dt == BI_F16) return qgemm_bits<__half>(bits, tx, tw, args, s);
    return BI_ERR_UNSUPPORTED;
}

}  // namespace bi
