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
// Roles (608 threads, persistent over (n block, token block) tiles):
//   warp 0 lane 0   TMA producer of the packed weights: stages of 128 rows x 128
//                   bytes (16/bits panels; whole 128-byte lines of each row,
//                   128-byte swizzle so that the dequantisers read without bank
//                   conflicts), and of the scales and biases: chunks of 8 groups
//                   x 128 rows
//   warp 18 lane 0  TMA producer of the x panels (the rows that exist, packed, so
//                   a decode step keeps up to 32 panels in flight)
//   warp 1          TMEM allocation (two 64-column accumulators and a ring of 8
//                   weight panels); lane 0 issues the MMAs
//   warps 2..17     dequantisers: warp w owns weight rows 32*(w%4)..+31 (its TMEM
//                   lane quarter) and k [16 part, 16 part + 16) of each panel,
//                   part = (w-2)/4; they write the 16-bit weights straight into
//                   tensor memory, where the MMA takes them as its A operand (no
//                   shared-memory round trip for the largest operand).  After a
//                   tile's last panel they run its epilogue (the warp's TMEM lane
//                   quarter, token columns 16 part..+15).
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
constexpr int QG_DQ = 16;      // dequantising warps: 4 per TMEM lane quarter
constexpr int QG_THREADS = (QG_DQ + 3) * 32;   // + weight producer, MMA issuer, x producer
constexpr int QG_XWARP = QG_DQ + 2;            // the x producer's warp
constexpr int QG_WS = 6;       // packed weight stages in flight (16 KB each)
constexpr int QG_SS = 4;       // scale/bias chunks in flight (4 KB each)
constexpr int QG_XS_MAX = 32;  // x panels in flight: 64 KB / (x_rows * 128 bytes), at most 32
constexpr int QG_DS = 8;       // dequantised weight panels in flight (tensor memory)
constexpr uint32_t QG_WSTAGE = QG_N * 128;      // 16 KB: 128 rows x 128 packed bytes
constexpr uint32_t QG_SCHUNK = QG_N * 16;       // 2 KB: 128 rows x 8 groups x 2 bytes
constexpr uint32_t QG_XREGION = 64 * 1024;      // x ring
// Tensor memory: two 64-column fp32 accumulators, then DS dequantised weight
// panels of 32 columns (64 16-bit weights per row, two per column).
constexpr uint32_t QG_A_COL = 2 * QG_T;         // first column of the weight panels
constexpr uint32_t QG_TMEM_COLS = 512;          // 128 + 8 * 32 = 384 used

// Panels per packed stage: 128 bytes of a row hold 1024 / BITS weights.
template <int BITS> __host__ __device__ constexpr int qg_pps() { return 16 / BITS; }

struct QgSmem {
    // byte offsets from the 1024-aligned base
    static constexpr uint32_t W = 0;                                // [WS] packed stages
    static constexpr uint32_t X = W + QG_WS * QG_WSTAGE;            // x panels, packed
    static constexpr uint32_t SB = X + QG_XREGION;                  // [SS] scales, biases
    static constexpr uint32_t BARS = SB + QG_SS * 2 * QG_SCHUNK;
    // w_full[WS] w_empty[WS] s_full[SS] s_empty[SS] x_full[XS_MAX] x_empty[XS_MAX]
    // a_full[DS] a_empty[DS] tfull[2] tempty[2] mma_done (the x and a rings are
    // used per batch of panels: fewer slots than their arrays hold)
    static constexpr uint32_t NBARS =
        2 * QG_WS + 2 * QG_SS + 2 * QG_XS_MAX + 2 * QG_DS + 4 + 1;
    static constexpr uint32_t MISC = BARS + NBARS * 8;               // tmem slot, abort flag
    static constexpr uint32_t END = MISC + 16;
    static constexpr size_t BYTES = 1024 + END;
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Fields 2j and 2j+1 (bit offsets OA and OA + BITS) of w in the two 16-bit halves.
template <int BITS, int OA>
__device__ __forceinline__ uint32_t field_pair(uint32_t w) {
    constexpr uint32_t MASK = (1u << BITS) - 1u;
    constexpr int OB = OA + BITS;
    const uint32_t lo = w >> OA;
    const uint32_t hi = OB >= 16 ? (w >> (OB - 16)) : (w << (16 - OB));
    return prmt(lo, hi, 0x7610u) & (MASK | (MASK << 16));   // low half of lo, high half of hi
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

// The 16-bit pattern whose low byte holds a field and whose value is MAGIC + field,
// with a unit in the last place of 1: bf16 0x43xx = 128 + q (q < 128), fp16
// 0x64xx = 1024 + q (q < 256 with a byte field).
template <typename T> struct Magic;
template <> struct Magic<__nv_bfloat16> { static constexpr uint32_t byte = 0x43u; };
template <> struct Magic<__half> { static constexpr uint32_t byte = 0x64u; };

// q pair from a pair whose two halves are (MAGIC + q): one exact subtraction.
template <typename T> __device__ __forceinline__ uint32_t q_from_magic(uint32_t v) {
    using P = typename Pair<T>::t;
    constexpr uint32_t mm = (Magic<T>::byte << 24) | (Magic<T>::byte << 8);
    return as_u32(__hsub2(as_pair<P>(v), as_pair<P>(mm)));
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
    constexpr uint32_t KM = Magic<T>::byte * 0x01010101u;
    uint32_t q[4];
    if constexpr (BITS == 4) {
        // nibbles n0..n7 of the word -> bytes [n0 n1 n2 n3], [n4 n5 n6 n7] -> pairs
        // [n, MAGIC, n', MAGIC] (value MAGIC + n in each half)
        const uint32_t ev = w[0] & 0x0F0F0F0Fu;          // n0 n2 n4 n6
        const uint32_t od = (w[0] >> 4) & 0x0F0F0F0Fu;   // n1 n3 n5 n7
        const uint32_t lo = prmt(ev, od, 0x5140u);       // n0 n1 n2 n3
        const uint32_t hi = prmt(ev, od, 0x7362u);       // n4 n5 n6 n7
        q[0] = q_from_magic<T>(prmt(lo, KM, 0x5140u));
        q[1] = q_from_magic<T>(prmt(lo, KM, 0x7362u));
        q[2] = q_from_magic<T>(prmt(hi, KM, 0x5140u));
        q[3] = q_from_magic<T>(prmt(hi, KM, 0x7362u));
    } else if constexpr (BITS == 2) {
        const uint32_t v = sub ? (w[0] >> 16) : w[0];
        constexpr uint32_t MM = (Magic<T>::byte << 24) | (Magic<T>::byte << 8);
        q[0] = q_from_magic<T>(field_pair<2, 0>(v) | MM);
        q[1] = q_from_magic<T>(field_pair<2, 4>(v) | MM);
        q[2] = q_from_magic<T>(field_pair<2, 8>(v) | MM);
        q[3] = q_from_magic<T>(field_pair<2, 12>(v) | MM);
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
            // bytes straight into the halves next to the magic byte: 1024 + q
            q[0] = q_from_magic<T>(prmt(w[0], KM, 0x4140u));
            q[1] = q_from_magic<T>(prmt(w[0], KM, 0x4342u));
            q[2] = q_from_magic<T>(prmt(w[1], KM, 0x4140u));
            q[3] = q_from_magic<T>(prmt(w[1], KM, 0x4342u));
        }
    }
    return make_uint4(deq_pair<T>(q[0], s2, b2), deq_pair<T>(q[1], s2, b2),
                      deq_pair<T>(q[2], s2, b2), deq_pair<T>(q[3], s2, b2));
}

template <typename T, int BITS>
__global__ void __launch_bounds__(QG_THREADS, 1)
    qgemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmB,
                 const QGemmArgs args) {
    using S = QgSmem;
    constexpr int PPS = qg_pps<BITS>();                 // panels per packed stage
    constexpr int KPT = QG_K / (QG_DQ / 4);             // k of a panel row per thread (16)
    constexpr uint32_t QB = KPT * BITS / 8;             // their packed bytes
    constexpr int QB_B = PPS < 4 ? PPS : 4;             // panels per dequantising batch
    constexpr uint32_t IDESC = mma_idesc(IsBf16<T>::value, QG_N, QG_T, false);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sW = smem + S::W;
    uint8_t *sX = smem + S::X;
    uint8_t *sSB = smem + S::SB;     // chunk c: scales at c * 4 KB, biases 2 KB further
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::BARS);
    uint64_t *w_full = bars;
    uint64_t *w_empty = w_full + QG_WS;
    uint64_t *s_full = w_empty + QG_WS;
    uint64_t *s_empty = s_full + QG_SS;
    uint64_t *x_full = s_empty + QG_SS;
    uint64_t *x_empty = x_full + QG_XS_MAX;
    uint64_t *a_full = x_empty + QG_XS_MAX;
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
    const int KW = (KP + PPS - 1) / PPS;                // packed stages per tile
    const int gs = args.group_size;
    const int lg = gs == 32 ? 5 : gs == 64 ? 6 : 7;     // log2(group size)
    const int PPC = gs / 8;                             // panels per scale chunk (8 groups)
    const int NC = static_cast<int>((K / gs + 7) / 8);  // scale chunks per tile
    // x panels are packed at x_rows * 128 bytes (a multiple of 2 KB, so every panel
    // starts on the 1024-byte swizzle period).  The MMA reads 64 token rows; rows
    // past x_rows hold whatever follows and only feed output columns that are
    // never stored.
    const uint32_t XB = static_cast<uint32_t>(args.x_rows) * 128;
    // The x ring and the tensor-memory weight ring go by batches of QB_B panels (one
    // barrier, one copy and one commit per batch): XS batch slots of QB_B x panels,
    // DSB batch slots of QB_B weight panels.
    const uint32_t XBB = XB * QB_B;                     // bytes of a batch of x panels
    const int XS = static_cast<int>(QG_XREGION / XBB < QG_XS_MAX ? QG_XREGION / XBB : QG_XS_MAX);
    constexpr int DSB = QG_DS / QB_B;

    if (threadIdx.x == 0) {
        for (int i = 0; i < QG_WS; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&w_empty[i], QG_DQ);  // the dequantisers
        }
        for (int i = 0; i < QG_SS; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], QG_DQ);
        }
        for (int i = 0; i < QG_XS_MAX; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 1);      // the MMA's commit
        }
        for (int i = 0; i < QG_DS; ++i) {
            mbar_init(&a_full[i], QG_DQ);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], QG_DQ);
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
            // ------------------------------------------------ TMA producer: weights, scales
            prefetch_tmap(&tmW);
            prefetch_tmap(&tmS);
            prefetch_tmap(&tmB);
            uint32_t nw = 0, ns = 0, ws = 0, wph = 0, ss = 0, sph = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; ok && t < total; t += gridDim.x) {
                const int32_t wrow = static_cast<int32_t>((t % num_n) * QG_N);
                int c = 0;
                for (int st = 0; ok && st < KW; ++st) {
                    if (!mbar_wait(&w_empty[ws], wph ^ 1u, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&w_full[ws], QG_WSTAGE);
                    tma_load_2d(sW + ws * QG_WSTAGE, &tmW, &w_full[ws], st * 32, wrow);
                    ++nw;
                    if (++ws == QG_WS) { ws = 0; wph ^= 1u; }
                    // the scale chunks whose first panel lies in this stage
                    for (; c < NC && c * PPC < (st + 1) * PPS; ++c) {
                        if (!mbar_wait(&s_empty[ss], sph ^ 1u, abort_flag)) { ok = false; break; }
                        mbar_arrive_expect_tx(&s_full[ss], 2 * QG_SCHUNK);
                        uint8_t *dst = sSB + ss * 2 * QG_SCHUNK;
                        tma_load_2d(dst, &tmS, &s_full[ss], c * 8, wrow);
                        tma_load_2d(dst + QG_SCHUNK, &tmB, &s_full[ss], c * 8, wrow);
                        ++ns;
                        if (++ss == QG_SS) { ss = 0; sph ^= 1u; }
                    }
                }
            }
            if (!ok) {
                // Let every copy already issued land before the block can exit.
                for (uint32_t i = nw > QG_WS ? nw - QG_WS : 0; i < nw; ++i)
                    mbar_wait_limited(&w_full[i % QG_WS], (i / QG_WS) & 1u, WAIT_LIMIT_NS);
                for (uint32_t i = ns > QG_SS ? ns - QG_SS : 0; i < ns; ++i)
                    mbar_wait_limited(&s_full[i % QG_SS], (i / QG_SS) & 1u, WAIT_LIMIT_NS);
            }
        }
    } else if (warp == QG_XWARP) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer: x panels
            prefetch_tmap(&tmX);
            uint32_t nx = 0;
            int xs = 0;
            uint32_t xph = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; ok && t < total; t += gridDim.x) {
                const int32_t trow = static_cast<int32_t>((t / num_n) * QG_T);
                for (int p0 = 0; p0 < KP; p0 += QB_B) {
                    const int nb_ = KP - p0 < QB_B ? KP - p0 : QB_B;
                    if (!mbar_wait(&x_empty[xs], xph ^ 1u, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&x_full[xs], XB * nb_);
                    for (int b = 0; b < nb_; ++b)
                        tma_load_2d(sX + xs * XBB + b * XB, &tmX, &x_full[xs], (p0 + b) * QG_K, trow);
                    ++nx;
                    if (++xs == XS) { xs = 0; xph ^= 1u; }
                }
            }
            if (!ok) {
                for (uint32_t i = nx > static_cast<uint32_t>(XS) ? nx - XS : 0; i < nx; ++i)
                    mbar_wait_limited(&x_full[i % XS], (i / XS) & 1u, WAIT_LIMIT_NS);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            const uint64_t x_desc0 = smem_desc(smem_u32(sX), 16, 1024);
            const uint64_t xb16 = XB >> 4;          // one x panel in descriptor units
            uint32_t tc = 0, xph = 0, d = 0, dph = 0;
            int xs = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; ok && t < total; t += gridDim.x, ++tc) {
                const uint32_t acc = tc & 1u;
                if (!mbar_wait(&tempty[acc], ((tc >> 1) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * QG_T;
                // Batches of QB_B panels, as the dequantisers hand them over: every
                // warp arrives on a batch's panels in order, so the last panel's
                // barrier completing means the batch is in tensor memory.
                for (int p0 = 0; ok && p0 < KP; p0 += QB_B) {
                    const int nb_ = KP - p0 < QB_B ? KP - p0 : QB_B;
                    if (!mbar_wait(&a_full[d], dph, abort_flag)) { ok = false; break; }
                    if (!mbar_wait(&x_full[xs], xph, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_tmem = tmem_base + QG_A_COL + d * QB_B * (QG_K / 2);
                    const uint64_t xd = x_desc0 + ((xs * XBB) >> 4);
                    // panel b: A columns a_tmem + 32 b (8 per 16 k), x panel b of the batch.
                    // 4-bit: a whole batch goes out from one asm block with its operands
                    // computed first (measured 5-7% faster, e.g. 26.6 -> 25.3 us at M = 1,
                    // N = 14336; flat to 2% slower at 2 and 8 bits, which keep the
                    // per-panel form).  The same MMAs in the same order either way.
                    if (BITS == 4 && nb_ == QB_B && (QB_B == 4 || QB_B == 2)) {
                        uint32_t av[4 * QB_B];
                        uint64_t bv[4 * QB_B];
#pragma unroll
                        for (int b = 0; b < QB_B; ++b)
#pragma unroll
                            for (int s4 = 0; s4 < 4; ++s4) {
                                av[4 * b + s4] = a_tmem + b * (QG_K / 2) + 8 * s4;
                                bv[4 * b + s4] = xd + b * xb16 + 2 * s4;
                            }
                        if constexpr (QB_B == 4)
                            mma16_f16_ts(d_tmem, av, bv, IDESC, p0 != 0 ? 1u : 0u);
                        else if constexpr (QB_B == 2)
                            mma8_f16_ts(d_tmem, av, bv, IDESC, p0 != 0 ? 1u : 0u);
                    } else {
                        mma4_f16_ts(d_tmem, a_tmem, xd, IDESC, p0 != 0 ? 1u : 0u);
#pragma unroll
                        for (int b = 1; b < QB_B; ++b)
                            if (b < nb_)
                                mma4_f16_ts(d_tmem, a_tmem + b * (QG_K / 2), xd + b * xb16, IDESC, 1u);
                    }
                    mma_commit(&a_empty[d]);
                    mma_commit(&x_empty[xs]);
                    if (++d == DSB) { d = 0; dph ^= 1u; }
                    if (++xs == XS) { xs = 0; xph ^= 1u; }
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
            }
            // All issued MMAs must be complete before TMEM is released.
            mma_commit(mma_done);
            mbar_wait_limited(mma_done, 0, WAIT_LIMIT_NS);
        }
    } else if (warp >= 2 && warp < 2 + QG_DQ) {
        // ------------------------------------------------ dequantisers + epilogue
        const uint32_t quarter = static_cast<uint32_t>(warp & 3);
        const int part = (warp - 2) >> 2;                        // k [KPT part, +KPT) of a panel
        const int r = static_cast<int>(quarter) * 32 + lane;     // weight row in the tile
        uint32_t tc = 0, ws = 0, wph = 0, ss = 0, sph = 0, d = 0, dph = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; ok && t < total; t += gridDim.x, ++tc) {
            const int64_t nb = t % num_n, tb = t / num_n;
            const int64_t n = nb * QG_N + r;
            // Panels go in batches of QB_B: one wait per packed stage and per scale chunk
            // (a batch never straddles either: QB_B divides both), the batch's math is
            // independent work, and one TMEM store completion covers the batch.
            for (int p0 = 0; ok && p0 < KP; p0 += QB_B) {
                const int il0 = p0 % PPS;                   // first panel within its stage
                if (il0 == 0 && !warp_wait(&w_full[ws], wph, abort_flag)) { ok = false; break; }
                if ((p0 & (PPC - 1)) == 0 && !warp_wait(&s_full[ss], sph, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint8_t *wrow = sW + ws * QG_WSTAGE + r * 128;
                const uint8_t *sbrow = sSB + ss * 2 * QG_SCHUNK + r * 16;
                uint32_t out[QB_B][KPT / 2];
#pragma unroll
                for (int b = 0; b < QB_B; ++b) {
                    const int p = p0 + b;
                    if (p < KP) {
                        // this thread's group (k0 = 64 p + KPT part lies in one group)
                        const int j = ((p * QG_K + part * KPT) >> lg) & 7;
                        const uint32_t sv = *reinterpret_cast<const uint16_t *>(sbrow + j * 2);
                        const uint32_t bv =
                            *reinterpret_cast<const uint16_t *>(sbrow + QG_SCHUNK + j * 2);
                        const uint32_t s2 = sv | (sv << 16), b2 = bv | (bv << 16);
                        // packed bytes for k in [64 p + KPT part, +KPT): byte offset o of
                        // the stage row's 128, in 16-byte chunks with the 128-byte swizzle
                        uint32_t wv[QB / 4];
                        const uint32_t o = static_cast<uint32_t>((il0 + b) * 8 * BITS) + part * QB;
                        const uint8_t *src = wrow + (((o >> 4) ^ (r & 7)) << 4) + (o & 15);
                        if constexpr (QB == 16) {
                            const uint4 u = *reinterpret_cast<const uint4 *>(src);
                            wv[0] = u.x; wv[1] = u.y; wv[2] = u.z; wv[3] = u.w;
                        } else if constexpr (QB == 8) {
                            const uint2 u = *reinterpret_cast<const uint2 *>(src);
                            wv[0] = u.x; wv[1] = u.y;
                        } else {
                            wv[0] = *reinterpret_cast<const uint32_t *>(src);
                        }
#pragma unroll
                        for (int c = 0; c < KPT / 8; ++c) {
                            uint4 v;
                            if constexpr (BITS == 4) v = deq8<T, 4>(&wv[c], 0, s2, b2);
                            else if constexpr (BITS == 8) v = deq8<T, 8>(&wv[2 * c], 0, s2, b2);
                            else v = deq8<T, 2>(&wv[0], c, s2, b2);
                            out[b][4 * c] = v.x; out[b][4 * c + 1] = v.y;
                            out[b][4 * c + 2] = v.z; out[b][4 * c + 3] = v.w;
                        }
                    }
                }
                // release the scale chunk / packed stage when this batch ends it
                const int pl = (p0 + QB_B < KP ? p0 + QB_B : KP) - 1;   // last panel of the batch
                if ((pl & (PPC - 1)) == PPC - 1 || pl == KP - 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s_empty[ss]);
                    if (++ss == QG_SS) { ss = 0; sph ^= 1u; }
                }
                if (pl % PPS == PPS - 1 || pl == KP - 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&w_empty[ws]);
                    if (++ws == QG_WS) { ws = 0; wph ^= 1u; }
                }
                // KPT weights = KPT/2 columns of this row's TMEM lane in each panel of
                // batch slot d
                if (!warp_wait(&a_empty[d], dph ^ 1u, abort_flag)) { ok = false; break; }
                const uint32_t a_col = tmem_base + ((quarter * 32u) << 16) + QG_A_COL +
                                       d * QB_B * (QG_K / 2) + part * (KPT / 2);
#pragma unroll
                for (int b = 0; b < QB_B; ++b)
                    if (p0 + b < KP) tmem_st8(a_col + b * (QG_K / 2), out[b]);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[d]);
                if (++d == DSB) { d = 0; dph ^= 1u; }
            }
            if (!ok) break;
            // ---------------- epilogue of this tile: rows r, token columns 16 part..+15
            const uint32_t acc = tc & 1u;
            if (!warp_wait(&tfull[acc], (tc >> 1) & 1u, abort_flag)) break;
            tc_fence_after();
            uint32_t v[16];
            tmem_ld16(tmem_base + ((quarter * 32u) << 16) + acc * QG_T + part * 16, v);
            tmem_wait_ld16(v);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            if (n < N) {
                const float bn = args.bias ? to_f32<T>(static_cast<const T *>(args.bias)[n]) : 0.0f;
                T *ycol = static_cast<T *>(args.y) + n;
                const int64_t m0 = tb * QG_T + part * 16;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
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
                                            static_cast<int>(QgSmem::BYTES)));
}

template <typename T, int BITS>
bi_status qgemm_launch(const CUtensorMap &tx, const CUtensorMap &tw, const CUtensorMap &ts,
                       const CUtensorMap &tb, const QGemmArgs &args, cudaStream_t s) {
    const int64_t tiles = ((args.N + QG_N - 1) / QG_N) * ((args.M + QG_T - 1) / QG_T);
    const int sms = device_sm_count();
    const int grid = static_cast<int>(tiles < sms ? tiles : sms);
    qgemm_kernel<T, BITS><<<grid, QG_THREADS, QgSmem::BYTES, s>>>(tx, tw, ts, tb, args);
    count_launch();
    return cuda_status(cudaGetLastError());
}

template <typename T>
bi_status qgemm_bits(int bits, const CUtensorMap &tx, const CUtensorMap &tw,
                     const CUtensorMap &ts, const CUtensorMap &tb, const QGemmArgs &args,
                     cudaStream_t s) {
    switch (bits) {
        case 2: return qgemm_launch<T, 2>(tx, tw, ts, tb, args, s);
        case 4: return qgemm_launch<T, 4>(tx, tw, ts, tb, args, s);
        case 8: return qgemm_launch<T, 8>(tx, tw, ts, tb, args, s);
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
    CUtensorMap tx, tw, ts, tb;
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
        const uint32_t box[2] = {32, QG_N};     // 128 packed bytes of 128 rows, 128-byte swizzle
        bi_status st =
            encode_tmap_u32(&tw, 2, const_cast<uint32_t *>(wq), dims, strides, box, true);
        if (st != BI_OK) return st;
    }
    {
        // scales and biases: [N, K/group_size] at row stride ldsb; boxes of 8 groups
        const uint64_t dims[2] = {static_cast<uint64_t>(args.K / args.group_size),
                                  static_cast<uint64_t>(args.N)};
        const uint64_t strides[1] = {static_cast<uint64_t>(args.ldsb) * 2};
        const uint32_t box[2] = {8, QG_N};
        bi_status st = encode_tmap(&ts, dt, 2, const_cast<void *>(args.scales), dims, strides,
                                   box, false);
        if (st != BI_OK) return st;
        st = encode_tmap(&tb, dt, 2, const_cast<void *>(args.biases), dims, strides, box, false);
        if (st != BI_OK) return st;
    }
    if (dt == BI_BF16) return qgemm_bits<__nv_bfloat16>(bits, tx, tw, ts, tb, args, s);
    if (dt == BI_F16) return qgemm_bits<__half>(bits, tx, tw, ts, tb, args, s);
    return BI_ERR_UNSUPPORTED;
}

}  // namespace bi
