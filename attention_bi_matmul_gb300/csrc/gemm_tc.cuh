// gemm_tc.cuh -- batch-invariant 16-bit GEMM on the 5th-generation tensor cores.
//
// "mlx-batch-invariant" README, "How the kernels work" / GEMM: one block owns
// the whole K reduction of its output tile, the K loop's trip count depends
// on K alone, and a given row always lands at the same place in the same tile,
// so nothing about the summation order can move when M changes; no split-K,
// no atomics, fp32 accumulators, bias added into the accumulator and rounded
// once.  The GB300 form of that rule:
//
//   * output tile 128 x 128 on one CTA, or 256 x 256 on a CTA pair (the form
//     chosen from (dtype, N, K, layout) only), one tcgen05.mma accumulator in
//     tensor memory per tile;
//   * K visited in ascending 64-wide blocks, each as four K=16 MMAs in
//     ascending order, always starting from a zero accumulator -- for every M;
//   * operands staged by TMA into a multi-stage shared-memory ring with
//     128-byte swizzle (rows beyond M or K are zero-filled by the copy engine,
//     which adds exact zeros);
//   * epilogue: tcgen05.ld of the fp32 accumulator, + bias / alpha,beta*c in
//     fp32 in a fixed order, one rounding to the output dtype.
//
// Roles (192 threads, persistent over output tiles):
//   warp 0 lane 0  TMA producer (ring of STAGES stages; a stage holds KP
//                  consecutive 64-wide K panels of A and of B)
//   warp 1         TMEM allocation; lane 0 issues the MMAs (4 per panel)
//   warps 2..5     epilogue (warp w reads TMEM lanes 32*(w%4) .. +31)
// A stage of KP panels changes only how often the MMA thread waits and
// commits, not the order of the MMAs: every output still sees its K = 16
// steps in ascending order.
// Two accumulator buffers in TMEM let the epilogue of tile i overlap the
// mainloop of tile i+1.  The order in which tiles are visited never changes
// any bit of the result.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace bi {

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <> __device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ __half from_f32<__half>(float x) {
    return __float2half_rn(x);
}
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }

template <typename T> struct IsBf16 { static constexpr bool value = false; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr bool value = true; };

// Pack 8 consecutive fp32 values into 8 16-bit values (16 bytes).
template <typename T>
__device__ __forceinline__ uint4 pack8(const float *v) {
    union {
        T h[8];
        uint4 u;
    } p;
#pragma unroll
    for (int i = 0; i < 8; ++i) p.h[i] = from_f32<T>(v[i]);
    return p.u;
}

// Epilogue of 32 consecutive output columns [n0, n0+32) of row m of batch entry e.
template <typename T>
__device__ __forceinline__ void gemm_epilogue32(const uint32_t (&r)[32], int64_t e, int64_t m,
                                                int64_t n0, const GemmArgs &a) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
    const int64_t N = a.N;
    if (a.epi == EPI_BIAS) {
        const T *bias = static_cast<const T *>(a.bias);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (n0 + i < N) v[i] = __fadd_rn(v[i], to_f32<T>(bias[n0 + i]));
    } else if (a.epi == EPI_ADDMM) {
        const T *crow = static_cast<const T *>(a.c) + (a.ldc ? m * a.ldc : 0);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (n0 + i < N)
                v[i] = __fadd_rn(__fmul_rn(a.alpha, v[i]), __fmul_rn(a.beta, to_f32<T>(crow[n0 + i])));
    }
    T *yrow = static_cast<T *>(a.y) + e * a.sy + m * a.ldy;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int64_t n = n0 + 8 * g;
        if (n + 8 <= N) {
            *reinterpret_cast<uint4 *>(yrow + n) = pack8<T>(v + 8 * g);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (n + i < N) yrow[n + i] = from_f32<T>(v[8 * g + i]);
        }
    }
}

constexpr int TC_BM = 128;
constexpr int TC_BK = 64;
constexpr int TC_THREADS = 192;
constexpr int TC_GROUP_M = 16;   // one-CTA tiles: groups of 16 row blocks of 128
// CTA-pair tiles: groups of 8 row blocks of 256.  Measured at 8192^3 (DRAM bytes
// per launch, time): 4 -> 1.53 GB, 0.624 ms; 8 -> 1.17 GB, 0.607 ms; 16 -> 1.39 GB,
// 0.609 ms; 32 -> 2.18 GB, 0.638 ms (algorithmic 0.40 GB).
constexpr int TC2_GROUP_M = 8;

__host__ __device__ constexpr uint32_t tc_tmem_cols(int bn) {
    // two accumulator buffers of bn fp32 columns, rounded up to a power of two >= 32
    return (2 * bn <= 32) ? 32u : (2 * bn <= 64) ? 64u : (2 * bn <= 128) ? 128u
           : (2 * bn <= 256) ? 256u : 512u;
}

// Pipeline shape of the one-CTA kernel, 192 KB of shared memory (with 128-row A
// panels; fewer A rows leave room for more stages, see the kernel): stages of 2
// K panels (8 MMAs of 64 cycles per barrier round trip), 3 stages at 128
// columns; stages of 1 K panel (4 MMAs of 128 cycles), 4 stages, at 256.  The
// library builds the 128-column form; 256-column tiles run on a CTA pair below.
template <int BN> __host__ __device__ constexpr int tc_kp() { return BN <= 128 ? 2 : 1; }
template <int BN> __host__ __device__ constexpr int tc_stages() { return BN <= 128 ? 3 : 4; }
template <int BN> __host__ __device__ constexpr bool tc_l2_prefetch() { return BN <= 128; }

// Ring bytes: tc_stages stages of full 128-row A panels.  With fewer A rows a
// stage is smaller and the same bytes hold more stages (up to TC_MAX_STAGES).
constexpr int TC_MAX_STAGES = 16;
template <int BN>
__host__ __device__ constexpr uint32_t tc_ring_bytes() {
    return (uint32_t)tc_stages<BN>() * tc_kp<BN>() * (TC_BM * TC_BK * 2 + BN * TC_BK * 2);
}
template <int BN>
__host__ __device__ constexpr size_t tc_smem_bytes() {
    return 1024 /* alignment slack */ + tc_ring_bytes<BN>() +
           (2 * TC_MAX_STAGES + 5) * 8 + 16 /* barriers, TMEM slot, abort flag */;
}

// Tile t -> (batch entry, m block, n block); within an entry, tiles are grouped GM
// row blocks at a time so that concurrently running tiles share A and B in L2.
template <int GM = TC_GROUP_M>
__device__ __forceinline__ void tc_tile_coords(int64_t t, int64_t num_m, int64_t num_n,
                                               int64_t &e, int64_t &mb, int64_t &nb) {
    const int64_t per_entry = num_m * num_n;
    e = t / per_entry;
    t -= e * per_entry;
    const int64_t in_group = (int64_t)GM * num_n;
    const int64_t g = t / in_group;
    const int64_t first_m = g * GM;
    const int64_t gm = (num_m - first_m) < GM ? (num_m - first_m) : GM;
    const int64_t r = t - g * in_group;
    mb = first_m + r % gm;
    nb = r / gm;
}

template <typename T, int BN, bool B_MN>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmArgs args) {
    constexpr int KP = tc_kp<BN>();
    constexpr uint32_t B_PANEL = BN * TC_BK * 2;
    constexpr uint32_t B_BYTES = KP * B_PANEL;        // per stage
    constexpr uint32_t TMEM_COLS = tc_tmem_cols(BN);
    constexpr uint32_t IDESC = mma_idesc(IsBf16<T>::value, TC_BM, BN, B_MN);
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "tile width");
    constexpr int EB = BN / 32 < 4 ? BN / 32 : 4;       // epilogue loads per wait
    static_assert(!B_MN || BN % 64 == 0, "MN-major B needs 64-column atoms");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    // Ring layout for this call: A panels hold the a_rows rows the copy moves (a
    // multiple of 16 rows, so every panel starts on the 1024-byte swizzle period),
    // then the B panels.  The MMA always reads 128 A rows; rows past a_rows hold
    // whatever follows (the next panel, or the first B panels) and only feed tile
    // rows that are never stored.  Fewer A rows -> more stages in the same bytes;
    // the ring depth changes only the scheduling, never the order of any MMA.
    const uint32_t A_PANEL = static_cast<uint32_t>(args.a_rows) * TC_BK * 2;
    const uint32_t A_BYTES = KP * A_PANEL;            // per stage
    const uint32_t ST_FIT = tc_ring_bytes<BN>() / (A_BYTES + B_BYTES);
    const int STAGES = static_cast<int>(ST_FIT < TC_MAX_STAGES ? ST_FIT : TC_MAX_STAGES);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + tc_ring_bytes<BN>());
    uint64_t *empty = full + TC_MAX_STAGES;
    uint64_t *tfull = empty + TC_MAX_STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int64_t M = args.M, N = args.N, K = args.K;
    const int64_t num_m = (M + TC_BM - 1) / TC_BM;
    const int64_t num_n = (N + BN - 1) / BN;
    const int64_t total = args.batch * num_m * num_n;
    const int KB = static_cast<int>((K + KP * TC_BK - 1) / (KP * TC_BK));   // stages per tile

    // The producer's copies.  The A copy moves only the rows that exist (a_rows <= 128);
    // tile rows past them are never stored, and no row's result depends on another row.
    const uint32_t tx = KP * (static_cast<uint32_t>(args.a_rows) * TC_BK * 2 + B_PANEL);
    // ring stage s <- K panels kb * KP.. of tile (mb, nb) of batch entries (ea, eb)
    auto copy_stage = [&](uint32_t s, int kb, int64_t mb, int64_t nb, int32_t ea, int32_t eb) {
        mbar_arrive_expect_tx(&full[s], tx);
#pragma unroll
        for (int p = 0; p < KP; ++p) {
            const int32_t k0 = (kb * KP + p) * TC_BK;   // beyond K: zero-filled
            tma_load_3d(sA + s * A_BYTES + p * A_PANEL, &tmA, &full[s], k0,
                        static_cast<int32_t>(mb * TC_BM), ea);
            if (!B_MN) {
                tma_load_3d(sB + s * B_BYTES + p * B_PANEL, &tmB, &full[s], k0,
                            static_cast<int32_t>(nb * BN), eb);
            } else {
#pragma unroll
                for (int j = 0; j < BN / 64; ++j)
                    tma_load_3d(sB + s * B_BYTES + p * B_PANEL + j * 8192, &tmB, &full[s],
                                static_cast<int32_t>(nb * BN + j * 64), k0, eb);
            }
        }
    };
    // 128-column tiles stream their weight panels from HBM; the producer asks for the
    // panels one ring further on to move into L2 as it copies a stage.  (Measured: +2-5%
    // for those; it costs the L2-resident 256-wide tiles 7%, so they do not.
    // Prefetching further ahead was slower.)
    auto prefetch_stage = [&](int kq_stage, int64_t nb, int32_t eb) {
#pragma unroll
        for (int p = 0; p < KP; ++p) {
            const int32_t kq = (kq_stage * KP + p) * TC_BK;
            if (!B_MN) {
                tma_prefetch_3d(&tmB, kq, static_cast<int32_t>(nb * BN), eb);
            } else {
#pragma unroll
                for (int j = 0; j < BN / 64; ++j)
                    tma_prefetch_3d(&tmB, static_cast<int32_t>(nb * BN + j * 64), kq, eb);
            }
        }
    };

    if (threadIdx.x == 0) {
        // Thread 0 is also the copy producer: it fetches the copy descriptors and sends
        // the block's first stage before the TMEM allocation and the block barrier, so
        // that the copy's latency overlaps the setup (the grid never exceeds the tiles).
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
        int64_t e, mb, nb;
        tc_tile_coords(blockIdx.x, num_m, num_n, e, mb, nb);
        const int32_t eb = args.sb ? static_cast<int32_t>(e) : 0;
        copy_stage(0, 0, mb, nb, args.sa ? static_cast<int32_t>(e) : 0, eb);
        if (tc_l2_prefetch<BN>() && STAGES < KB) prefetch_stage(STAGES, nb, eb);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            // Stage 0 of the first tile went out during the setup.
            uint32_t it = 1, s = 1, ph = 0;
            if (s == static_cast<uint32_t>(STAGES)) { s = 0; ph = 1u; }
            bool ok = true;
            for (int64_t t = blockIdx.x; ok && t < total; t += gridDim.x) {
                int64_t e, mb, nb;
                tc_tile_coords(t, num_m, num_n, e, mb, nb);
                // A shared operand is a tensor map with one batch entry.
                const int32_t ea = args.sa ? static_cast<int32_t>(e) : 0;
                const int32_t eb = args.sb ? static_cast<int32_t>(e) : 0;
                for (int kb = t == blockIdx.x ? 1 : 0; kb < KB; ++kb, ++it) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
                    copy_stage(s, kb, mb, nb, ea, eb);
                    if (tc_l2_prefetch<BN>() && kb + STAGES < KB) prefetch_stage(kb + STAGES, nb, eb);
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // Let every copy already issued land before the block can exit.
                const uint32_t first = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0;
                for (uint32_t i = first; i < it; ++i)
                    mbar_wait_limited(&full[i % STAGES], (i / STAGES) & 1u, WAIT_LIMIT_NS);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            // Descriptors of stage 0; stage s adds s * (stage bytes >> 4) to the start
            // address field, and K step j adds j * 32 bytes (K-major) or j * 2048
            // bytes (MN-major B) the same way.
            const uint64_t a_desc0 = smem_desc(smem_u32(sA), 16, 1024);
            const uint64_t b_desc0 = B_MN ? smem_desc(smem_u32(sB), 8192, 1024)
                                          : smem_desc(smem_u32(sB), 16, 1024);
            const uint64_t A_STEP = A_BYTES >> 4, AP_STEP = A_PANEL >> 4;
            constexpr uint64_t B_STEP = B_BYTES >> 4, BP_STEP = B_PANEL >> 4;
            constexpr uint64_t BK_STEP = B_MN ? (2048 >> 4) : (32 >> 4);
            uint32_t tc = 0, s = 0, ph = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; ok && t < total; t += gridDim.x, ++tc) {
                const uint32_t acc = tc & 1u;
                const uint32_t aph = (tc >> 1) & 1u;
                if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[s], ph, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = a_desc0 + s * A_STEP;
                    const uint64_t bd = b_desc0 + s * B_STEP;
#pragma unroll
                    for (int p = 0; p < KP; ++p)
#pragma unroll
                        for (int j = 0; j < TC_BK / 16; ++j)
                            mma_f16_ss(d_tmem, ad + p * AP_STEP + j * (32 >> 4),
                                       bd + p * BP_STEP + j * BK_STEP, IDESC,
                                       (kb | p | j) != 0 ? 1u : 0u);
                    mma_commit(&empty[s]);
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
            }
            // All issued MMAs must be complete before TMEM is released.
            mma_commit(mma_done);
            mbar_wait_limited(mma_done, 0, WAIT_LIMIT_NS);
        }
    } else if (warp >= 2 && warp <= 5) {
        // ------------------------------------------------ epilogue (warps 2..5)
        const uint32_t quarter = static_cast<uint32_t>(warp & 3);
        const int row_in_tile = static_cast<int>(quarter) * 32 + lane;
        uint32_t tc = 0;
        for (int64_t t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            int64_t e, mb, nb;
            tc_tile_coords(t, num_m, num_n, e, mb, nb);
            const uint32_t acc = tc & 1u;
            const uint32_t aph = (tc >> 1) & 1u;
            if (!warp_wait(&tfull[acc], aph, abort_flag)) break;
            tc_fence_after();
            const int64_t m = mb * TC_BM + row_in_tile;
            // EB 32-column loads in flight per wait (the wait's latency, not the
            // bandwidth, bounds a tile's epilogue)
#pragma unroll 1
            for (int c0 = 0; c0 < BN / 32; c0 += EB) {
                uint32_t r[EB][32];
#pragma unroll
                for (int u = 0; u < EB; ++u)
                    tmem_ld32(tmem_base + ((quarter * 32u) << 16) + acc * BN + (c0 + u) * 32, r[u]);
                tmem_wait_ld(r[0]);
#pragma unroll
                for (int u = 1; u < EB; ++u) tmem_tie(r[u]);
                if (m < M) {
#pragma unroll
                    for (int u = 0; u < EB; ++u)
                        gemm_epilogue32<T>(r[u], e, m, nb * BN + (c0 + u) * 32, args);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(args.err, ERR_TIMEOUT);
}

// ------------------------------------------------------------------ CTA-pair form
//
// The same rule on a pair of SMs (a cluster of two CTAs, cta_group::2): the
// output tile is 256 x BN, one accumulator split over the pair's tensor
// memories (rows 0-127 in the even CTA, 128-255 in the odd one).  Each CTA
// stages its own 128 A rows and one half (BN/2 rows) of the B tile; the even
// CTA's MMA thread issues the 256 x BN x 16 MMAs, which read both CTAs' shared
// memory.  Per SM that is a 128 x BN output from 128 x 64 A plus BN/2 x 64 B
// bytes per K panel -- a third fewer bytes into each SM than the one-CTA tile of
// the same width, which is what bounds the one-CTA kernel on large GEMMs.
// K is still visited in ascending 64-wide panels of four K = 16 steps from a zero
// accumulator, and the tile of a row depends on nothing but the row.
//
// Barriers: full[s] lives in the even CTA and collects both CTAs' copy bytes;
// empty[s] and tfull[b] exist in both CTAs and are signalled together by a
// multicast commit; tempty[b] lives in the even CTA and counts the epilogue
// warps of both.
constexpr int TC2_BM = 256;         // rows per pair tile (128 per CTA)
constexpr int TC2_RING_PANELS = 6;  // ring size in panels of 128-row A and BN/2-row B

template <int BN>
__host__ __device__ constexpr uint32_t tc2_ring_bytes() {
    return (uint32_t)TC2_RING_PANELS * (TC_BM * TC_BK * 2 + (BN / 2) * TC_BK * 2);
}
template <int BN>
__host__ __device__ constexpr size_t tc2_smem_bytes() {
    return 1024 + tc2_ring_bytes<BN>() + (2 * TC_MAX_STAGES + 5) * 8 + 16;
}

// KPP: 64-wide K panels per ring stage (scheduling only: every output sees the
// same K = 16 steps in the same order).  Two panels halve the MMA thread's
// barrier waits per MMA (each wait leaves the tensor pipe idle for a few hundred
// cycles); one keeps twice as many stages in flight.
template <typename T, int BN, bool B_MN, int KPP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(TC_THREADS, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const GemmArgs args) {
    constexpr int BH = BN / 2;                               // B rows per CTA
    constexpr uint32_t B_PANEL = BH * TC_BK * 2;
    constexpr uint32_t B_BYTES = KPP * B_PANEL;              // per stage
    constexpr uint32_t TMEM_COLS = tc_tmem_cols(BN);
    constexpr uint32_t IDESC = mma_idesc(IsBf16<T>::value, TC2_BM, BN, B_MN);
    static_assert(BN == 128 || BN == 256, "pair tile width");
    constexpr int EB = 2;                                // epilogue loads per wait

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    // A stages first (a_rows rows each), then the B stages; the MMA reads 128 A
    // rows, and rows past a_rows only feed tile rows that are never stored.  Both
    // CTAs lay the ring out identically, so one descriptor addresses both.
    const uint32_t A_PANEL = static_cast<uint32_t>(args.a_rows) * TC_BK * 2;
    const uint32_t A_BYTES = KPP * A_PANEL;
    const uint32_t ST_FIT = tc2_ring_bytes<BN>() / (A_BYTES + B_BYTES);
    const int STAGES = static_cast<int>(ST_FIT < TC_MAX_STAGES ? ST_FIT : TC_MAX_STAGES);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + tc2_ring_bytes<BN>());
    uint64_t *empty = full + TC_MAX_STAGES;
    uint64_t *tfull = empty + TC_MAX_STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    const int64_t M = args.M, N = args.N, K = args.K;
    const int64_t num_m = (M + TC2_BM - 1) / TC2_BM;
    const int64_t num_n = (N + BN - 1) / BN;
    const int64_t total = args.batch * num_m * num_n;
    const int KB = static_cast<int>((K + KPP * TC_BK - 1) / (KPP * TC_BK));   // stages per tile
    const int64_t pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        // fetch the copy descriptors while the block sets up (the first copy waits for them)
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
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
        tmem_alloc_pair(tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncwarp();
    cluster_sync();     // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            const uint32_t tx = 2u * (A_BYTES + B_BYTES);       // both CTAs' bytes
            uint32_t it = 0, s = 0, ph = 0;
            bool ok = true;
            for (int64_t t = pair; ok && t < total; t += num_pairs) {
                int64_t e, mb, nb;
                tc_tile_coords<TC2_GROUP_M>(t, num_m, num_n, e, mb, nb);
                const int32_t ea = args.sa ? static_cast<int32_t>(e) : 0;
                const int32_t eb = args.sb ? static_cast<int32_t>(e) : 0;
                const int32_t row0 = static_cast<int32_t>(mb * TC2_BM + rank * TC_BM);
                const int32_t col0 = static_cast<int32_t>(nb * BN + rank * BH);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
                    const uint32_t fb = cluster_addr(&full[s], 0);
                    if (leader) mbar_arrive_expect_tx(&full[s], tx);
#pragma unroll
                    for (int p = 0; p < KPP; ++p) {
                        const int32_t k0 = (kb * KPP + p) * TC_BK;   // beyond K: zero-filled
                        tma_load_3d_pair(sA + s * A_BYTES + p * A_PANEL, &tmA, fb, k0, row0, ea);
                        if (!B_MN) {
                            tma_load_3d_pair(sB + s * B_BYTES + p * B_PANEL, &tmB, fb, k0, col0, eb);
                        } else {
#pragma unroll
                            for (int j = 0; j < BH / 64; ++j)
                                tma_load_3d_pair(sB + s * B_BYTES + p * B_PANEL + j * 8192, &tmB, fb,
                                                 col0 + j * 64, k0, eb);
                        }
                    }
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // Let the copies already issued land before the pair can exit.  The
                // even CTA's barriers see both CTAs' bytes; the odd CTA cannot wait on
                // them, so it gives its own copies a fixed time instead.
                if (leader) {
                    const uint32_t first = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0;
                    for (uint32_t i = first; i < it; ++i)
                        mbar_wait_limited(&full[i % STAGES], (i / STAGES) & 1u, WAIT_LIMIT_NS);
                } else {
                    const uint64_t t0 = globaltimer_ns();
                    for (uint32_t i = 0; i < WAIT_MAX_ROUNDS && globaltimer_ns() - t0 < 1000000ull; ++i)
                        __nanosleep(1000);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer (even CTA)
            const uint64_t a_desc0 = smem_desc(smem_u32(sA), 16, 1024);
            const uint64_t b_desc0 = B_MN ? smem_desc(smem_u32(sB), 8192, 1024)
                                          : smem_desc(smem_u32(sB), 16, 1024);
            const uint64_t A_STEP = A_BYTES >> 4, AP_STEP = A_PANEL >> 4;
            constexpr uint64_t B_STEP = B_BYTES >> 4, BP_STEP = B_PANEL >> 4;
            constexpr uint64_t BK_STEP = B_MN ? (2048 >> 4) : (32 >> 4);
            const int panels = static_cast<int>((K + TC_BK - 1) / TC_BK);
            uint32_t tc = 0, s = 0, ph = 0;
            bool ok = true;
            for (int64_t t = pair; ok && t < total; t += num_pairs, ++tc) {
                const uint32_t acc = tc & 1u;
                const uint32_t aph = (tc >> 1) & 1u;
                if (!mbar_wait_cluster(&tempty[acc], aph ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[s], ph, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = a_desc0 + s * A_STEP;
                    const uint64_t bd = b_desc0 + s * B_STEP;
                    // A panel wholly past K is not multiplied, so the MMA sequence of
                    // a tile is the same with one or two panels per stage (the stage
                    // shape depends on the number of tiles, hence on M).
                    const int live = panels - kb * KPP;
#pragma unroll
                    for (int p = 0; p < KPP; ++p) {
                        if (p == 0 || p < live) {
#pragma unroll
                            for (int j = 0; j < TC_BK / 16; ++j)
                                mma_f16_ss_pair(d_tmem, ad + p * AP_STEP + j * (32 >> 4),
                                                bd + p * BP_STEP + j * BK_STEP, IDESC,
                                                (kb | p | j) != 0 ? 1u : 0u);
                        }
                    }
                    mma_commit_pair_mc(&empty[s], 0x3);
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                mma_commit_pair_mc(&tfull[acc], 0x3);
            }
            // All issued MMAs must be complete before either CTA releases TMEM or
            // shared memory.
            mma_commit_pair(mma_done);
            mbar_wait_limited(mma_done, 0, WAIT_LIMIT_NS);
        }
    } else if (warp >= 2 && warp <= 5) {
        // ------------------------------------------------ epilogue (both CTAs)
        const uint32_t quarter = static_cast<uint32_t>(warp & 3);
        const int row_in_tile = static_cast<int>(rank) * TC_BM + static_cast<int>(quarter) * 32 + lane;
        uint32_t tc = 0;
        for (int64_t t = pair; t < total; t += num_pairs, ++tc) {
            int64_t e, mb, nb;
            tc_tile_coords<TC2_GROUP_M>(t, num_m, num_n, e, mb, nb);
            const uint32_t acc = tc & 1u;
            const uint32_t aph = (tc >> 1) & 1u;
            if (!warp_wait(&tfull[acc], aph, abort_flag)) break;
            tc_fence_after();
            const int64_t m = mb * TC2_BM + row_in_tile;
            // EB 32-column loads in flight per wait (the wait's latency, not the
            // bandwidth, bounds a tile's epilogue)
#pragma unroll 1
            for (int c0 = 0; c0 < BN / 32; c0 += EB) {
                uint32_t r[EB][32];
#pragma unroll
                for (int u = 0; u < EB; ++u)
                    tmem_ld32(tmem_base + ((quarter * 32u) << 16) + acc * BN + (c0 + u) * 32, r[u]);
                tmem_wait_ld(r[0]);
#pragma unroll
                for (int u = 1; u < EB; ++u) tmem_tie(r[u]);
                if (m < M) {
#pragma unroll
                    for (int u = 0; u < EB; ++u)
                        gemm_epilogue32<T>(r[u], e, m, nb * BN + (c0 + u) * 32, args);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(cluster_addr(&tempty[acc], 0));
        }
    }

    tc_fence_before();
    __syncwarp();
    cluster_sync();     // no MMA, copy or arrival is still headed for either CTA
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(args.err, ERR_TIMEOUT);
}

// Host side: instantiate and launch one configuration.
// Shared-memory attribute of one instantiation (per device; done at library init).
template <typename T, int BN, bool B_MN>
bi_status init_tc_inst() {
    return cuda_status(cudaFuncSetAttribute(gemm_tc_kernel<T, BN, B_MN>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(tc_smem_bytes<BN>())));
}

// Pair kernel: the shared-memory attribute and how many pairs fit on the device
// at once (the persistent grid must never exceed it: a pair that is not resident
// would only start once another has finished all its tiles).
constexpr int TC2_MAX_DEVICES = 64;
template <typename T, int BN, bool B_MN, int KPP>
int &tc2_max_pairs(int dev) {
    static int v[TC2_MAX_DEVICES] = {};
    return v[dev];
}

template <typename T, int BN, bool B_MN, int KPP>
bi_status init_tc2_inst() {
    constexpr size_t SMEM = tc2_smem_bytes<BN>();
    bi_status st = cuda_status(cudaFuncSetAttribute(gemm_tc2_kernel<T, BN, B_MN, KPP>,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    static_cast<int>(SMEM)));
    if (st != BI_OK) return st;
    int dev = 0;
    if ((st = cuda_status(cudaGetDevice(&dev))) != BI_OK) return st;
    if (dev < 0 || dev >= TC2_MAX_DEVICES) return BI_ERR_UNSUPPORTED;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(2 * static_cast<unsigned>(device_sm_count()));
    lc.blockDim = dim3(TC_THREADS);
    lc.dynamicSmemBytes = SMEM;
    int clusters = 0;
    if ((st = cuda_status(cudaOccupancyMaxActiveClusters(
             &clusters, gemm_tc2_kernel<T, BN, B_MN, KPP>, &lc))) != BI_OK)
        return st;
    if (clusters <= 0) return BI_ERR_UNSUPPORTED;
    tc2_max_pairs<T, BN, B_MN, KPP>(dev) = clusters;
    return BI_OK;
}

template <typename T>
bi_status init_tc_all() {
    bi_status st;
    if ((st = init_tc_inst<T, 128, false>()) != BI_OK) return st;
    if ((st = init_tc_inst<T, 128, true>()) != BI_OK) return st;
    if ((st = init_tc2_inst<T, 256, false, 1>()) != BI_OK) return st;
    if ((st = init_tc2_inst<T, 256, false, 2>()) != BI_OK) return st;
    if ((st = init_tc2_inst<T, 256, true, 1>()) != BI_OK) return st;
    return init_tc2_inst<T, 256, true, 2>();
}

template <typename T, int BN, bool B_MN>
bi_status launch_tc_inst(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &args,
                         int stages_req, cudaStream_t s) {
    (void)stages_req;
    constexpr size_t SMEM = tc_smem_bytes<BN>();
    const int64_t tiles =
        args.batch * ((args.M + TC_BM - 1) / TC_BM) * ((args.N + BN - 1) / BN);
    const int sms = device_sm_count();
    const int grid = static_cast<int>(tiles < sms ? tiles : sms);
    gemm_tc_kernel<T, BN, B_MN><<<grid, TC_THREADS, SMEM, s>>>(ta, tb, args);
    count_launch();
    return cuda_status(cudaGetLastError());
}

template <typename T, int BN, bool B_MN>
bi_status launch_tc2_inst(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &args,
                          cudaStream_t s) {
    constexpr size_t SMEM = tc2_smem_bytes<BN>();
    const int64_t tiles =
        args.batch * ((args.M + TC2_BM - 1) / TC2_BM) * ((args.N + BN - 1) / BN);
    int dev = 0;
    bi_status st = cuda_status(cudaGetDevice(&dev));
    if (st != BI_OK) return st;
    if (dev < 0 || dev >= TC2_MAX_DEVICES) return BI_ERR_UNSUPPORTED;
    const int max_pairs = tc2_max_pairs<T, BN, B_MN, 1>(dev);
    if (max_pairs <= 0 || tc2_max_pairs<T, BN, B_MN, 2>(dev) != max_pairs)
        return BI_ERR_CUDA;    // not initialised on this device
    const int pairs = static_cast<int>(tiles < max_pairs ? tiles : max_pairs);
    // Stage shape (scheduling only, the bits are the same): two K panels per stage
    // when every pair has at least two tiles to run (measured on GB300: 8192^3
    // 1.86 against 1.81 PFLOP/s), one when the pairs are not all busy for long
    // (M = 512, N = 14336, K = 8192: 85 against 88-92 us).
    if (tiles >= 2 * static_cast<int64_t>(max_pairs))
        gemm_tc2_kernel<T, BN, B_MN, 2><<<2 * pairs, TC_THREADS, SMEM, s>>>(ta, tb, args);
    else
        gemm_tc2_kernel<T, BN, B_MN, 1><<<2 * pairs, TC_THREADS, SMEM, s>>>(ta, tb, args);
    count_launch();
    return cuda_status(cudaGetLastError());
}

// Dispatch on the configured tile width; builds the tensor maps.
template <typename T>
bi_status launch_gemm_tc_typed(const void *a, int64_t lda, const void *b, int64_t ldb, bool b_nk,
                               const GemmArgs &args, bi_dtype dt, const TcConfig &cfg,
                               cudaStream_t s) {
    const int BN = cfg.block_n;
    CUtensorMap ta, tb;
    // Third dimension: the batch entry.  A shared operand (batch stride 0) gets one
    // entry, with the packed stride standing in for the unused one.
    {
        const uint64_t ea = args.sa ? static_cast<uint64_t>(args.batch) : 1;
        const uint64_t dims[3] = {static_cast<uint64_t>(args.K), static_cast<uint64_t>(args.M), ea};
        const uint64_t strides[2] = {static_cast<uint64_t>(lda) * 2,
                                     static_cast<uint64_t>(args.sa ? args.sa : lda * args.M) * 2};
        const uint32_t box[3] = {TC_BK, static_cast<uint32_t>(args.a_rows), 1};
        bi_status st = encode_tmap(&ta, dt, 3, const_cast<void *>(a), dims, strides, box, true);
        if (st != BI_OK) return st;
    }
    {
        const uint64_t eb = args.sb ? static_cast<uint64_t>(args.batch) : 1;
        const uint64_t inner = b_nk ? args.K : args.N, outer = b_nk ? args.N : args.K;
        const uint64_t dims[3] = {inner, outer, eb};
        const uint64_t strides[2] = {static_cast<uint64_t>(ldb) * 2,
                                     static_cast<uint64_t>(args.sb ? args.sb : ldb * outer) * 2};
        // K-major B: one box of the tile's rows (half of them per CTA in the pair
        // form); MN-major B: 64-column boxes.
        const uint32_t b_rows = static_cast<uint32_t>(cfg.pair ? BN / 2 : BN);
        const uint32_t box[3] = {b_nk ? static_cast<uint32_t>(TC_BK) : 64u,
                                 b_nk ? b_rows : static_cast<uint32_t>(TC_BK), 1};
        bi_status st = encode_tmap(&tb, dt, 3, const_cast<void *>(b), dims, strides, box, true);
        if (st != BI_OK) return st;
    }
    // Built forms: 128-column tiles on one CTA, 256-column tiles on a CTA pair.
    if (cfg.pair && BN == 256)
        return b_nk ? launch_tc2_inst<T, 256, false>(ta, tb, args, s)
                    : launch_tc2_inst<T, 256, true>(ta, tb, args, s);
    if (!cfg.pair && BN == 128)
        return b_nk ? launch_tc_inst<T, 128, false>(ta, tb, args, cfg.stages, s)
                    : launch_tc_inst<T, 128, true>(ta, tb, args, cfg.stages, s);
    return BI_ERR_UNSUPPORTED;
}

}  // namespace bi
