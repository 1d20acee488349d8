// sdpa_pair.cu -- the attention of sdpa.cu with two query tiles per block, for
// calls that have at least two (prefill).  Every row is computed exactly as the
// one-tile kernel computes it -- the same chunks, the same S and P V MMAs, the
// same visibility tests, shift, exponentials, partial sums in the same order,
// the same rounding of P and of the output -- so a token's bits are the same
// whichever kernel serves the call; only the scheduling differs.
//
// "mlx-batch-invariant" README, "How the kernels work" / Attention (one pass over
// the keys in a fixed order, online softmax in fp32, no split over the keys).
//
// Why two tiles: in the one-tile kernel the row warps' softmax of a chunk is the
// critical path and the tensor pipe idles more than half the time.  Here the
// MMAs of one tile run while the other tile's rows work.
//
// Layout per block (384 threads, three warpgroups):
//   warp 0 lane 0   copy producer: Q of both tiles once; K and V chunks through
//                   2-deep rings shared by the tiles
//   warp 1          TMEM allocation; lane 0 issues the MMAs
//   warps 2, 3      idle (they complete the first warpgroup)
//   warps 4..7      rows of tile a (the later positions), one warp per TMEM lane
//                   quarter, one thread per row
//   warps 8..11     rows of tile b (the Qt positions before tile a), when the call
//                   has them
// The first warpgroup gives up registers (56 a thread) and the two row warpgroups
// take them (224): 128 * 56 + 256 * 224 = 384 * 168, the registers the block is
// launched with.  The host checks that the compiled kernel asks for exactly 168
// before it ever launches it.
//
// Tensor memory (512 columns): tile t owns [256 t, 256 t + 256): S (C fp32
// columns), then O (DP columns).  P (C keys of the input dtype, two to a column)
// is written over the first C/2 columns of its own S once the row has read S.
//
// MMA order, step j = 0..n (n = chunks of tile a; tile b, which ends at most one
// chunk earlier, visits the same chunks: a chunk entirely masked for a row leaves
// its bits alone):
//   wait for K_j and V_{j-1};
//   for each tile: wait for P_{j-1}; P_{j-1} V_{j-1}; then, once that P V has
//   completed (its S buffer holds P_{j-1}), S(j);
//   one commit frees K slot j % 2 (both tiles' S(j)), one frees V slot (j-1) % 2.
// The rows wait only for S(j): its commit follows the MMA thread's wait for
// P_{j-1} V_{j-1}, so O is also ready for a rescale by then.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_tc.cuh"  // IsBf16
#include "internal.cuh"
#include "ptx.cuh"
#include "sdpa_common.cuh"

namespace bi {

namespace {

constexpr int P2_ROWS = 128;
constexpr int P2_THREADS = 384;
constexpr int P2_LAUNCH_REGS = 168;                // 65536 / 384, rounded down to 8
constexpr int P2_REGS_LOW = 56;                    // producer / MMA warpgroup
constexpr int P2_REGS_HIGH = 224;                  // row warpgroups
static_assert(128 * P2_REGS_LOW + 256 * P2_REGS_HIGH <= P2_THREADS * P2_LAUNCH_REGS,
              "register split above the launch's registers");
constexpr uint32_t P2_QPANEL = P2_ROWS * 128;      // 16 KB: 128 rows x 64 elements
constexpr float P2_LAG = 8.0f;                     // as in sdpa.cu

template <int DP, int C>
struct P2Smem {
    static constexpr uint32_t NP = DP / 64;
    static constexpr uint32_t KPANEL = C * 128;
    static constexpr uint32_t QB = NP * P2_QPANEL;
    static constexpr uint32_t KV = NP * KPANEL;
    static constexpr uint32_t QA = 0;
    static constexpr uint32_t QBT = QA + QB;
    static constexpr uint32_t K = QBT + QB;
    static constexpr uint32_t V = K + 2 * KV;
    static constexpr uint32_t BARS = V + 2 * KV;
    // bar_q kvfull[2] kfree[2] vfree[2] sfull[2] pfull[2] pvdone[2] mma_done
    static constexpr uint32_t NBARS = 1 + 2 + 2 + 2 + 2 + 2 + 2 + 1;
    static constexpr uint32_t MISC = BARS + NBARS * 8;
    static constexpr uint32_t END = MISC + 16;
    static constexpr size_t BYTES = 1024 + END;
    static constexpr uint32_t TILE_COLS = 256;     // S (C) then O (DP) per tile
    static constexpr uint32_t O_OFF = C;
    static_assert(C + DP <= TILE_COLS, "tensor memory per tile");
};

__device__ __forceinline__ void setmaxnreg_inc224() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 224;" ::: "memory");
}
__device__ __forceinline__ void setmaxnreg_dec56() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
}
static_assert(P2_REGS_HIGH == 224 && P2_REGS_LOW == 56, "the asm above names the split");

template <typename T, bool ARR, int DP, int C>
__global__ void __launch_bounds__(P2_THREADS, 1)
    sdpa_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const SdpaArgs args) {
    using Sm = P2Smem<DP, C>;
    constexpr uint32_t NP = Sm::NP;
    constexpr int HK = 64;               // keys of one half (the one-tile kernel's row warp share)
    constexpr int NH = C / HK;           // halves per chunk
    static_assert(C == 128 && (DP == 64 || DP == 128), "built shapes");
    constexpr uint32_t IDESC_S = mma_idesc(IsBf16<T>::value, P2_ROWS, C, false);
    constexpr uint32_t IDESC_PV = mma_idesc(IsBf16<T>::value, P2_ROWS, DP, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sQ[2] = {smem + Sm::QA, smem + Sm::QBT};
    uint8_t *sK = smem + Sm::K;
    uint8_t *sV = smem + Sm::V;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Sm::BARS);
    uint64_t *bar_q = bars;
    uint64_t *kvfull = bar_q + 1;        // [j & 1] step j: K_j and V_{j-1} have landed
    uint64_t *kfree = kvfull + 2;        // [j & 1] both tiles' S(j) done: K slot j % 2 free
    uint64_t *vfree = kfree + 2;         // [i & 1] both tiles' P_i V_i done: V slot i % 2 free
    uint64_t *sfull = vfree + 2;         // [t] S(j) of tile t in its buffer
    uint64_t *pfull = sfull + 2;         // [t] P_j of tile t written, O rescaled
    uint64_t *pvdone = pfull + 2;        // [t] P_i V_i of tile t added into O
    uint64_t *mma_done = pvdone + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Sm::MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Sm::MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int G = args.group;
    const int Qt = args.qt;
    const int64_t q_offset = args.q_offset;
    const int64_t Lq = args.Lq, Lkv = args.Lkv;
    const int64_t t_first = q_offset / Qt;
    const int64_t t_last = (q_offset + Lq - 1) / Qt;
    const int64_t tile_a = t_last - 2 * static_cast<int64_t>(blockIdx.x);
    const bool has_b = tile_a - 1 >= t_first;
    const int NT = has_b ? 2 : 1;
    const int kvh = static_cast<int>(blockIdx.y);
    const int b = static_cast<int>(blockIdx.z);
    int64_t p_max = tile_a * Qt + Qt - 1;
    if (p_max > q_offset + Lq - 1) p_max = q_offset + Lq - 1;
    const int nchunks = args.mode == 1 ? static_cast<int>(p_max / C + 1)
                                       : static_cast<int>((Lkv + C - 1) / C);

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        mbar_init(bar_q, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&kvfull[i], 1);
            mbar_init(&kfree[i], 1);
            mbar_init(&vfree[i], 1);
            mbar_init(&sfull[i], 1);
            mbar_init(&pfull[i], 4);
            mbar_init(&pvdone[i], 1);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp < 4) {
        setmaxnreg_dec56();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------ copy producer
            const int32_t qi0 = static_cast<int32_t>(tile_a * Qt - q_offset);   // may be negative
            mbar_arrive_expect_tx(bar_q, static_cast<uint32_t>(NT) * Sm::QB);
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (uint32_t pn = 0; pn < NP; ++pn)
                    tma_load_4d(sQ[t] + pn * P2_QPANEL, &tmQ, bar_q, 64 * pn, kvh * G, qi0 - t * Qt, b);
            // Step j puts K_j and V_{j-1} on one barrier, after both tiles' S(j-2) have
            // freed K slot j % 2 and both tiles' P_{j-3} V_{j-3} V slot (j-1) % 2.  Those
            // commits follow the MMA thread's wait on step j-2's barrier, so it is never
            // armed again before that phase has been consumed.
            int armed = 0;
            bool ok = true;
            for (int j = 0; j <= nchunks; ++j) {
                const bool has_k = j < nchunks, has_v = j >= 1;
                if (!mbar_wait(&kfree[j & 1], ((j >> 1) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                if (has_v && !mbar_wait(&vfree[(j - 1) & 1], (((j - 1) >> 1) & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&kvfull[j & 1], (has_k ? Sm::KV : 0u) + (has_v ? Sm::KV : 0u));
                if (has_k) {
#pragma unroll
                    for (uint32_t pn = 0; pn < NP; ++pn)
                        tma_load_4d(sK + (j & 1) * Sm::KV + pn * Sm::KPANEL, &tmK, &kvfull[j & 1],
                                    64 * pn, j * C, kvh, b);
                }
                if (has_v) {
#pragma unroll
                    for (uint32_t pn = 0; pn < NP; ++pn)
                        tma_load_4d(sV + ((j - 1) & 1) * Sm::KV + pn * Sm::KPANEL, &tmV, &kvfull[j & 1],
                                    64 * pn, (j - 1) * C, kvh, b);
                }
                armed = j + 1;
            }
            if (!ok) {
                mbar_wait_limited(bar_q, 0, WAIT_LIMIT_NS);
                for (int j = armed - 2 < 0 ? 0 : armed - 2; j < armed; ++j)
                    mbar_wait_limited(&kvfull[j & 1], (j >> 1) & 1u, WAIT_LIMIT_NS);
            }
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------ MMA issuer
            bool ok = mbar_wait(bar_q, 0, abort_flag);
            tc_fence_after();
            for (int j = 0; ok && j <= nchunks; ++j) {
                if (!mbar_wait(&kvfull[j & 1], (j >> 1) & 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                for (int t = 0; ok && t < NT; ++t) {
                    const uint32_t s_col = tmem_base + t * Sm::TILE_COLS;
                    const uint32_t o_col = s_col + Sm::O_OFF;
                    if (j >= 1) {
                        // O_t (+)= P_i V_i, i = j - 1, P from the first C/2 columns of S_t
                        const int i = j - 1;
                        if (!mbar_wait(&pfull[t], i & 1u, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t v_addr = smem_u32(sV + (i & 1) * Sm::KV);
#pragma unroll
                        for (int kk = 0; kk < C / 16; ++kk)
                            mma_f16_ts(o_col, s_col + kk * 8,
                                       smem_desc(v_addr + kk * 2048, Sm::KPANEL, 1024), IDESC_PV,
                                       (i > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(&pvdone[t]);
                    }
                    if (j < nchunks) {
                        // S_t holds P_{j-1}: wait until its P V has read it
                        if (j >= 1) {
                            if (!mbar_wait(&pvdone[t], (j - 1) & 1u, abort_flag)) { ok = false; break; }
                            tc_fence_after();
                        }
                        const uint32_t q_addr = smem_u32(sQ[t]);
                        const uint32_t k_addr = smem_u32(sK + (j & 1) * Sm::KV);
#pragma unroll
                        for (int kk = 0; kk < DP / 16; ++kk)
                            mma_f16_ss(s_col,
                                       smem_desc(q_addr + (kk >> 2) * P2_QPANEL + (kk & 3) * 32, 16, 1024),
                                       smem_desc(k_addr + (kk >> 2) * Sm::KPANEL + (kk & 3) * 32, 16, 1024),
                                       IDESC_S, kk > 0 ? 1u : 0u);
                        mma_commit(&sfull[t]);
                    }
                }
                if (!ok) break;
                if (j < nchunks) mma_commit(&kfree[j & 1]);
                if (j >= 1) mma_commit(&vfree[(j - 1) & 1]);
            }
            mma_commit(mma_done);
            mbar_wait_limited(mma_done, 0, WAIT_LIMIT_NS);
        }
    } else {
        setmaxnreg_inc224();
        // ------------------------------------------------ rows: one thread per query row
        const int t = (warp - 4) >> 2;
        if (t < NT) {
            const uint32_t quarter = static_cast<uint32_t>(warp & 3);
            const int r = static_cast<int>(quarter) * 32 + lane;
            const int qi = r / G, g = r - (r / G) * G;
            const int64_t pos = (tile_a - t) * Qt + qi;
            const bool valid = pos >= q_offset && pos < q_offset + Lq;
            const bool warp_valid = __any_sync(0xffffffffu, valid) != 0;
            const uint32_t lane_base = (quarter * 32u) << 16;
            const uint32_t s_addr = tmem_base + lane_base + t * Sm::TILE_COLS;
            const uint32_t o_addr = s_addr + Sm::O_OFF;
            const float sl2 = args.scale_log2;
            const int h = kvh * G + g;
            int64_t vis_end = args.mode == 1 ? pos + 1 : Lkv;
            if (vis_end > Lkv) vis_end = Lkv;
            if (!valid) vis_end = INT64_MAX / 2;
            const uint8_t *mrow = nullptr;
            if (ARR && valid)
                mrow = args.mask + b * args.ms[0] + h * args.ms[1] + (pos - q_offset) * args.ms[2];
            float m_run = -INFINITY, l_run = 0.0f;
            if (args.sinks) {
                m_run = __fmul_rn(args.sinks[h], 1.44269504088896341f);
                l_run = 1.0f;
            }

            for (int j = 0; j < nchunks; ++j) {
                // per half: visibility (array mask bits or the causal / length limit)
                uint64_t vis[NH];
                int lim[NH];
                bool full[NH];
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) {
                    const int64_t key0 = static_cast<int64_t>(j) * C + hh * HK;
                    vis[hh] = ~0ull;
                    if (ARR && mrow) vis[hh] = mask_bits64(mrow + key0, Lkv - key0);
                    lim[hh] = HK;
                    if (!ARR) {
                        const int64_t lim64 = vis_end - key0;
                        lim[hh] = lim64 < 0 ? 0 : (lim64 > HK ? HK : static_cast<int>(lim64));
                    }
                }
                warp_wait(&sfull[t], j & 1u, abort_flag);
                tc_fence_after();
#pragma unroll
                for (int hh = 0; hh < NH; ++hh)
                    full[hh] = __all_sync(0xffffffffu, ARR ? vis[hh] == ~0ull : lim[hh] == HK) != 0;
                float x[C];
                float mh[NH];
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) mh[hh] = -INFINITY;
                if (warp_valid) {
#pragma unroll
                    for (int c32 = 0; c32 < C / 32; ++c32) {
                        uint32_t(&xu)[32] = *reinterpret_cast<uint32_t(*)[32]>(x + 32 * c32);
                        tmem_ld32(s_addr + 32 * c32, xu);
                    }
                    tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(x));
#pragma unroll
                    for (int c32 = 1; c32 < C / 32; ++c32)
                        tmem_tie(*reinterpret_cast<uint32_t(*)[32]>(x + 32 * c32));
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh) {
                        const float *xh = x + hh * HK;
                        if (full[hh]) {
#pragma unroll
                            for (int i = 0; i < HK; i += 2) mh[hh] = fmax3(mh[hh], xh[i], xh[i + 1]);
                        } else {
#pragma unroll
                            for (int i = 0; i < HK; ++i)
                                if (ARR ? ((vis[hh] >> i) & 1u) != 0 : i < lim[hh]) mh[hh] = fmaxf(mh[hh], xh[i]);
                        }
                    }
                }
                float mraw = mh[0];
#pragma unroll
                for (int hh = 1; hh < NH; ++hh) mraw = fmaxf(mraw, mh[hh]);
                const bool any = mraw != -INFINITY;
                const float cand = __fmul_rn(mraw, sl2);
                const bool raise = any && cand > __fadd_rn(m_run, P2_LAG);
                const float m_new = raise ? cand : m_run;
                const float alpha = raise ? ex2_approx(__fsub_rn(m_run, m_new)) : 1.0f;
                // each half's keys in pairs, partial sum (key mod 4) k in ls01 (k = 0, 1)
                // or ls23 (k = 2, 3), added in ascending key order, as the one-tile
                // kernel's row warps do; P packed two keys to a 32-bit word
                float lsh[NH];
                uint32_t pw[C / 2];
                if (warp_valid) {
                    const float2 c2 = make_float2(sl2, sl2), nm2 = make_float2(-m_new, -m_new);
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh) {
                        const float *xh = x + hh * HK;
                        float2 ls01 = make_float2(0.0f, 0.0f), ls23 = make_float2(0.0f, 0.0f);
                        if (full[hh]) {
#pragma unroll
                            for (int i = 0; i < HK; i += 2) {
                                const float2 tt = __ffma2_rn(make_float2(xh[i], xh[i + 1]), c2, nm2);
                                const float e0 = ex2_approx(tt.x), e1 = ex2_approx(tt.y);
                                pw[(hh * HK + i) >> 1] = cvt2<T>(e0, e1);
                                if ((i & 2) == 0) ls01 = __fadd2_rn(ls01, make_float2(e0, e1));
                                else ls23 = __fadd2_rn(ls23, make_float2(e0, e1));
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < HK; i += 2) {
                                const float2 tt = __ffma2_rn(make_float2(xh[i], xh[i + 1]), c2, nm2);
                                float e0 = ex2_approx(tt.x), e1 = ex2_approx(tt.y);
                                if (ARR ? ((vis[hh] >> i) & 1u) == 0 : i >= lim[hh]) e0 = 0.0f;
                                if (ARR ? ((vis[hh] >> (i + 1)) & 1u) == 0 : i + 1 >= lim[hh]) e1 = 0.0f;
                                pw[(hh * HK + i) >> 1] = cvt2<T>(e0, e1);
                                if ((i & 2) == 0) ls01 = __fadd2_rn(ls01, make_float2(e0, e1));
                                else ls23 = __fadd2_rn(ls23, make_float2(e0, e1));
                            }
                        }
                        lsh[hh] = __fadd_rn(__fadd_rn(ls01.x, ls01.y), __fadd_rn(ls23.x, ls23.y));
                    }
                    // P over the first C/2 columns of S (this thread has read its row of S)
#pragma unroll
                    for (int w32 = 0; w32 < C / 64; ++w32)
                        tmem_st32(s_addr + 32 * w32, *reinterpret_cast<const uint32_t(*)[32]>(pw + 32 * w32));
                } else {
#pragma unroll
                    for (int hh = 0; hh < NH; ++hh) lsh[hh] = 0.0f;
                }
                // O *= alpha (skipped when every row of the warp has alpha 1).  P_{j-1} V_{j-1}
                // is complete: the MMA thread waited for it before issuing S(j).
                if (j >= 1 && warp_valid && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
                    for (int c4 = 0; c4 < DP / 32; ++c4) {
                        uint32_t ov[32];
                        tmem_ld32(o_addr + c4 * 32, ov);
                        tmem_wait_ld(ov);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            ov[e] = __float_as_uint(__fmul_rn(__uint_as_float(ov[e]), alpha));
                        tmem_st32(o_addr + c4 * 32, ov);
                    }
                }
                if (warp_valid) tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&pfull[t]);
                if (any) {
                    // the halves' sums as the one-tile kernel adds its two row warps' sums
                    float lchunk = lsh[0];
#pragma unroll
                    for (int hh = 1; hh < NH; ++hh) lchunk = __fadd_rn(lchunk, lsh[hh]);
                    l_run = __fadd_rn(__fmul_rn(l_run, alpha), lchunk);
                    m_run = m_new;
                }
            }
            // the last P V, then o = acc / l
            warp_wait(&pvdone[t], (nchunks - 1) & 1u, abort_flag);
            tc_fence_after();
            if (warp_valid) {
                T *orow = static_cast<T *>(args.o) + b * args.os[0] + h * args.os[1] +
                          (pos - q_offset) * args.os[2];
#pragma unroll 1
                for (int c4 = 0; c4 < DP / 32; ++c4) {
                    uint32_t ov[32];
                    tmem_ld32(o_addr + c4 * 32, ov);
                    tmem_wait_ld(ov);
                    if (valid && !*abort_flag) {
#pragma unroll
                        for (int d8 = 0; d8 < 4; ++d8) {
                            const int col = c4 * 32 + d8 * 8;
                            if (col >= args.D) break;        // padded columns past the head dim
                            float v[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                v[e] = __fdiv_rn(__uint_as_float(ov[d8 * 8 + e]), l_run);
                            *reinterpret_cast<uint4 *>(orow + col) = pack8<T>(v);
                        }
                    }
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(args.err, ERR_TIMEOUT);
}

// Per instantiation: set up at library initialisation; usable only if the compiled
// kernel asks for exactly the registers the split above is computed from.
template <typename T, bool ARR, int DP, int C>
bool &p2_usable() {
    static bool ok = false;
    return ok;
}

template <typename T, bool ARR, int DP, int C>
bi_status p2_init() {
    auto *fn = sdpa_pair_kernel<T, ARR, DP, C>;
    bi_status st = cuda_status(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    static_cast<int>(P2Smem<DP, C>::BYTES)));
    if (st != BI_OK) return st;
    cudaFuncAttributes fa;
    if ((st = cuda_status(cudaFuncGetAttributes(&fa, fn))) != BI_OK) return st;
    p2_usable<T, ARR, DP, C>() = fa.numRegs == P2_LAUNCH_REGS && fa.maxThreadsPerBlock >= P2_THREADS;
    return BI_OK;
}

template <typename T, bool ARR, int DP, int C>
bi_status p2_launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                    const SdpaArgs &args, cudaStream_t s, bool *used) {
    if (!p2_usable<T, ARR, DP, C>()) return BI_OK;
    const int64_t tiles = (args.q_offset + args.Lq - 1) / args.qt - args.q_offset / args.qt + 1;
    if (tiles < 2) return BI_OK;
    const int64_t blocks = (tiles + 1) / 2;
    if (blocks > 0x7fffffff || args.Hkv > 65535 || args.B > 65535) return BI_ERR_UNSUPPORTED;
    dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(args.Hkv),
              static_cast<unsigned>(args.B));
    sdpa_pair_kernel<T, ARR, DP, C><<<grid, P2_THREADS, P2Smem<DP, C>::BYTES, s>>>(tq, tk, tv, args);
    count_launch();
    *used = true;
    return cuda_status(cudaGetLastError());
}

template <typename T, int DP>
bi_status p2_mask(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                  const SdpaArgs &args, cudaStream_t s, bool *used) {
    return args.mode == 2 ? p2_launch<T, true, DP, 128>(tq, tk, tv, args, s, used)
                          : p2_launch<T, false, DP, 128>(tq, tk, tv, args, s, used);
}

template <typename T>
bi_status p2_shape(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                   const SdpaArgs &args, cudaStream_t s, bool *used) {
    if (args.chunk != 128) return BI_OK;
    if (args.dp == 128) return p2_mask<T, 128>(tq, tk, tv, args, s, used);
    if (args.dp == 64) return p2_mask<T, 64>(tq, tk, tv, args, s, used);
    return BI_OK;
}

template <typename T>
bi_status p2_inits() {
    bi_status (*const fns[])() = {p2_init<T, false, 128, 128>, p2_init<T, true, 128, 128>,
                                  p2_init<T, false, 64, 128>, p2_init<T, true, 64, 128>};
    for (auto f : fns) {
        const bi_status st = f();
        if (st != BI_OK) return st;
    }
    return BI_OK;
}

}  // namespace

bi_status init_sdpa_pair() {
    const bi_status st = p2_inits<__nv_bfloat16>();
    return st != BI_OK ? st : p2_inits<__half>();
}

bi_status launch_sdpa_pair(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const SdpaArgs &args, bi_dtype dt, cudaStream_t s, bool *used) {
    *used = false;
    if (dt == BI_BF16) return p2_shape<__nv_bfloat16>(tq, tk, tv, args, s, used);
    if (dt == BI_F16) return p2_shape<__half>(tq, tk, tv, args, s, used);
    return BI_OK;
}

}  // namespace bi
