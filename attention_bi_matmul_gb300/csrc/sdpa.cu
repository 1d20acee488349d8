// sdpa.cu -- batch-invariant causal GQA attention on the 5th-generation tensor
// cores, the output accumulated in tensor memory.
//
// "mlx-batch-invariant" README, "How the kernels work" / Attention: a single
// pass over the keys in a fixed order with an online softmax in fp32, no split
// over the keys, no second pass, no route switching; "Why MLX is not
// invariant" / Attention: the answer for a token must not change with the
// query length (decode vs chunked prefill), the GQA factor times query length,
// or with keys appended to the cache; the closing limits paragraph: head dims
// are multiples of 32.  The GB300 form of that rule:
//
//   * one block per (query tile, kv head, batch).  A query tile holds 128 rows:
//     Qt = 128 / G absolute positions [t*Qt, t*Qt+Qt) times the G = H/Hkv query
//     heads that share the kv head, row = (position mod Qt) * G + head.  A token
//     therefore sits in the same row of the same tile for every query length;
//   * keys are visited in chunks of C at absolute key positions 0, C, 2C, ...
//     in ascending order, C = 128 for head dims up to 128 and 64 above (a
//     function of the head dim alone).  For each chunk: S = Q K^T
//     (tcgen05.mma into tensor memory); the mask (causal: key j visible iff
//     j <= position; none; or a boolean array); with c = scale * log2 e and
//     x = (max of the visible s_j) * c, the row's shift m moves to m' = x only
//     if x > m + 8, and otherwise stays (m' = m): the shift may lag the
//     running maximum by up to 8, so p <= 2^8, and most chunks leave it and
//     the accumulator alone; alpha = 2^(m - m') (exactly 1 when m' = m);
//     p_j = 2^(fma(s_j, c, -m')); l = l * alpha + (half sum + half sum), each
//     half summed as four interleaved partial sums (key mod 4) added as
//     (0+1)+(2+3); P rounded to the input dtype;
//   * P is written into tensor memory and read from there by the P V MMA (its A
//     operand); the output is one fp32 accumulator in tensor memory that the
//     P V MMA adds into: before chunk j's P V, every row rescales it by alpha_j (one fp32
//     multiply per element, rounded to nearest).  A warp whose 32 rows all have
//     alpha = 1 skips the rescale: multiplying by 1 is exact, so the bits do
//     not depend on which rows share the warp.  2^x is the hardware's
//     ex2.approx.ftz.f32;
//   * a chunk entirely masked for a row has alpha = 1 and p = 0: the rescale
//     and the added zeros leave m, l and the accumulator unchanged, so extra
//     chunks that a longer query tile visits, or keys appended beyond a token,
//     change none of its bits;
//   * o = acc * (1 / l) (the reciprocal correctly rounded, then one fp32 multiply),
//     rounded once to the output dtype;
//   * an attention sink (one extra logit per head, no value) enters as the
//     initial state m = sink * log2 e, l = 1.
// Head dims that are not a multiple of 64 are loaded with the copy engine's zero
// fill past D (they add exact zeros to Q K^T) and the columns past D are never
// stored.  Every quantity of a row depends only on that row's query, the keys and
// values, the chunk positions and the row's absolute position -- never on which
// other rows share the tile.
//
// Roles (320 threads):
//   warp 0 lane 0   TMA producer (Q once; K and V chunks through 2-deep rings)
//   warp 1          TMEM allocation (S0, S1 of C columns, O of DP, P0, P1 of
//                   C/2); lane 0 issues the MMAs, waiting for K_j before S(j)
//                   and for P_{j-1} and V_{j-1} before P V(j-1)
//   warps 2..9      row warps: warp w serves TMEM lane quarter w % 4 and half
//                   (w-2)/4 of the keys (C/2) and of the output columns (DP/2);
//                   the two warps of a row exchange the chunk maximum and the
//                   half sums through shared memory (named barrier per quarter).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "gemm_tc.cuh"  // IsBf16 / pack8
#include "internal.cuh"
#include "ptx.cuh"
#include "sdpa_common.cuh"

namespace bi {

namespace {

constexpr int S2_ROWS = 128;       // rows per query tile
constexpr int S2_KST = 2;          // K ring depth
constexpr int S2_VST = 2;          // V ring depth
// The slot releases are the MMA's completion barriers sfull[j & 1] and pvdone[i & 1],
// so each ring has as many slots as those barriers have entries.
static_assert(S2_KST == 2 && S2_VST == 2, "ring depth tied to the completion barriers");
constexpr int S2_THREADS = 320;
constexpr uint32_t S2_QPANEL = S2_ROWS * 128;     // 16 KB: 128 rows x 64 elements
constexpr float S2_LAG = 8.0f;     // how far a row's shift may lag its running maximum (log2)

// DP: padded head dim (64, 128, 256); C: keys per chunk (64 or 128).
template <int DP, int C>
struct S2Smem {
    static constexpr uint32_t NP = DP / 64;                      // head-dim panels
    static constexpr uint32_t KPANEL = C * 128;                  // C keys x 64 elements
    static constexpr uint32_t QB = NP * S2_QPANEL;
    static constexpr uint32_t KV = NP * KPANEL;                  // one K or V chunk
    static constexpr uint32_t Q = 0;
    static constexpr uint32_t K = Q + QB;
    static constexpr uint32_t V = K + S2_KST * KV;
    static constexpr uint32_t MX = V + S2_VST * KV;              // float[2][128] half maxima
    static constexpr uint32_t LS = MX + 2 * 128 * 4;             // float[2][128] half sums
    static constexpr uint32_t BARS = LS + 2 * 128 * 4;
    // bar_q kfull[2] vfull[2] sfull[2] pfull[2] pvdone[2] mma_done
    static constexpr uint32_t NBARS = 1 + 2 + 2 + 2 + 2 + 2 + 1;
    static constexpr uint32_t MISC = BARS + NBARS * 8;           // tmem slot, abort flag
    static constexpr uint32_t END = MISC + 16;
    static constexpr size_t BYTES = 1024 + END;
    // tensor memory: S0 [0, C), S1 [C, 2C), O [2C, 2C + DP), then P0 and P1 of C/2
    // columns each (C keys of the input dtype, two to a column)
    static constexpr uint32_t O_COL = 2 * C;
    static constexpr uint32_t P_COL = 2 * C + DP;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(P_COL + C <= TMEM_COLS, "tensor memory");
};

template <typename T, bool ARR, int DP, int C>
__global__ void __launch_bounds__(S2_THREADS, 1)
    sdpa_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const SdpaArgs args) {
    using S2Smem = bi::S2Smem<DP, C>;
    constexpr uint32_t NP = S2Smem::NP;
    constexpr uint32_t S2_KPANEL = S2Smem::KPANEL;
    constexpr uint32_t S2_KV = S2Smem::KV;
    constexpr uint32_t S2_O_COL = S2Smem::O_COL;
    constexpr uint32_t S2_P_COL = S2Smem::P_COL;
    constexpr uint32_t S2_TMEM_COLS = S2Smem::TMEM_COLS;
    constexpr int S2_C = C;
    constexpr int HK = C / 2;            // keys per row warp
    constexpr int HD = DP / 2;           // output columns per row warp
    static_assert(HK == 64 || HK == 32, "row warps hold 32 or 64 keys of a chunk");
    constexpr uint32_t IDESC_S = mma_idesc(IsBf16<T>::value, S2_ROWS, C, false);
    constexpr uint32_t IDESC_PV = mma_idesc(IsBf16<T>::value, S2_ROWS, DP, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem + S2Smem::Q;
    uint8_t *sK = smem + S2Smem::K;
    uint8_t *sV = smem + S2Smem::V;
    float *mx_s = reinterpret_cast<float *>(smem + S2Smem::MX);
    float *ls_s = reinterpret_cast<float *>(smem + S2Smem::LS);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S2Smem::BARS);
    uint64_t *bar_q = bars;
    uint64_t *kfull = bar_q + 1;         // [j & 1]: K_j has landed in K slot j % 2
    uint64_t *vfull = kfull + 2;         // [i & 1]: V_i has landed in V slot i % 2
    // S(j) done: S buffer j & 1 written, and K slot j % 2 read (the producer's
    // release too)
    uint64_t *sfull = vfull + 2;         // [2]
    // [j & 1]: P_j in tensor memory and O rescaled for chunk j.  Two barriers, not one:
    // a row warp with no valid rows may arrive for chunk j + 1 (S(j + 1) is issued
    // before the MMA thread waits for P_j) before the others arrive for chunk j, and
    // one barrier would then count that arrival towards chunk j.  It cannot get two
    // chunks ahead: S(j + 2) is issued only after P_j's barrier has completed.
    uint64_t *pfull = sfull + 2;         // [2]
    // P_i V_i added into O, i.e. P buffer i & 1 free, O readable, V slot i % 2 read: [i & 1]
    uint64_t *pvdone = pfull + 2;        // [2]
    uint64_t *mma_done = pvdone + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S2Smem::MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S2Smem::MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int G = args.group;
    const int Qt = args.qt;
    const int64_t q_offset = args.q_offset;
    const int64_t Lq = args.Lq, Lkv = args.Lkv;
    // Query tiles of this call, heaviest (latest positions) first.
    const int64_t t_last = (q_offset + Lq - 1) / Qt;
    const int64_t tile = t_last - static_cast<int64_t>(blockIdx.x);
    const int kvh = static_cast<int>(blockIdx.y);
    const int b = static_cast<int>(blockIdx.z);
    const int64_t p_lo = tile * Qt;
    int64_t p_max = p_lo + Qt - 1;
    if (p_max > q_offset + Lq - 1) p_max = q_offset + Lq - 1;
    const int nchunks = args.mode == 1 ? static_cast<int>(p_max / S2_C + 1)
                                       : static_cast<int>((Lkv + S2_C - 1) / S2_C);

    if (threadIdx.x == 0) {
        // Thread 0 is also the copy producer: the copy descriptors are fetched and the
        // block's first copies (Q, and K_0 for step 0) go out before the rest of the
        // block's setup, so that their latency overlaps it.
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        mbar_init(bar_q, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&kfull[s], 1);
            mbar_init(&vfull[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sfull[i], 1);
        }
        mbar_init(&pfull[0], 8);
        mbar_init(&pfull[1], 8);
        mbar_init(&pvdone[0], 1);
        mbar_init(&pvdone[1], 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
        const int32_t qi0 = static_cast<int32_t>(p_lo - q_offset);  // may be negative
        mbar_arrive_expect_tx(bar_q, S2Smem::QB);
#pragma unroll
        for (uint32_t pn = 0; pn < NP; ++pn)
            tma_load_4d(sQ + pn * S2_QPANEL, &tmQ, bar_q, 64 * pn, kvh * G, qi0, b);
        // K_0 (nchunks >= 1), into K slot 0
        mbar_arrive_expect_tx(&kfull[0], S2_KV);
#pragma unroll
        for (uint32_t pn = 0; pn < NP; ++pn)
            tma_load_4d(sK + pn * S2_KPANEL, &tmK, &kfull[0], 64 * pn, 0, kvh, b);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, S2_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            // Q and K_0 were issued during the block's setup.  Step j loads K_j once S(j-2)
            // is done (K slot j % 2 read), then V_{j-1} once P_{j-3} V_{j-3} is done (V slot
            // (j-1) % 2 read); each onto its own barrier, so that K_j, which S(j) needs
            // first, does not wait for a V slot.  The slot releases are the MMA's own
            // completion barriers.  A fill barrier is armed again only after the MMA that
            // read its previous contents is done, and the MMA thread waited for that
            // phase before issuing it, so no phase is armed before it has been consumed.
            int k_armed = 1, v_armed = 0;    // K_0..K_{k_armed-1}, V_0..V_{v_armed-1} issued
            bool ok = true;
            for (int j = 1; j <= nchunks; ++j) {
                if (j < nchunks) {
                    if (!mbar_wait(&sfull[j & 1], ((j >> 1) & 1u) ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&kfull[j & 1], S2_KV);
#pragma unroll
                    for (uint32_t pn = 0; pn < NP; ++pn)
                        tma_load_4d(sK + (j % S2_KST) * S2_KV + pn * S2_KPANEL, &tmK, &kfull[j & 1],
                                    64 * pn, j * S2_C, kvh, b);
                    k_armed = j + 1;
                }
                const int i = j - 1;
                if (!mbar_wait(&pvdone[i & 1], ((i >> 1) & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&vfull[i & 1], S2_KV);
#pragma unroll
                for (uint32_t pn = 0; pn < NP; ++pn)
                    tma_load_4d(sV + (i % S2_VST) * S2_KV + pn * S2_KPANEL, &tmV, &vfull[i & 1],
                                64 * pn, i * S2_C, kvh, b);
                v_armed = j;
            }
            if (!ok) {
                // Let every copy already issued land before the block can exit.
                mbar_wait_limited(bar_q, 0, WAIT_LIMIT_NS);
                for (int k = k_armed - 2 < 0 ? 0 : k_armed - 2; k < k_armed; ++k)
                    mbar_wait_limited(&kfull[k & 1], (k >> 1) & 1u, WAIT_LIMIT_NS);
                for (int k = v_armed - 2 < 0 ? 0 : v_armed - 2; k < v_armed; ++k)
                    mbar_wait_limited(&vfull[k & 1], (k >> 1) & 1u, WAIT_LIMIT_NS);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            // Every descriptor the loop uses, computed once (before Q has landed): Q's,
            // and K's and V's for both ring slots.  The MMAs then go out with no
            // arithmetic between them (the issuing thread shares its SMSP with row warps).
            constexpr int NS = DP / 16, NV = C / 16;
            uint64_t qd[NS], kd[2][NS], vd[2][NV];
            {
                const uint32_t q_addr = smem_u32(sQ);
#pragma unroll
                for (int kk = 0; kk < NS; ++kk) {
                    qd[kk] = smem_desc(q_addr + (kk >> 2) * S2_QPANEL + (kk & 3) * 32, 16, 1024);
#pragma unroll
                    for (int sl = 0; sl < 2; ++sl)
                        kd[sl][kk] = smem_desc(smem_u32(sK + sl * S2_KV) + (kk >> 2) * S2_KPANEL +
                                                   (kk & 3) * 32, 16, 1024);
                }
#pragma unroll
                for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                    for (int sl = 0; sl < 2; ++sl)
                        vd[sl][kk] = smem_desc(smem_u32(sV + sl * S2_KV) + kk * 2048, S2_KPANEL, 1024);
            }
            bool ok = mbar_wait(bar_q, 0, abort_flag);
            auto issue_s = [&](const uint64_t (&kds)[NS], uint32_t s_tmem) {
#pragma unroll
                for (int kk = 0; kk < NS; ++kk) mma_f16_ss(s_tmem, qd[kk], kds[kk], IDESC_S, kk > 0 ? 1u : 0u);
            };
            // P from tensor memory (8 columns per 16 keys); V: MN-major, 64-column atoms
            auto issue_pv = [&](const uint64_t (&vds)[NV], uint32_t p_tmem, bool first) {
#pragma unroll
                for (int kk = 0; kk < NV; ++kk)
                    mma_f16_ts(tmem_base + S2_O_COL, p_tmem + kk * 8, vds[kk], IDESC_PV,
                               (!first || kk > 0) ? 1u : 0u);
            };
            for (int j = 0; ok && j <= nchunks; ++j) {
                if (j < nchunks) {
                    if (!mbar_wait(&kfull[j & 1], (j >> 1) & 1u, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    // S(j) = Q K_j^T into S buffer j & 1 (DP / 16 steps over the head dim).
                    // That buffer held S(j-2), which the row warps read before writing
                    // P(j-2), whose barrier this thread waited for at step j-1.
                    const uint32_t sb = j & 1;
                    if (j % S2_KST == 0) issue_s(kd[0], tmem_base + sb * S2_C);
                    else issue_s(kd[1], tmem_base + sb * S2_C);
                    mma_commit(&sfull[sb]);
                }
                if (j >= 1) {
                    // O (+)= P_i V_i, i = j - 1 (the rows rescaled O before signalling)
                    const int i = j - 1;
                    if (!mbar_wait(&pfull[i & 1], (i >> 1) & 1u, abort_flag) ||
                        !mbar_wait(&vfull[i & 1], (i >> 1) & 1u, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t p_tmem = tmem_base + S2_P_COL + (i & 1) * (C / 2);
                    if (i % S2_VST == 0) issue_pv(vd[0], p_tmem, i == 0);
                    else issue_pv(vd[1], p_tmem, i == 0);
                    mma_commit(&pvdone[i & 1]);
                }
            }
            mma_commit(mma_done);
            mbar_wait_limited(mma_done, 0, WAIT_LIMIT_NS);
        }
    } else {
        // ------------------------------------------------ row warps (2..9)
        // As in the 128-wide kernel these warps never leave the chunk loop early, so
        // the two warps of a lane quarter always meet at the same named barriers.
        const uint32_t quarter = static_cast<uint32_t>(warp & 3);
        const int half = (warp - 2) >> 2;   // keys HK*half..+HK-1; output columns HD*half..+HD-1
        const int r = static_cast<int>(quarter) * 32 + lane;
        const int qi = r / G, g = r - (r / G) * G;
        const int64_t pos = p_lo + qi;
        const bool valid = pos >= q_offset && pos < q_offset + Lq;
        const bool warp_valid = __any_sync(0xffffffffu, valid) != 0;
        const uint32_t lane_base = (quarter * 32u) << 16;
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
        const uint32_t o_addr = tmem_base + lane_base + S2_O_COL + half * HD;

        for (int j = 0; j < nchunks; ++j) {
            const uint32_t sb = j & 1;
            const int64_t key0 = static_cast<int64_t>(j) * S2_C + half * HK;
            using VisT = typename std::conditional<HK == 64, uint64_t, uint32_t>::type;
            VisT vis = ~VisT(0);
            if constexpr (HK == 64) {
                if (ARR && mrow) vis = mask_bits64(mrow + key0, Lkv - key0);
            } else {
                if (ARR && mrow) vis = mask_bits32(mrow + key0, Lkv - key0);
            }
            warp_wait(&sfull[sb], (j >> 1) & 1u, abort_flag);
            tc_fence_after();
            int lim = HK;
            if (!ARR) {
                const int64_t lim64 = vis_end - key0;
                lim = lim64 < 0 ? 0 : (lim64 > HK ? HK : static_cast<int>(lim64));
            }
            const bool full = __all_sync(0xffffffffu, ARR ? vis == ~VisT(0) : lim == HK) != 0;
            float x[HK];
            float mloc = -INFINITY;
            if (warp_valid) {
                // every load of the row's keys in flight before the one wait
#pragma unroll
                for (int c32 = 0; c32 < HK / 32; ++c32) {
                    uint32_t(&xu)[32] = *reinterpret_cast<uint32_t(*)[32]>(x + 32 * c32);
                    tmem_ld32(tmem_base + lane_base + sb * S2_C + half * HK + 32 * c32, xu);
                }
                tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(x));
#pragma unroll
                for (int c32 = 1; c32 < HK / 32; ++c32)
                    tmem_tie(*reinterpret_cast<uint32_t(*)[32]>(x + 32 * c32));
                if (full) {
#pragma unroll
                    for (int i = 0; i < HK; i += 2) mloc = fmax3(mloc, x[i], x[i + 1]);
                } else {
#pragma unroll
                    for (int i = 0; i < HK; ++i)
                        if (ARR ? ((vis >> i) & 1u) != 0 : i < lim) mloc = fmaxf(mloc, x[i]);
                }
            }
            mx_s[half * 128 + r] = mloc;
            pair_sync(quarter);
            const float mraw = fmaxf(mx_s[r], mx_s[128 + r]);
            const bool any = mraw != -INFINITY;
            const float cand = __fmul_rn(mraw, sl2);
            const bool raise = any && cand > __fadd_rn(m_run, S2_LAG);
            const float m_new = raise ? cand : m_run;
            const float alpha = raise ? ex2_approx(__fsub_rn(m_run, m_new)) : 1.0f;
            // Keys in pairs with the packed fp32 forms (each lane rounds as the scalar
            // operation does): partial sum (key mod 4) k lives in ls01 (k = 0, 1) or
            // ls23 (k = 2, 3) and is added in ascending key order.
            float2 ls01 = make_float2(0.0f, 0.0f), ls23 = make_float2(0.0f, 0.0f);
            // P_j goes to P buffer j & 1, which held P_{j-2}.  P_{j-2} V_{j-2} is
            // complete: the MMA thread issued it before S(j), and S(j)'s commit (waited
            // for above) arrives only once every MMA issued before it has completed.
            // Keys HK*half.. of row r, two to a 32-bit column (lower key in the low
            // half), stored 32 keys at a time so that one store is in flight while the
            // next 32 exponentials are computed.
            if (warp_valid) {
                const float2 c2 = make_float2(sl2, sl2), nm2 = make_float2(-m_new, -m_new);
                const uint32_t p_addr = tmem_base + lane_base + S2_P_COL + sb * (C / 2) + half * (HK / 2);
                auto store32 = [&](int k0) {
                    uint32_t pw[16];
#pragma unroll
                    for (int w = 0; w < 16; ++w) pw[w] = cvt2<T>(x[k0 + 2 * w], x[k0 + 2 * w + 1]);
                    tmem_st16(p_addr + k0 / 2, pw);
                };
                // Two copies of the loop, so that the common (unmasked) one has no
                // test between the exponentials; both do the same arithmetic.
                if (full) {
#pragma unroll
                    for (int k0 = 0; k0 < HK; k0 += 32) {
#pragma unroll
                        for (int i = k0; i < k0 + 32; i += 2) {
                            const float2 t = __ffma2_rn(make_float2(x[i], x[i + 1]), c2, nm2);
                            const float e0 = ex2_approx(t.x), e1 = ex2_approx(t.y);
                            x[i] = e0;
                            x[i + 1] = e1;
                            if ((i & 2) == 0) ls01 = __fadd2_rn(ls01, make_float2(e0, e1));
                            else ls23 = __fadd2_rn(ls23, make_float2(e0, e1));
                        }
                        store32(k0);
                    }
                } else {
#pragma unroll
                    for (int k0 = 0; k0 < HK; k0 += 32) {
#pragma unroll
                        for (int i = k0; i < k0 + 32; i += 2) {
                            const float2 t = __ffma2_rn(make_float2(x[i], x[i + 1]), c2, nm2);
                            float e0 = ex2_approx(t.x), e1 = ex2_approx(t.y);
                            if (ARR ? ((vis >> i) & 1u) == 0 : i >= lim) e0 = 0.0f;
                            if (ARR ? ((vis >> (i + 1)) & 1u) == 0 : i + 1 >= lim) e1 = 0.0f;
                            x[i] = e0;
                            x[i + 1] = e1;
                            if ((i & 2) == 0) ls01 = __fadd2_rn(ls01, make_float2(e0, e1));
                            else ls23 = __fadd2_rn(ls23, make_float2(e0, e1));
                        }
                        store32(k0);
                    }
                }
            }
            const float lsum = __fadd_rn(__fadd_rn(ls01.x, ls01.y), __fadd_rn(ls23.x, ls23.y));
            // O *= alpha for this warp's HD columns, after P_{j-1} V_{j-1} is added in
            // (skipped, wait included, when every row has alpha 1)
            if (j >= 1 && warp_valid && __any_sync(0xffffffffu, alpha != 1.0f)) {
                warp_wait(&pvdone[(j - 1) & 1], ((j - 1) >> 1) & 1u, abort_flag);
                tc_fence_after();
#pragma unroll 1
                for (int c4 = 0; c4 < HD / 32; ++c4) {
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
            if (lane == 0) mbar_arrive(&pfull[sb]);
            ls_s[half * 128 + r] = lsum;
            pair_sync(quarter);
            if (any) {
                l_run = __fadd_rn(__fmul_rn(l_run, alpha), __fadd_rn(ls_s[r], ls_s[128 + r]));
                m_run = m_new;
            }
        }
        // the last P V, then o = acc * (1 / l): one correctly rounded reciprocal per row
        warp_wait(&pvdone[(nchunks - 1) & 1], ((nchunks - 1) >> 1) & 1u, abort_flag);
        tc_fence_after();
        const float inv_l = __frcp_rn(l_run);
        if (warp_valid) {
            T *orow = static_cast<T *>(args.o) + b * args.os[0] + h * args.os[1] +
                      (pos - q_offset) * args.os[2] + half * HD;
            // two 32-column loads in flight per wait
            constexpr int OB = HD / 32 < 2 ? HD / 32 : 2;
#pragma unroll 1
            for (int c0 = 0; c0 < HD / 32; c0 += OB) {
                uint32_t ov[OB][32];
#pragma unroll
                for (int u = 0; u < OB; ++u) tmem_ld32(o_addr + (c0 + u) * 32, ov[u]);
                tmem_wait_ld(ov[0]);
#pragma unroll
                for (int u = 1; u < OB; ++u) tmem_tie(ov[u]);
                if (valid && !*abort_flag) {
#pragma unroll
                    for (int u = 0; u < OB; ++u)
#pragma unroll
                        for (int d8 = 0; d8 < 4; ++d8) {
                            const int c4 = c0 + u;
                            const int col = half * HD + c4 * 32 + d8 * 8;
                            if (col >= args.D) break;        // padded columns past the head dim
                            float v[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                v[e] = __fmul_rn(__uint_as_float(ov[u][d8 * 8 + e]), inv_l);
                            *reinterpret_cast<uint4 *>(orow + c4 * 32 + d8 * 8) = pack8<T>(v);
                        }
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, S2_TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(args.err, ERR_TIMEOUT);
}

template <typename T, bool ARR, int DP, int C>
bi_status s2_attr() {
    return cuda_status(cudaFuncSetAttribute(sdpa_kernel<T, ARR, DP, C>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(S2Smem<DP, C>::BYTES)));
}

template <typename T, bool ARR, int DP, int C>
bi_status s2_launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                    const SdpaArgs &args, cudaStream_t s) {
    const int64_t t_first = args.q_offset / args.qt;
    const int64_t t_last = (args.q_offset + args.Lq - 1) / args.qt;
    const int64_t tiles = t_last - t_first + 1;
    if (tiles > 0x7fffffff || args.Hkv > 65535 || args.B > 65535) return BI_ERR_UNSUPPORTED;
    dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(args.Hkv),
              static_cast<unsigned>(args.B));
    sdpa_kernel<T, ARR, DP, C><<<grid, S2_THREADS, S2Smem<DP, C>::BYTES, s>>>(tq, tk, tv, args);
    count_launch();
    return cuda_status(cudaGetLastError());
}

template <typename T, int DP, int C>
bi_status s2_mask(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                  const SdpaArgs &args, cudaStream_t s) {
    return args.mode == 2 ? s2_launch<T, true, DP, C>(tq, tk, tv, args, s)
                          : s2_launch<T, false, DP, C>(tq, tk, tv, args, s);
}

template <typename T>
bi_status s2_shape(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                   const SdpaArgs &args, cudaStream_t s) {
    if (args.dp == 256 && args.chunk == 64) return s2_mask<T, 256, 64>(tq, tk, tv, args, s);
    if (args.dp == 128 && args.chunk == 128) return s2_mask<T, 128, 128>(tq, tk, tv, args, s);
    if (args.dp == 64 && args.chunk == 128) return s2_mask<T, 64, 128>(tq, tk, tv, args, s);
    return BI_ERR_UNSUPPORTED;
}

template <typename T>
bi_status s2_attrs() {
    bi_status (*const fns[])() = {
        s2_attr<T, false, 256, 64>, s2_attr<T, true, 256, 64>, s2_attr<T, false, 128, 128>,
        s2_attr<T, true, 128, 128>, s2_attr<T, false, 64, 128>, s2_attr<T, true, 64, 128>};
    for (auto f : fns) {
        const bi_status st = f();
        if (st != BI_OK) return st;
    }
    return BI_OK;
}

}  // namespace

bi_status init_sdpa() {
    const bi_status st = s2_attrs<__nv_bfloat16>();
    return st != BI_OK ? st : s2_attrs<__half>();
}

bi_status launch_sdpa(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                      const SdpaArgs &args, bi_dtype dt, cudaStream_t s) {
    if (dt == BI_BF16) return s2_shape<__nv_bfloat16>(tq, tk, tv, args, s);
    if (dt == BI_F16) return s2_shape<__half>(tq, tk, tv, args, s);
    return BI_ERR_UNSUPPORTED;
}

}  // namespace bi
