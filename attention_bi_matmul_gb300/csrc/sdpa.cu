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
//     p_j = 2^(fma(s_j, c, -m')); P rounded to the input dtype.  The row sum is
//     kept as two partial sums, one over the even chunks and one over the odd
//     ones, added once at the end (even first): each takes
//     l_e = l_e * alpha + chunk sum at its own chunks and l_e = l_e * alpha at
//     the others; a chunk sum is (sum of keys 0..63 + sum of keys 64..127) for
//     C = 128 and the sum of its 64 keys for C = 64, each such sum taken as four
//     interleaved partial sums (key mod 4) added as (0+1)+(2+3);
//   * P is written into tensor memory, over the chunk's own S columns, and read from
//     there by the P V MMA (its A operand); the output is one fp32 accumulator in
//     tensor memory that the
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
//     initial state m = sink * log2 e and 1 in the even chunks' sum.
// Head dims that are not a multiple of 64 are loaded with the copy engine's zero
// fill past D (they add exact zeros to Q K^T) and the columns past D are never
// stored.  Every quantity of a row depends only on that row's query, the keys and
// values, the chunk positions and the row's absolute position -- never on which
// other rows share the tile.
//
// Roles (384 threads):
//   warp 0 lane 0   K producer (Q and K chunks, the K ring 2 deep)
//   warp 1          TMEM allocation (three S buffers of C columns, O of DP);
//                   lane 0 issues S(t) into buffer t % 3 once K_t has landed and
//                   P V(t-3) is done, so S runs up to three chunks ahead of P V
//   warps 2..9      row warps (sdpa_rows.cuh): warp w serves TMEM lane quarter w % 4
//                   and the chunks j with j % 2 == (w-2)/4, all keys of each; the
//                   two warps of a quarter pass the shift on through a named
//                   barrier per direction, and each writes half of the output
//                   columns (DP/2) at the end
//   warp 10 lane 0  V producer (the V ring 2 deep), apart from K so that a V slot
//                   released late never holds back a K chunk
//   warp 11 lane 0  issues P V(i) once V_i has landed, the MMAs of the lower half of
//                   the keys once the rows have written that half of P_i, the rest
//                   once they have written the upper half
// Measured on B4 H32/8 L4096 D128 causal: one thread issuing both kinds of MMA in
// alternation kept the rows waiting about 0.3 us per chunk for S (the chain
// P_{j-1} -> P V(j-1) -> S(j+1) lay on every chunk's path); with separate S and P V
// threads and three S buffers the call went from 0.528 to 0.477 ms; with the chunks
// taken in turn by the two warps of a quarter (no longer in step with each other) and
// P published in halves, to 0.466 ms (D 64: 0.454 to 0.398 ms).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "gemm_tc.cuh"  // IsBf16 / pack8
#include "internal.cuh"
#include "ptx.cuh"
#include "sdpa_common.cuh"
#include "sdpa_rows.cuh"

namespace bi {

namespace {

constexpr int S2_ROWS = 128;       // rows per query tile
constexpr int S2_KST = 2;          // K ring depth
constexpr int S2_VST = 2;          // V ring depth
// The slot releases are the MMAs' completion barriers: K slot j % 2 is free once S(j-2)
// is done (sfull[(j-2) % 3]), V slot i % 2 once P V(i-2) is (pvdone[(i-2) % 4]).
static_assert(S2_KST == 2 && S2_VST == 2, "ring depth tied to the completion barriers");
constexpr int S2_THREADS = 384;
constexpr int S2_V_WARP = 10;       // the V producer's warp (after the eight row warps)
constexpr int S2_PV_WARP = 11;      // the warp that issues the P V MMAs
constexpr uint32_t S2_QPANEL = S2_ROWS * 128;     // 16 KB: 128 rows x 64 elements

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
    // (the two row sums of a row meet, at the very end, in K slot 0)
    static constexpr uint32_t BARS = MX + 2 * 128 * 4;
    // bar_q kfull[2] vfull[2] sfull[3] pfull[3] phi[3] pvdone[4] mma_done
    static constexpr uint32_t NBARS = 1 + 2 + 2 + 3 + 3 + 3 + 4 + 1;
    static constexpr uint32_t MISC = BARS + NBARS * 8;           // tmem slot, abort flag
    static constexpr uint32_t END = MISC + 16;
    static constexpr size_t BYTES = 1024 + END;
    // tensor memory: S buffers [0, C), [C, 2C), [2C, 3C) -- chunk j's S and then its P
    // (C keys of the input dtype, two to a column, over the first half of each row
    // warp's columns) in buffer j % 3 -- and O [3C, 3C + DP)
    static constexpr uint32_t O_COL = 3 * C;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(O_COL + DP <= TMEM_COLS, "tensor memory");
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
    constexpr uint32_t S2_TMEM_COLS = S2Smem::TMEM_COLS;
    constexpr int S2_C = C;
    constexpr uint32_t IDESC_S = mma_idesc(IsBf16<T>::value, S2_ROWS, C, false);
    constexpr uint32_t IDESC_PV = mma_idesc(IsBf16<T>::value, S2_ROWS, DP, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem + S2Smem::Q;
    uint8_t *sK = smem + S2Smem::K;
    uint8_t *sV = smem + S2Smem::V;
    float *mx_s = reinterpret_cast<float *>(smem + S2Smem::MX);
    // The two warps of a lane quarter add their row sums once, after their last chunk:
    // by then S of the last chunk is done, so no copy or MMA touches K slot 0 any more,
    // and the 1 KB exchange lives there.  One KB less keeps the block in the next smaller
    // shared-memory carve-out (more L1) at head dims 128 and 256: ~1 % at D 256.
    float *ls_s = reinterpret_cast<float *>(sK);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S2Smem::BARS);
    uint64_t *bar_q = bars;
    uint64_t *kfull = bar_q + 1;         // [j & 1]: K_j has landed in K slot j % 2
    uint64_t *vfull = kfull + 2;         // [i & 1]: V_i has landed in V slot i % 2
    // [j % 3]: S(j) done: S buffer j % 3 written, and K slot j % 2 read (the K
    // producer's release too)
    uint64_t *sfull = vfull + 2;
    // [j % 3]: P_j in tensor memory and O rescaled for chunk j (the 8 row warps).  Three
    // barriers: a row warp with no valid rows may run ahead to chunk j + 2 (S(j + 2) is
    // issued once P V(j - 1) is, before the MMA thread waits for P_j) while others still
    // arrive for chunk j, and a shared barrier would then count its arrival towards
    // chunk j.  It cannot get three chunks ahead: S(j + 3) is issued only after P V(j),
    // which waits for P_j's barrier to complete.
    uint64_t *pfull = sfull + 3;
    // [i % 4]: P_i V_i added into O (O readable, V slot i % 2 read, S buffer i % 3 free).
    // Four barriers: S(i+3), which the S thread issues only after P V(i) is done, may
    // let P V(i+1) .. P V(i+2) run while a waiter is still at P V(i)'s phase; with four
    // entries no barrier can move two phases ahead of a wait.
    // [j % 3]: P_j of the chunk's upper half of keys (C/2..C-1) in tensor memory; pfull
    // covers the lower half and the rescale, so that the P V MMAs of the lower half go
    // out while the rows still work on the upper one.  Same argument as for pfull.
    uint64_t *phi = pfull + 3;
    uint64_t *pvdone = phi + 3;
    uint64_t *mma_done = pvdone + 4;    // every P V done (the last, and so every S before it)
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
        for (int i = 0; i < 2; ++i) {
            mbar_init(&kfull[i], 1);
            mbar_init(&vfull[i], 1);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&pvdone[i], 1);
        for (int i = 0; i < 3; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&pfull[i], 4);
            mbar_init(&phi[i], 4);
        }
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
        // Blocks start in about their linear order, one per SM at a time, so the block
        // that runs on an SM about one wave after this one is some %nsmid blocks on.
        // Bringing its Q tile into L2 now (a hint; nothing waits for it) takes its first
        // copy off HBM latency: ~1.3 % on causal prefill.
        {
            uint32_t nsm;
            asm("mov.u32 %0, %%nsmid;" : "=r"(nsm));
            const uint64_t lin = blockIdx.x + static_cast<uint64_t>(gridDim.x) *
                                                  (blockIdx.y + static_cast<uint64_t>(gridDim.y) * blockIdx.z);
            const uint64_t later = lin + nsm;
            if (later < static_cast<uint64_t>(gridDim.x) * gridDim.y * gridDim.z) {
                const uint32_t lx = static_cast<uint32_t>(later % gridDim.x);
                const uint64_t lyz = later / gridDim.x;
                const int32_t ly = static_cast<int32_t>(lyz % gridDim.y);
                const int32_t lz = static_cast<int32_t>(lyz / gridDim.y);
                const int32_t lq0 = static_cast<int32_t>((t_last - lx) * Qt - q_offset);
                if (lq0 >= 0) {
#pragma unroll
                    for (uint32_t pn = 0; pn < NP; ++pn) tma_prefetch_4d(&tmQ, 64 * pn, ly * G, lq0, lz);
                }
            }
        }
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
            // ------------------------------------------------ K producer
            // Q and K_0 were issued during the block's setup.  K_j goes out once S(j-2) is
            // done (K slot j % 2 read); the slot release is the MMA's own completion
            // barrier sfull[(j-2) % 3], which cannot move on to S(j+1) before K_{j+1} is
            // copied.  kfull[j & 1] is armed again only after S(j-2) is done, and the MMA
            // thread waited for K_{j-2}'s phase before issuing it, so no phase is armed
            // before it has been consumed.
            int k_armed = 1;                 // K_0..K_{k_armed-1} issued
            bool ok = true;
            for (int j = 1; j < nchunks; ++j) {
                if (j >= 2 && !mbar_wait(&sfull[(j - 2) % 3], static_cast<uint32_t>((j - 2) / 3) & 1u,
                                         abort_flag)) {
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
            if (!ok) {
                // Let every copy already issued land before the block can exit.
                mbar_wait_limited(bar_q, 0, WAIT_LIMIT_NS);
                for (int k = k_armed - 2 < 0 ? 0 : k_armed - 2; k < k_armed; ++k)
                    mbar_wait_limited(&kfull[k & 1], (k >> 1) & 1u, WAIT_LIMIT_NS);
            }
        }
    } else if (warp == S2_V_WARP) {
        if (lane == 0) {
            // ------------------------------------------------ V producer
            // V_i goes out once P_{i-2} V_{i-2} is done (V slot i % 2 read), on its own
            // thread so that a V slot released late never holds back a K chunk.  Same
            // arming argument as for K, with pvdone and vfull.
            int v_armed = 0;                 // V_0..V_{v_armed-1} issued
            bool ok = true;
            for (int i = 0; i < nchunks; ++i) {
                if (i >= 2 && !mbar_wait(&pvdone[(i - 2) % 4], static_cast<uint32_t>((i - 2) / 4) & 1u,
                                         abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&vfull[i & 1], S2_KV);
#pragma unroll
                for (uint32_t pn = 0; pn < NP; ++pn)
                    tma_load_4d(sV + (i % S2_VST) * S2_KV + pn * S2_KPANEL, &tmV, &vfull[i & 1],
                                64 * pn, i * S2_C, kvh, b);
                v_armed = i + 1;
            }
            if (!ok) {
                for (int k = v_armed - 2 < 0 ? 0 : v_armed - 2; k < v_armed; ++k)
                    mbar_wait_limited(&vfull[k & 1], (k >> 1) & 1u, WAIT_LIMIT_NS);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ S thread
            // S(t) = Q K_t^T into S buffer t % 3 once K_t has landed and P V(t-3), which
            // read P_{t-3} out of that buffer, is done.  S runs up to three chunks ahead of
            // P V, so a chunk's scores are ready long before its rows need them.  Every
            // descriptor is computed once; the MMAs go out with no arithmetic between them.
            constexpr int NS = DP / 16;
            uint64_t qd[NS], kd[2][NS];
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
            }
            auto issue_s = [&](const uint64_t (&kds)[NS], uint32_t s_tmem) {
#pragma unroll
                for (int kk = 0; kk < NS; ++kk) mma_f16_ss(s_tmem, qd[kk], kds[kk], IDESC_S, kk > 0 ? 1u : 0u);
            };
            bool ok = mbar_wait(bar_q, 0, abort_flag);
            for (int t = 0; ok && t < nchunks; ++t) {
                if (!mbar_wait(&kfull[t & 1], (t >> 1) & 1u, abort_flag) ||
                    (t >= 3 && !mbar_wait(&pvdone[(t - 3) % 4], static_cast<uint32_t>((t - 3) / 4) & 1u,
                                          abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sb = static_cast<uint32_t>(t % 3);
                if (t % S2_KST == 0) issue_s(kd[0], tmem_base + sb * S2_C);
                else issue_s(kd[1], tmem_base + sb * S2_C);
                mma_commit(&sfull[sb]);
            }
        }
    } else if (warp == S2_PV_WARP) {
        if (lane == 0) {
            // ------------------------------------------------ P V thread
            // O (+)= P_i V_i once the rows have written P_i (and rescaled O) and V_i has
            // landed.  P from S buffer i % 3: keys 16 kk.. in the columns of row-warp half
            // kk / (HK / 16), 8 per 16 keys; V: MN-major, 64-column atoms.
            constexpr int NV = C / 16, HK = C / 2, KPH = HK / 16;
            uint64_t vd[2][NV];
#pragma unroll
            for (int kk = 0; kk < NV; ++kk)
#pragma unroll
                for (int sl = 0; sl < 2; ++sl)
                    vd[sl][kk] = smem_desc(smem_u32(sV + sl * S2_KV) + kk * 2048, S2_KPANEL, 1024);
            // K = 16 steps kk0..kk1-1 of P_i V_i, in ascending order
            auto issue_pv = [&](const uint64_t (&vds)[NV], uint32_t p_tmem, bool first, int kk0, int kk1) {
#pragma unroll
                for (int kk = 0; kk < NV; ++kk)
                    if (kk >= kk0 && kk < kk1)
                        mma_f16_ts(tmem_base + S2_O_COL, p_tmem + (kk / KPH) * HK + (kk % KPH) * 8, vds[kk],
                                   IDESC_PV, (!first || kk > 0) ? 1u : 0u);
            };
            bool ok = true;
            for (int i = 0; ok && i < nchunks; ++i) {
                if (!mbar_wait(&pfull[i % 3], static_cast<uint32_t>(i / 3) & 1u, abort_flag) ||
                    !mbar_wait(&vfull[i & 1], (i >> 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t p_tmem = tmem_base + static_cast<uint32_t>(i % 3) * S2_C;
                if (i % S2_VST == 0) issue_pv(vd[0], p_tmem, i == 0, 0, NV / 2);
                else issue_pv(vd[1], p_tmem, i == 0, 0, NV / 2);
                if (!mbar_wait(&phi[i % 3], static_cast<uint32_t>(i / 3) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (i % S2_VST == 0) issue_pv(vd[0], p_tmem, i == 0, NV / 2, NV);
                else issue_pv(vd[1], p_tmem, i == 0, NV / 2, NV);
                mma_commit(&pvdone[i % 4]);
            }
            // P V(n-1) follows S(n-1) (its P needs S(n-1)), so this covers every MMA.
            mma_commit(mma_done);
            mbar_wait_limited(mma_done, 0, WAIT_LIMIT_NS);
        }
    } else if (warp >= SDPA_ROW_WARP0 && warp < SDPA_ROW_WARP0 + 8) {
        sdpa_rows<T, ARR, DP, C>(args, warp, lane, tmem_base, p_lo, kvh, b, nchunks, sfull, pvdone,
                                 mma_done, mx_s, ls_s, abort_flag,
                                 [&](uint32_t sb, int part) { mbar_arrive(part == 0 ? &pfull[sb] : &phi[sb]); });
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
