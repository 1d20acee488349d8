// sdpa.cu -- batch-invariant causal GQA attention on the 5th-generation tensor cores.
//
// "mlx-batch-invariant" README, "How the kernels work" / Attention: a single
// pass over the keys in a fixed order with an online softmax in fp32, no
// split over the keys, no second pass, no route switching; and "Why MLX is not
// invariant" / Attention: the answer for a token must not change with the
// query length (decode vs chunked prefill), the GQA factor times query length,
// or with keys appended to the cache.  The GB300 form of that rule:
//
//   * one block per (query tile, kv head, batch).  A query tile holds 128 rows:
//     Qt = 128 / G absolute positions [t*Qt, t*Qt+Qt) times the G = H/Hkv query
//     heads that share the kv head, row = (position mod Qt) * G + head.  A token
//     therefore sits in the same row of the same tile for every query length;
//   * keys are visited in chunks of 128 at absolute key positions 0,128,256,...
//     in ascending order.  For each chunk: S = Q K^T (tcgen05.mma into tensor
//     memory); the causal mask (key j visible iff j <= position);
//     m' = max(m, (max of the visible s_j) * c) with c = scale * log2 e;
//     alpha = 2^(m - m');  p_j = 2^(fma(s_j, c, -m'));  l = l * alpha + (half
//     sum over keys 0..63 + half sum over keys 64..127), each half summed as
//     four interleaved partial sums (key mod 4) added as (0+1)+(2+3);  P rounded
//     to the input dtype;  O_chunk = P V (tcgen05.mma);  acc = fma(acc, alpha,
//     O_chunk) in fp32 registers.  2^x is the hardware's ex2.approx.ftz.f32;
//   * a chunk that is entirely masked for a row leaves m, l and acc bit-for-bit
//     unchanged (alpha = 1, p = 0), so extra chunks that a longer query tile
//     visits, or keys appended beyond a token, change none of its bits;
//   * o = acc / l (IEEE division), rounded once to the output dtype;
//   * masks: causal (key j visible iff j <= position), none, or a boolean array
//     mask per (batch, head, query, key); an attention sink (one extra logit
//     per head, no value) enters as the initial state m = sink * log2 e, l = 1.
// Every quantity of a row depends only on that row's query, the keys/values,
// the chunk positions and the row's absolute position -- never on which other
// rows share the tile.
//
// Roles (320 threads):
//   warp 0 lane 0   TMA producer (Q once; K and V chunks through 2-deep rings,
//                   plus L2 prefetch of the next chunks)
//   warp 1          TMEM allocation (512 columns); lane 0 issues the MMAs
//   warps 2..9      row warps: warp w serves tile rows 32*(w%4)..+31 (its TMEM
//                   lane quarter) and key/head-dim half (w-2)/4: softmax of its
//                   64 score columns, P for that half, and the fp32
//                   accumulator of its 64 output columns.  The two warps of a
//                   row exchange the chunk maximum and the half sums through
//                   shared memory (named barrier per lane quarter).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_tc.cuh"  // to_f32 / from_f32 / IsBf16 / pack8
#include "internal.cuh"
#include "ptx.cuh"
#include "sdpa_common.cuh"

namespace bi {

namespace {

constexpr int SD_C = 128;       // keys per chunk
constexpr int SD_ROWS = 128;    // rows per query tile
constexpr int SD_KST = 2;       // K ring depth
constexpr int SD_VST = 2;       // V ring depth
constexpr int SD_PF = 2;        // chunks prefetched into L2 beyond the rings
constexpr int SD_THREADS = 320;
constexpr uint32_t SD_PANEL = SD_ROWS * 128;        // 16 KB: 128 rows x 64 elements
constexpr uint32_t SD_PTILE = 2 * SD_PANEL;         // P: 128 rows x 128 keys
constexpr uint32_t SD_TMEM_COLS = 512;              // S0 S1 (128 columns each), O0 O1 (DP each)

// DP: the head dim padded to whole 64-element panels (64 or 128).  Head dims
// that are not a multiple of 64 are loaded with the TMA's zero fill past D, so
// the padded columns add exact zeros to Q K^T and produce O columns that are
// never stored.
template <int DP>
struct SdSmem {
    static constexpr uint32_t NP = DP / 64;                      // panels per Q/K/V tile
    static constexpr uint32_t TILE = NP * SD_PANEL;              // 128 rows x DP elements
    // byte offsets from the 1024-aligned base
    static constexpr uint32_t Q = 0;
    static constexpr uint32_t K = Q + TILE;
    static constexpr uint32_t V = K + SD_KST * TILE;
    static constexpr uint32_t P = V + SD_VST * TILE;
    static constexpr uint32_t MX = P + SD_PTILE;                 // float[2][128] half maxima
    static constexpr uint32_t LS = MX + 2 * 128 * 4;             // float[2][128] half sums
    static constexpr uint32_t BARS = LS + 2 * 128 * 4;           // uint64 barriers
    static constexpr uint32_t NBARS = 1 + 2 * SD_KST + 2 * SD_VST + 4 + 2 + 4 + 1;
    static constexpr uint32_t MISC = BARS + NBARS * 8;           // tmem slot, abort flag
    static constexpr uint32_t END = MISC + 16;
    static constexpr size_t BYTES = 1024 + END;
};

// Registers are granted to warps in groups of four, so a 10-warp block is
// budgeted as 12 warps: at most 168 registers per thread.
// ARR: the boolean array mask form (the causal and unmasked forms need no mask
// bytes and keep their visibility as one bound per row).  DP: padded head dim.
template <typename T, bool ARR, int DP>
__global__ void __launch_bounds__(SD_THREADS, 1)
    sdpa_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const SdpaArgs args) {
    using SdSmem = bi::SdSmem<DP>;
    constexpr uint32_t NP = SdSmem::NP;
    constexpr uint32_t SD_TILE = SdSmem::TILE;
    constexpr int DH = DP / 2;                 // output columns per row warp
    constexpr uint32_t IDESC_S = mma_idesc(IsBf16<T>::value, SD_ROWS, SD_C, false);
    constexpr uint32_t IDESC_PV = mma_idesc(IsBf16<T>::value, SD_ROWS, DP, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem + SdSmem::Q;
    uint8_t *sK = smem + SdSmem::K;
    uint8_t *sV = smem + SdSmem::V;
    uint8_t *sP = smem + SdSmem::P;
    float *mx_s = reinterpret_cast<float *>(smem + SdSmem::MX);
    float *ls_s = reinterpret_cast<float *>(smem + SdSmem::LS);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SdSmem::BARS);
    uint64_t *bar_q = bars;
    uint64_t *kfull = bar_q + 1;
    uint64_t *kempty = kfull + SD_KST;
    uint64_t *vfull = kempty + SD_KST;
    uint64_t *vempty = vfull + SD_VST;
    uint64_t *sfull = vempty + SD_VST;   // [2]
    uint64_t *sempty = sfull + 2;        // [2]
    uint64_t *pfull = sempty + 2;        // [1]
    uint64_t *pempty = pfull + 1;        // [1]
    uint64_t *ofull = pempty + 1;        // [2]
    uint64_t *oempty = ofull + 2;        // [2]
    uint64_t *mma_done = oempty + 2;     // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SdSmem::MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SdSmem::MISC + 4);

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
    const int64_t p_lo = tile * Qt;                         // first position of the tile
    int64_t p_max = p_lo + Qt - 1;                          // last valid position in the tile
    if (p_max > q_offset + Lq - 1) p_max = q_offset + Lq - 1;
    const int nchunks = args.mode == 1 ? static_cast<int>(p_max / SD_C + 1)
                                       : static_cast<int>((Lkv + SD_C - 1) / SD_C);

    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < SD_KST; ++s) { mbar_init(&kfull[s], 1); mbar_init(&kempty[s], 1); }
        for (int s = 0; s < SD_VST; ++s) { mbar_init(&vfull[s], 1); mbar_init(&vempty[s], 1); }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&sempty[i], 8);
            mbar_init(&ofull[i], 1);
            mbar_init(&oempty[i], 8);
        }
        mbar_init(pfull, 8);
        mbar_init(pempty, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, SD_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            const int32_t qi0 = static_cast<int32_t>(p_lo - q_offset);  // may be negative
            mbar_arrive_expect_tx(bar_q, SD_TILE);
#pragma unroll
            for (uint32_t pn = 0; pn < NP; ++pn)
                tma_load_4d(sQ + pn * SD_PANEL, &tmQ, bar_q, 64 * pn, kvh * G, qi0, b);
            for (int j = SD_KST; j < SD_KST + SD_PF && j < nchunks; ++j) {
#pragma unroll
                for (uint32_t pn = 0; pn < NP; ++pn) {
                    tma_prefetch_4d(&tmK, 64 * pn, j * SD_C, kvh, b);
                    tma_prefetch_4d(&tmV, 64 * pn, j * SD_C, kvh, b);
                }
            }
            int armed = 0;
            bool ok = true;
            for (int j = 0; j < nchunks; ++j) {
                const uint32_t sk = j % SD_KST, phk = (j / SD_KST) & 1u;
                if (!mbar_wait(&kempty[sk], phk ^ 1u, abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(&kfull[sk], SD_TILE);
#pragma unroll
                for (uint32_t pn = 0; pn < NP; ++pn)
                    tma_load_4d(sK + sk * SD_TILE + pn * SD_PANEL, &tmK, &kfull[sk], 64 * pn,
                                j * SD_C, kvh, b);
                const uint32_t sv = j % SD_VST, phv = (j / SD_VST) & 1u;
                if (!mbar_wait(&vempty[sv], phv ^ 1u, abort_flag)) { ok = false; armed = 2 * j + 1; break; }
                mbar_arrive_expect_tx(&vfull[sv], SD_TILE);
#pragma unroll
                for (uint32_t pn = 0; pn < NP; ++pn)
                    tma_load_4d(sV + sv * SD_TILE + pn * SD_PANEL, &tmV, &vfull[sv], 64 * pn,
                                j * SD_C, kvh, b);
                armed = 2 * j + 2;
                const int jp = j + SD_KST + SD_PF;   // next chunk not yet asked for
                if (jp < nchunks) {
#pragma unroll
                    for (uint32_t pn = 0; pn < NP; ++pn) {
                        tma_prefetch_4d(&tmK, 64 * pn, jp * SD_C, kvh, b);
                        tma_prefetch_4d(&tmV, 64 * pn, jp * SD_C, kvh, b);
                    }
                }
            }
            if (!ok) {
                // Let every copy already issued land before the block can exit.
                mbar_wait_limited(bar_q, 0, WAIT_LIMIT_NS);
                const int nk = (armed + 1) / 2, nv = armed / 2;
                for (int j = nk - SD_KST < 0 ? 0 : nk - SD_KST; j < nk; ++j)
                    mbar_wait_limited(&kfull[j % SD_KST], (j / SD_KST) & 1u, WAIT_LIMIT_NS);
                for (int j = nv - SD_VST < 0 ? 0 : nv - SD_VST; j < nv; ++j)
                    mbar_wait_limited(&vfull[j % SD_VST], (j / SD_VST) & 1u, WAIT_LIMIT_NS);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            bool ok = mbar_wait(bar_q, 0, abort_flag);
            const uint32_t q_addr = smem_u32(sQ);
            const uint32_t p_addr = smem_u32(sP);
            for (int j = 0; ok && j <= nchunks; ++j) {
                if (j < nchunks) {
                    // S(j) = Q K_j^T into S buffer j&1
                    const uint32_t sk = j % SD_KST;
                    const uint32_t sb = j & 1;
                    if (!mbar_wait(&kfull[sk], (j / SD_KST) & 1u, abort_flag)) { ok = false; break; }
                    if (!mbar_wait(&sempty[sb], ((j >> 1) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t k_addr = smem_u32(sK + sk * SD_TILE);
#pragma unroll
                    for (int kk = 0; kk < DP / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * SD_PANEL + (kk & 3) * 32;
                        mma_f16_ss(tmem_base + sb * 128, smem_desc(q_addr + off, 16, 1024),
                                   smem_desc(k_addr + off, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&kempty[sk]);
                    mma_commit(&sfull[sb]);
                }
                if (j >= 1) {
                    // O(i) = P_i V_i into O buffer i&1, i = j-1
                    const int i = j - 1;
                    const uint32_t sv = i % SD_VST;
                    const uint32_t ob = i & 1;
                    if (!mbar_wait(pfull, i & 1u, abort_flag)) { ok = false; break; }
                    if (!mbar_wait(&vfull[sv], (i / SD_VST) & 1u, abort_flag)) { ok = false; break; }
                    if (!mbar_wait(&oempty[ob], ((i >> 1) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t v_addr = smem_u32(sV + sv * SD_TILE);
#pragma unroll
                    for (int kk = 0; kk < SD_C / 16; ++kk) {
                        const uint32_t aoff = (kk >> 2) * SD_PANEL + (kk & 3) * 32;
                        mma_f16_ss(tmem_base + 256 + ob * DP, smem_desc(p_addr + aoff, 16, 1024),
                                   smem_desc(v_addr + kk * 2048, SD_PANEL, 1024), IDESC_PV,
                                   kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&vempty[sv]);
                    mma_commit(pempty);
                    mma_commit(&ofull[ob]);
                }
            }
            mma_commit(mma_done);
            mbar_wait_limited(mma_done, 0, WAIT_LIMIT_NS);
        }
    } else {
        // ------------------------------------------------ row warps (2..9)
        // These warps never leave the chunk loop early: a failed wait (the CTA is
        // aborting) only turns the remaining work into no-ops, so the two warps of
        // a lane quarter always meet at the same named barriers.
        const uint32_t quarter = static_cast<uint32_t>(warp & 3);
        const int half = (warp - 2) >> 2;  // keys 64*half..+63; output dims DH*half..+DH-1
        const int r = static_cast<int>(quarter) * 32 + lane; // tile row == TMEM lane
        const int qi = r / G, g = r - (r / G) * G;
        const int64_t pos = p_lo + qi;
        const bool valid = pos >= q_offset && pos < q_offset + Lq;
        const bool warp_valid = __any_sync(0xffffffffu, valid) != 0;
        const uint32_t lane_base = (quarter * 32u) << 16;
        const float sl2 = args.scale_log2;
        const int h = kvh * G + g;
        // Causal / no mask: keys [0, vis_end) are visible to this row.  Rows of the
        // tile that hold no query of this call compute as if every key were
        // visible; their results stay in their own rows and are never stored.
        int64_t vis_end = args.mode == 1 ? pos + 1 : Lkv;
        if (vis_end > Lkv) vis_end = Lkv;
        if (!valid) vis_end = INT64_MAX / 2;
        // Array mask: this row's mask bytes.
        const uint8_t *mrow = nullptr;
        if (ARR && valid)
            mrow = args.mask + b * args.ms[0] + h * args.ms[1] + (pos - q_offset) * args.ms[2];

        float acc[DH];
#pragma unroll
        for (int d = 0; d < DH; ++d) acc[d] = 0.0f;
        // A sink enters as the running state before the first key: m = sink * log2 e,
        // l = 2^(m - m) = 1, acc = 0.
        float m_run = -INFINITY, l_run = 0.0f, alpha_prev = 1.0f;
        if (args.sinks) {
            m_run = __fmul_rn(args.sinks[h], 1.44269504088896341f);
            l_run = 1.0f;
        }

        for (int j = 0; j <= nchunks; ++j) {
            float alpha = 1.0f;
            if (j < nchunks) {
                // ---------------- softmax of chunk j over this half's 64 keys
                const uint32_t sb = j & 1;
                // Visibility of this half's 64 keys key0 + i: bit i of `vis` (array
                // mask; read before the wait to hide its latency), else i < lim.
                const int64_t key0 = static_cast<int64_t>(j) * SD_C + half * 64;
                uint64_t vis = ~0ull;
                if (ARR && mrow) vis = mask_bits64(mrow + key0, Lkv - key0);
                warp_wait(&sfull[sb], (j >> 1) & 1u, abort_flag);
                tc_fence_after();
                int lim = 64;
                if (!ARR) {
                    const int64_t lim64 = vis_end - key0;
                    lim = lim64 < 0 ? 0 : (lim64 > 64 ? 64 : static_cast<int>(lim64));
                }
                const bool full =
                    __all_sync(0xffffffffu, ARR ? vis == ~0ull : lim == 64) != 0;
                float x[64];
                float mloc = -INFINITY;
                if (warp_valid) {
                    uint32_t(&x0)[32] = *reinterpret_cast<uint32_t(*)[32]>(x);
                    uint32_t(&x1)[32] = *reinterpret_cast<uint32_t(*)[32]>(x + 32);
                    const uint32_t s_addr = tmem_base + lane_base + sb * 128 + half * 64;
                    tmem_ld32(s_addr, x0);
                    tmem_ld32(s_addr + 32, x1);
                    tmem_wait_ld(x0);
                    tmem_wait_ld(x1);
                    // Raw-score maximum of the visible keys; scaling by sl2 > 0 after the
                    // maximum gives exactly the maximum of the scaled scores.
                    if (full) {
#pragma unroll
                        for (int i = 0; i < 64; ++i) mloc = fmaxf(mloc, x[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            if (ARR ? ((vis >> i) & 1ull) != 0 : i < lim) mloc = fmaxf(mloc, x[i]);
                    }
                }
                // S(j) is in registers: release its TMEM buffer for S(j+2).
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sempty[sb]);
                mx_s[half * 128 + r] = mloc;
                pair_sync(quarter);
                const float mraw = fmaxf(mx_s[r], mx_s[128 + r]);
                const bool any = mraw != -INFINITY;                 // some key of the chunk visible
                const float m_new = any ? fmaxf(m_run, __fmul_rn(mraw, sl2)) : m_run;
                if (any) alpha = ex2_approx(__fsub_rn(m_run, m_new));
                // p = 2^(s * sl2 - m') for the visible keys, 0 for the others
                float ls4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (warp_valid) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        float e = ex2_approx(__fmaf_rn(x[i], sl2, -m_new));
                        if (!full && (ARR ? ((vis >> i) & 1ull) == 0 : i >= lim)) e = 0.0f;
                        x[i] = e;
                        ls4[i & 3] = __fadd_rn(ls4[i & 3], e);
                    }
                }
                const float lsum = __fadd_rn(__fadd_rn(ls4[0], ls4[1]), __fadd_rn(ls4[2], ls4[3]));
                // P_j -> shared memory (panel `half`), once PV(j-1) has read P_{j-1}
                warp_wait(pempty, (j & 1u) ^ 1u, abort_flag);
                if (warp_valid) {
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const uint4 v = pack8x2<T>(x + cc * 8);
                        uint8_t *dst = sP + half * SD_PANEL + r * 128 + ((cc ^ (r & 7)) << 4);
                        *reinterpret_cast<uint4 *>(dst) = v;
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(pfull);
                ls_s[half * 128 + r] = lsum;
                pair_sync(quarter);
                if (any) {
                    l_run = __fadd_rn(__fmul_rn(l_run, alpha), __fadd_rn(ls_s[r], ls_s[128 + r]));
                    m_run = m_new;
                }
            }
            if (j >= 1) {
                // ---------------- accumulate O of chunk j-1 (its alpha was computed last round)
                const int i = j - 1;
                const uint32_t ob = i & 1;
                warp_wait(&ofull[ob], (i >> 1) & 1u, abort_flag);
                tc_fence_after();
                if (warp_valid) {
                    const uint32_t o_addr = tmem_base + lane_base + 256 + ob * DP + half * DH;
                    if constexpr (DH == 64) {
                        uint32_t o0[32], o1[32];
                        tmem_ld32(o_addr, o0);
                        tmem_ld32(o_addr + 32, o1);
                        tmem_wait_ld(o0);
                        tmem_wait_ld(o1);
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            acc[e] = __fmaf_rn(acc[e], alpha_prev, __uint_as_float(o0[e]));
                            acc[32 + e] = __fmaf_rn(acc[32 + e], alpha_prev, __uint_as_float(o1[e]));
                        }
                    } else {
                        uint32_t o0[32];
                        tmem_ld32(o_addr, o0);
                        tmem_wait_ld(o0);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            acc[e] = __fmaf_rn(acc[e], alpha_prev, __uint_as_float(o0[e]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&oempty[ob]);
            }
            alpha_prev = alpha;
        }
        if (valid && !*abort_flag) {
            T *orow = static_cast<T *>(args.o) + b * args.os[0] + h * args.os[1] +
                      (pos - q_offset) * args.os[2] + half * DH;
#pragma unroll
            for (int d8 = 0; d8 < DH / 8; ++d8) {
                if (half * DH + d8 * 8 >= args.D) break;   // padded columns past the head dim
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = __fdiv_rn(acc[d8 * 8 + e], l_run);
                *reinterpret_cast<uint4 *>(orow + d8 * 8) = pack8<T>(v);
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, SD_TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(args.err, ERR_TIMEOUT);
}

template <typename T, bool ARR, int DP>
bi_status launch_sdpa_typed(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const SdpaArgs &args, cudaStream_t s) {
    const int64_t t_first = args.q_offset / args.qt;
    const int64_t t_last = (args.q_offset + args.Lq - 1) / args.qt;
    const int64_t tiles = t_last - t_first + 1;
    if (tiles > 0x7fffffff || args.Hkv > 65535 || args.B > 65535) return BI_ERR_UNSUPPORTED;
    dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(args.Hkv),
              static_cast<unsigned>(args.B));
    sdpa_kernel<T, ARR, DP><<<grid, SD_THREADS, SdSmem<DP>::BYTES, s>>>(tq, tk, tv, args);
    count_launch();
    return cuda_status(cudaGetLastError());
}

}  // namespace

namespace {
template <typename T, bool ARR, int DP>
bi_status set_smem_attr() {
    return cuda_status(cudaFuncSetAttribute(sdpa_kernel<T, ARR, DP>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(SdSmem<DP>::BYTES)));
}
template <typename T, int DP>
bi_status dispatch_mask(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const SdpaArgs &args, cudaStream_t s) {
    return args.mode == 2 ? launch_sdpa_typed<T, true, DP>(tq, tk, tv, args, s)
                          : launch_sdpa_typed<T, false, DP>(tq, tk, tv, args, s);
}
template <typename T>
bi_status dispatch_dp(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                      const SdpaArgs &args, cudaStream_t s) {
    if (args.dp == 64) return dispatch_mask<T, 64>(tq, tk, tv, args, s);
    if (args.dp == 128) return dispatch_mask<T, 128>(tq, tk, tv, args, s);
    return BI_ERR_UNSUPPORTED;
}
}  // namespace

bi_status init_sdpa() {
    bi_status (*const fns[])() = {
        set_smem_attr<__nv_bfloat16, false, 64>, set_smem_attr<__nv_bfloat16, true, 64>,
        set_smem_attr<__nv_bfloat16, false, 128>, set_smem_attr<__nv_bfloat16, true, 128>,
        set_smem_attr<__half, false, 64>,        set_smem_attr<__half, true, 64>,
        set_smem_attr<__half, false, 128>,       set_smem_attr<__half, true, 128>};
    for (auto f : fns) {
        const bi_status st = f();
        if (st != BI_OK) return st;
    }
    return BI_OK;
}

bi_status launch_sdpa(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                      const SdpaArgs &args, bi_dtype dt, cudaStream_t s) {
    if (args.dp == 256) return launch_sdpa256(tq, tk, tv, args, dt, s);
    if (dt == BI_BF16) return dispatch_dp<__nv_bfloat16>(tq, tk, tv, args, s);
    if (dt == BI_F16) return dispatch_dp<__half>(tq, tk, tv, args, s);
    return BI_ERR_UNSUPPORTED;
}

}  // namespace bi
