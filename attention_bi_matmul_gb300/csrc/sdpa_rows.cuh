// sdpa_rows.cuh -- the row warps of the attention kernel (sdpa.cu): the online softmax
// and the output of one 128-row query tile.
//
// "mlx-batch-invariant" README, "How the kernels work" / Attention: one pass over the
// key chunks in order with an online softmax in fp32 (the rule is spelled out at the
// top of sdpa.cu).  The pages' kernel hands a row's keys to several walkers, each with
// its own running sum, and adds those together once at the end in a fixed order; here
// the walkers are two warps, which take the chunks in turn.
//
// Eight row warps (SDPA_ROW_WARP0 ..+7).  Warp w serves TMEM lane quarter w % 4 (32
// rows) and, as group (w - SDPA_ROW_WARP0) / 4, the chunks j with j % 2 == group: all C
// keys of each.  The two warps of a lane quarter share the running shift.  After its
// chunk's maximum a warp publishes the shift it chose (mx_s[j % 2][row]) and arrives at
// a named barrier that the other warp waits at before it chooses the next one, so the
// shifts follow the chunks in order while the two warps' exponentials overlap.  Each
// warp keeps the sum of its own chunks (rescaled at every shift change); the two sums
// meet once after the last chunk (ls_s[group][row]), group 0's first.
//
// Tensor memory: three S buffers of C columns at 0, C, 2 C, O at 3 C.  A warp writes P
// of chunk j over the S buffer j % 3 it has read out: the keys of each half h of the
// chunk, 2 c and 2 c + 1 (the lower in the low half), in column (C / 2) h + c.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_tc.cuh"  // pack8
#include "internal.cuh"
#include "ptx.cuh"
#include "sdpa_common.cuh"

namespace bi {
namespace {

constexpr int SDPA_ROW_WARP0 = 2;        // first row warp of a block
constexpr float SDPA_LAG = 8.0f;         // how far a row's shift may lag its running maximum (log2)

// Named barriers 5..12: the shift of lane quarter q chosen by group g, 5 + 4 g + q.  The
// choosing warp arrives, the other warp waits; 1..4 (pair_sync) join both at the end.
__device__ __forceinline__ void shift_publish(int grp, uint32_t quarter) {
    asm volatile("bar.arrive %0, 64;" ::"r"(5u + 4u * static_cast<uint32_t>(grp) + quarter) : "memory");
}
__device__ __forceinline__ void shift_receive(int from_grp, uint32_t quarter) {
    asm volatile("bar.sync %0, 64;" ::"r"(5u + 4u * static_cast<uint32_t>(from_grp) + quarter) : "memory");
}

// One row warp's whole share of a query tile: for each of its chunks j, S from
// sfull[j % 3], O rescaled (after P V(j-1), pvdone[(j-1) % 4]), then P_j written and
// published in two halves, arrive_p(j % 3, 0) for keys 0..C/2-1 and arrive_p(j % 3, 1)
// for the rest; the output read once every MMA is done (mma_done, one phase).
// p_lo: absolute position of the tile's first query row.
//
// S(j) is issued only after P V(j-3) is done, so at chunk j pvdone[(j-1) % 4]'s phase
// before P V(j-1)'s (P V(j-5)) is complete and a parity wait on it cannot pass early.
// The same bound keeps a warp from arriving for chunk j + 3 on pfull[j % 3] before
// chunk j's four arrivals are in: it waits for S(j + 3) first.
template <typename T, bool ARR, int DP, int C, typename ArriveP>
__device__ __forceinline__ void sdpa_rows(const SdpaArgs &args, int warp, int lane, uint32_t tmem_base,
                                          int64_t p_lo, int kvh, int b, int nchunks, uint64_t *sfull,
                                          uint64_t *pvdone, uint64_t *mma_done, float *mx_s,
                                          float *ls_s, volatile int *abort_flag, ArriveP arrive_p) {
    constexpr uint32_t O_COL = 3 * C;
    constexpr int NH = C / 64;           // 64-key halves of a chunk held in registers at once
    constexpr int PH = C / 2;            // P columns of a 32-key block k0: PH (k0 / PH) + (k0 % PH) / 2
    constexpr int HD = DP / 2;           // output columns per warp at the read-out
    static_assert(C == 128 || C == 64, "chunks of 64 or 128 keys");
    const int G = args.group;
    const int64_t q_offset = args.q_offset;
    const int64_t Lq = args.Lq, Lkv = args.Lkv;
    const uint32_t quarter = static_cast<uint32_t>(warp & 3);
    const int grp = (warp - SDPA_ROW_WARP0) >> 2;    // chunks j with j % 2 == grp; output columns HD grp..
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
    float m_run = -INFINITY, l_own = 0.0f;
    if (args.sinks) {
        m_run = __fmul_rn(args.sinks[h], 1.44269504088896341f);
        l_own = grp == 0 ? 1.0f : 0.0f;          // the sink's own term, counted once
    }
    // The other warp's choice for chunk jp: its shift, and l_own rescaled by the factor
    // that warp applied (same operands, same instruction).
    auto receive = [&](int jp) {
        shift_receive(grp ^ 1, quarter);
        const float m_new = mx_s[(jp & 1) * 128 + r];
        if (m_new != m_run) {
            l_own = __fmul_rn(l_own, ex2_approx(__fsub_rn(m_run, m_new)));
            m_run = m_new;
        }
    };

    for (int j = grp; j < nchunks; j += 2) {
        const uint32_t sb = static_cast<uint32_t>(j % 3);    // S buffer (and P) of chunk j
        const uint32_t sph = static_cast<uint32_t>(j / 3) & 1u;
        const int64_t key0 = static_cast<int64_t>(j) * C;
        uint64_t vis[NH];
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
            vis[hh] = ~0ull;
            if (ARR && mrow) vis[hh] = mask_bits64(mrow + key0 + 64 * hh, Lkv - key0 - 64 * hh);
        }
        int lim = C;
        if (!ARR) {
            const int64_t lim64 = vis_end - key0;
            lim = lim64 < 0 ? 0 : (lim64 > C ? C : static_cast<int>(lim64));
        }
        bool all_vis = ARR ? vis[0] == ~0ull : lim == C;
        if (ARR && NH == 2) all_vis = all_vis && vis[NH - 1] == ~0ull;
        const bool full = __all_sync(0xffffffffu, all_vis) != 0;
        auto visible = [&](int k) {        // key k of the chunk, 0 <= k < C
            return ARR ? ((vis[k >> 6] >> (k & 63)) & 1u) != 0 : k < lim;
        };
        warp_wait(&sfull[sb], sph, abort_flag);
        tc_fence_after();
        const uint32_t s_addr = tmem_base + lane_base + sb * C;
        float x[64];
        uint32_t(&x0)[32] = *reinterpret_cast<uint32_t(*)[32]>(x);
        uint32_t(&x1)[32] = *reinterpret_cast<uint32_t(*)[32]>(x + 32);
        // ---- the chunk's maximum (exact in any order): the upper half first, so that
        // the lower one stays in x
        float mloc = -INFINITY;
        if (warp_valid) {
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int hh = NH - 1; hh >= 0; --hh) {
                tmem_ld32(s_addr + 64 * hh, x0);
                tmem_ld32(s_addr + 64 * hh + 32, x1);
                tmem_wait_ld(x0);
                tmem_tie(x1);
                if (full) {
#pragma unroll
                    for (int i = 0; i < 64; i += 8)
#pragma unroll
                        for (int c = 0; c < 4; ++c) m4[c] = fmax3(m4[c], x[i + 2 * c], x[i + 2 * c + 1]);
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        if (visible(64 * hh + i)) m4[i & 3] = fmaxf(m4[i & 3], x[i]);
                }
            }
            mloc = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        // ---- the shift: chunk j-1's (the other warp's) first, then this chunk's
        if (j >= 1) receive(j - 1);
        const bool any = mloc != -INFINITY;
        const float cand = __fmul_rn(mloc, sl2);
        const bool raise = any && cand > __fadd_rn(m_run, SDPA_LAG);
        const float m_new = raise ? cand : m_run;
        const float alpha = raise ? ex2_approx(__fsub_rn(m_run, m_new)) : 1.0f;
        mx_s[(j & 1) * 128 + r] = m_new;
        shift_publish(grp, quarter);
        // ---- O *= alpha for these 32 rows, after P_{j-1} V_{j-1} is added in (skipped,
        // wait included, when every row has alpha 1), before P V(j) can start
        if (j >= 1 && warp_valid && __any_sync(0xffffffffu, alpha != 1.0f)) {
            warp_wait(&pvdone[(j - 1) % 4], static_cast<uint32_t>((j - 1) / 4) & 1u, abort_flag);
            tc_fence_after();
            const uint32_t o_all = tmem_base + lane_base + O_COL;
#pragma unroll 1
            for (int c4 = 0; c4 < DP / 32; ++c4) {
                uint32_t ov[32];
                tmem_ld32(o_all + c4 * 32, ov);
                tmem_wait_ld(ov);
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    ov[e] = __float_as_uint(__fmul_rn(__uint_as_float(ov[e]), alpha));
                tmem_st32(o_all + c4 * 32, ov);
            }
        }
        // ---- P = 2^(S scale - shift) over the chunk: the lower half of the keys (in x)
        // first, published on its own (part 0) while the upper half is reloaded 32 keys
        // at a time as registers free up, then the upper half (part 1).
        // Partial sum (key mod 4) k of half hh lives in ls01[hh] (k = 0, 1) or ls23[hh]
        // (k = 2, 3) and takes its keys in ascending order.
        float2 ls01[NH], ls23[NH];
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) ls01[hh] = ls23[hh] = make_float2(0.0f, 0.0f);
        auto publish_p = [&](int part) {
            if (warp_valid) tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_p(sb, part);
        };
        {
            const float2 c2 = make_float2(sl2, sl2), nm2 = make_float2(-m_new, -m_new);
            // x[i0..i0+31] holds keys 64 hh + i0.. of the chunk
            auto exp_block = [&](int hh, int i0, bool chk) {
                uint32_t pw[16];
#pragma unroll
                for (int i = i0; i < i0 + 32; i += 2) {
                    const float2 t = __ffma2_rn(make_float2(x[i], x[i + 1]), c2, nm2);
                    float e0 = ex2_approx(t.x), e1 = ex2_approx(t.y);
                    if (chk) {
                        if (!visible(64 * hh + i)) e0 = 0.0f;
                        if (!visible(64 * hh + i + 1)) e1 = 0.0f;
                    }
                    if ((i & 2) == 0) ls01[hh] = __fadd2_rn(ls01[hh], make_float2(e0, e1));
                    else ls23[hh] = __fadd2_rn(ls23[hh], make_float2(e0, e1));
                    pw[(i - i0) / 2] = cvt2<T>(e0, e1);
                }
                const int k0 = 64 * hh + i0;
                tmem_st16(s_addr + PH * (k0 / PH) + (k0 % PH) / 2, pw);
            };
            auto exp_chunk = [&](bool chk) {
                if (NH == 2) {
                    if (warp_valid) {
                        exp_block(0, 0, chk);
                        tmem_ld32(s_addr + 64, x0);
                        exp_block(0, 32, chk);
                        tmem_ld32(s_addr + 96, x1);
                    }
                    publish_p(0);
                    if (warp_valid) {
                        tmem_wait_ld(x0);
                        tmem_tie(x1);
                        exp_block(1, 0, chk);
                        exp_block(1, 32, chk);
                    }
                } else {
                    if (warp_valid) exp_block(0, 0, chk);
                    publish_p(0);
                    if (warp_valid) exp_block(0, 32, chk);
                }
                publish_p(1);
            };
            // Two copies, so that the common (unmasked) one has no test between the
            // exponentials; both do the same arithmetic.
            if (full) exp_chunk(false);
            else exp_chunk(true);
        }
        float lsum = __fadd_rn(__fadd_rn(ls01[0].x, ls01[0].y), __fadd_rn(ls23[0].x, ls23[0].y));
        if (NH == 2)
            lsum = __fadd_rn(lsum, __fadd_rn(__fadd_rn(ls01[NH - 1].x, ls01[NH - 1].y),
                                             __fadd_rn(ls23[NH - 1].x, ls23[NH - 1].y)));
        if (any) {
            l_own = __fadd_rn(__fmul_rn(l_own, alpha), lsum);
            m_run = m_new;
        }
    }
    // the last chunk's shift, if the other warp chose it; then the two sums
    if (nchunks >= 1 && ((nchunks - 1) & 1) != grp) receive(nchunks - 1);
    ls_s[grp * 128 + r] = l_own;
    pair_sync(quarter);
    const float l_run = __fadd_rn(ls_s[r], ls_s[128 + r]);
    // every P V, then o = acc * (1 / l): one correctly rounded reciprocal per row
    warp_wait(mma_done, 0, abort_flag);
    tc_fence_after();
    const float inv_l = __frcp_rn(l_run);
    const uint32_t o_addr = tmem_base + lane_base + O_COL + grp * HD;
    if (warp_valid) {
        T *orow = static_cast<T *>(args.o) + b * args.os[0] + h * args.os[1] +
                  (pos - q_offset) * args.os[2] + grp * HD;
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
                        const int col = grp * HD + c4 * 32 + d8 * 8;
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

}  // namespace
}  // namespace bi
