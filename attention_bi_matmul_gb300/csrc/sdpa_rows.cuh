// sdpa_rows.cuh -- the row warps of the attention kernel (sdpa.cu): the online softmax
// and the output of one 128-row query tile.
//
// "mlx-batch-invariant" README, "How the kernels work" / Attention: one pass over the
// key chunks in order with an online softmax in fp32 (the rule is spelled out at the
// top of sdpa.cu).  Eight row warps (SDPA_ROW_WARP0 ..+7): warp w serves TMEM lane
// quarter w % 4 and half (w - SDPA_ROW_WARP0) / 4 of the chunk's keys (C / 2) and of the
// output columns (DP / 2); the two warps of a row exchange the chunk maximum and the
// half sums through shared memory (mx_s, ls_s: float[2][128]) under a named barrier
// per lane quarter.  Tensor memory: three S buffers of C columns at 0, C, 2 C, O at
// 3 C.  A row warp writes its P of chunk j over the first half of its own columns of
// S buffer j % 3, which it has read out already: keys HK h + 2 c and HK h + 2 c + 1 (the
// lower in the low half) in column HK h + c of the buffer, h = the warp's half.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "gemm_tc.cuh"  // pack8
#include "internal.cuh"
#include "ptx.cuh"
#include "sdpa_common.cuh"

namespace bi {
namespace {

constexpr int SDPA_ROW_WARP0 = 2;        // first row warp of a block
constexpr float SDPA_LAG = 8.0f;         // how far a row's shift may lag its running maximum (log2)

// One row warp's whole share of a query tile: chunk j's S from sfull[j % 3], P_j written
// and O rescaled (after P V(j-1), pvdone[(j-1) % 4]) before arrive_p(j % 3), the output
// read once every MMA is done (mma_done, one phase).
// p_lo: absolute position of the tile's first query row.
//
// S(j) is issued only after P V(j-3) is done, so at chunk j pvdone[(j-1) % 4]'s phase
// before P V(j-1)'s (P V(j-5)) is complete and a parity wait on it cannot pass early.
// After the last chunk that holds only up to P V(n-4), hence the separate barrier for
// the read-out.
template <typename T, bool ARR, int DP, int C, typename ArriveP>
__device__ __forceinline__ void sdpa_rows(const SdpaArgs &args, int warp, int lane, uint32_t tmem_base,
                                          int64_t p_lo, int kvh, int b, int nchunks, uint64_t *sfull,
                                          uint64_t *pvdone, uint64_t *mma_done, float *mx_s,
                                          float *ls_s, volatile int *abort_flag, ArriveP arrive_p) {
    constexpr uint32_t O_COL = 3 * C;
    constexpr int HK = C / 2;            // keys per row warp
    constexpr int HD = DP / 2;           // output columns per row warp
    static_assert(HK == 64 || HK == 32, "row warps hold 32 or 64 keys of a chunk");
    const int G = args.group;
    const int64_t q_offset = args.q_offset;
    const int64_t Lq = args.Lq, Lkv = args.Lkv;
    // These warps never leave the chunk loop early, so the two warps of a lane
    // quarter always meet at the same named barriers.
    const uint32_t quarter = static_cast<uint32_t>(warp & 3);
    const int half = (warp - SDPA_ROW_WARP0) >> 2;   // keys HK*half..+HK-1; output columns HD*half..+HD-1
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
    const uint32_t o_addr = tmem_base + lane_base + O_COL + half * HD;

    for (int j = 0; j < nchunks; ++j) {
        const uint32_t sb = static_cast<uint32_t>(j % 3);    // S buffer (and P) of chunk j
        const uint32_t sph = static_cast<uint32_t>(j / 3) & 1u;
        const int64_t key0 = static_cast<int64_t>(j) * C + half * HK;
        using VisT = typename std::conditional<HK == 64, uint64_t, uint32_t>::type;
        VisT vis = ~VisT(0);
        if constexpr (HK == 64) {
            if (ARR && mrow) vis = mask_bits64(mrow + key0, Lkv - key0);
        } else {
            if (ARR && mrow) vis = mask_bits32(mrow + key0, Lkv - key0);
        }
        warp_wait(&sfull[sb], sph, abort_flag);
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
                tmem_ld32(tmem_base + lane_base + sb * C + half * HK + 32 * c32, xu);
            }
            tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(x));
#pragma unroll
            for (int c32 = 1; c32 < HK / 32; ++c32)
                tmem_tie(*reinterpret_cast<uint32_t(*)[32]>(x + 32 * c32));
        }
        if (warp_valid) {
            if (full) {
                // four independent chains (the maximum is exact in any order)
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int i = 0; i < HK; i += 8)
#pragma unroll
                    for (int c = 0; c < 4; ++c) m4[c] = fmax3(m4[c], x[i + 2 * c], x[i + 2 * c + 1]);
                mloc = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
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
        const bool raise = any && cand > __fadd_rn(m_run, SDPA_LAG);
        const float m_new = raise ? cand : m_run;
        const float alpha = raise ? ex2_approx(__fsub_rn(m_run, m_new)) : 1.0f;
        // Keys in pairs with the packed fp32 forms (each lane rounds as the scalar
        // operation does): partial sum (key mod 4) k lives in ls01 (k = 0, 1) or
        // ls23 (k = 2, 3) and is added in ascending key order.
        float2 ls01 = make_float2(0.0f, 0.0f), ls23 = make_float2(0.0f, 0.0f);
        // P_j goes over this warp's columns of S buffer j % 3, already in registers;
        // nothing else reads them before P V(j), and S(j+3), which next writes the
        // buffer, follows P V(j) in the MMA thread's order.  Keys HK*half.. of row r,
        // two to a 32-bit column (lower key in the low half), stored 32 keys at a time
        // so that one store is in flight while the next 32 exponentials are computed.
        if (warp_valid) {
            const float2 c2 = make_float2(sl2, sl2), nm2 = make_float2(-m_new, -m_new);
            // over this warp's own columns of S buffer j % 3, read out above
            const uint32_t p_addr = tmem_base + lane_base + sb * C + half * HK;
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
            warp_wait(&pvdone[(j - 1) % 4], static_cast<uint32_t>((j - 1) / 4) & 1u, abort_flag);
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
        if (lane == 0) arrive_p(sb);
        ls_s[half * 128 + r] = lsum;
        pair_sync(quarter);
        if (any) {
            l_run = __fadd_rn(__fmul_rn(l_run, alpha), __fadd_rn(ls_s[r], ls_s[128 + r]));
            m_run = m_new;
        }
    }
    // every P V, then o = acc * (1 / l): one correctly rounded reciprocal per row
    warp_wait(mma_done, 0, abort_flag);
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

}  // namespace
}  // namespace bi
