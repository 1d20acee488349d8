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
//     memory), one thread per row applies the causal mask (key j visible iff
//     j <= position), m' = max(m, max_j s_j*scale*log2 e),  alpha = 2^(m - m'),
//     p_j = 2^(s_j*scale*log2 e - m'), l = l*alpha + sum_j p_j (sequential j),
//     P rounded to the input dtype, O_chunk = P V (tcgen05.mma), and
//     acc = fma(acc, alpha, O_chunk) in fp32 registers;
//   * a chunk that is entirely masked for a row leaves m, l and acc bit-for-bit
//     unchanged (alpha = 2^0 = 1, p = 0), so extra chunks that a longer query
//     tile visits, or keys appended beyond a token, change none of its bits;
//   * o = acc / l (IEEE division), rounded once to the output dtype.
//
// Roles (448 threads):
//   warp 0 lane 0   TMA producer (Q once; K and V chunks through 2-deep rings)
//   warp 1          TMEM allocation (512 columns); lane 0 issues the MMAs
//   warps 2..5      softmax: one thread per row, S from TMEM, P to shared memory
//   warps 6..13     correction: one thread per (row, half of the head dim), O
//                   chunks from TMEM into the fp32 accumulator, final
//                   normalisation and store
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_tc.cuh"  // to_f32 / from_f32 / IsBf16
#include "internal.cuh"
#include "ptx.cuh"

namespace bi {

namespace {

constexpr int SD_D = 128;       // head dim
constexpr int SD_C = 128;       // keys per chunk
constexpr int SD_ROWS = 128;    // rows per query tile
constexpr int SD_KST = 2;       // K ring depth
constexpr int SD_VST = 2;       // V ring depth
constexpr int SD_THREADS = 448;
constexpr uint32_t SD_PANEL = SD_ROWS * 128;        // 16 KB: 128 rows x 64 elements
constexpr uint32_t SD_TILE = 2 * SD_PANEL;          // 32 KB: 128 rows x 128 elements
constexpr uint32_t SD_TMEM_COLS = 512;              // S0 S1 O0 O1, 128 columns each

struct SdSmem {
    // byte offsets from the 1024-aligned base
    static constexpr uint32_t Q = 0;
    static constexpr uint32_t K = Q + SD_TILE;
    static constexpr uint32_t V = K + SD_KST * SD_TILE;
    static constexpr uint32_t P = V + SD_VST * SD_TILE;
    static constexpr uint32_t ALPHA = P + SD_TILE;              // float[2][128]
    static constexpr uint32_t LFIN = ALPHA + 2 * 128 * 4;        // float[128]
    static constexpr uint32_t BARS = LFIN + 128 * 4;             // uint64 barriers
    static constexpr uint32_t NBARS = 1 + 2 * SD_KST + 2 * SD_VST + 4 + 2 + 4 + 4 + 1 + 1;
    static constexpr uint32_t MISC = BARS + NBARS * 8;           // tmem slot, abort flag
    static constexpr uint32_t END = MISC + 16;
};
constexpr size_t SD_SMEM_BYTES = 1024 + SdSmem::END;

template <typename T>
__global__ void __launch_bounds__(SD_THREADS, 1)
    sdpa_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const SdpaArgs args) {
    constexpr uint32_t IDESC_S = mma_idesc(IsBf16<T>::value, SD_ROWS, SD_C, false);
    constexpr uint32_t IDESC_PV = mma_idesc(IsBf16<T>::value, SD_ROWS, SD_D, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem + SdSmem::Q;
    uint8_t *sK = smem + SdSmem::K;
    uint8_t *sV = smem + SdSmem::V;
    uint8_t *sP = smem + SdSmem::P;
    float *alpha_s = reinterpret_cast<float *>(smem + SdSmem::ALPHA);
    float *lfin_s = reinterpret_cast<float *>(smem + SdSmem::LFIN);
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
    uint64_t *afull = oempty + 2;        // [2]
    uint64_t *aempty = afull + 2;        // [2]
    uint64_t *lfull = aempty + 2;        // [1]
    uint64_t *mma_done = lfull + 1;      // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SdSmem::MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SdSmem::MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int G = args.group;
    const int Qt = args.qt;
    const int64_t q_offset = args.q_offset;
    const int64_t Lq = args.Lq, Lkv = args.Lkv;
    // Query tiles of this call, heaviest (latest positions) first.
    const int64_t t_first = q_offset / Qt;
    const int64_t t_last = (q_offset + Lq - 1) / Qt;
    const int64_t tile = t_last - static_cast<int64_t>(blockIdx.x);
    const int kvh = static_cast<int>(blockIdx.y);
    const int b = static_cast<int>(blockIdx.z);
    const int64_t p_lo = tile * Qt;                         // first position of the tile
    int64_t p_max = p_lo + Qt - 1;                          // last valid position in the tile
    if (p_max > q_offset + Lq - 1) p_max = q_offset + Lq - 1;
    const int nchunks = args.causal ? static_cast<int>(p_max / SD_C + 1)
                                    : static_cast<int>((Lkv + SD_C - 1) / SD_C);
    (void)t_first;

    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < SD_KST; ++s) { mbar_init(&kfull[s], 1); mbar_init(&kempty[s], 1); }
        for (int s = 0; s < SD_VST; ++s) { mbar_init(&vfull[s], 1); mbar_init(&vempty[s], 1); }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&sempty[i], 4);
            mbar_init(&ofull[i], 1);
            mbar_init(&oempty[i], 8);
            mbar_init(&afull[i], 4);
            mbar_init(&aempty[i], 8);
        }
        mbar_init(pfull, 4);
        mbar_init(pempty, 1);
        mbar_init(lfull, 4);
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
            tma_load_4d(sQ, &tmQ, bar_q, 0, kvh * G, qi0, b);
            tma_load_4d(sQ + SD_PANEL, &tmQ, bar_q, 64, kvh * G, qi0, b);
            int armed = 0;
            bool ok = true;
            for (int j = 0; j < nchunks; ++j) {
                const uint32_t sk = j % SD_KST, phk = (j / SD_KST) & 1u;
                if (!mbar_wait(&kempty[sk], phk ^ 1u, abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(&kfull[sk], SD_TILE);
                tma_load_4d(sK + sk * SD_TILE, &tmK, &kfull[sk], 0, j * SD_C, kvh, b);
                tma_load_4d(sK + sk * SD_TILE + SD_PANEL, &tmK, &kfull[sk], 64, j * SD_C, kvh, b);
                const uint32_t sv = j % SD_VST, phv = (j / SD_VST) & 1u;
                if (!mbar_wait(&vempty[sv], phv ^ 1u, abort_flag)) { ok = false; armed = 2 * j + 1; break; }
                mbar_arrive_expect_tx(&vfull[sv], SD_TILE);
                tma_load_4d(sV + sv * SD_TILE, &tmV, &vfull[sv], 0, j * SD_C, kvh, b);
                tma_load_4d(sV + sv * SD_TILE + SD_PANEL, &tmV, &vfull[sv], 64, j * SD_C, kvh, b);
                armed = 2 * j + 2;
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
                    for (int kk = 0; kk < SD_D / 16; ++kk) {
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
                        mma_f16_ss(tmem_base + 256 + ob * 128, smem_desc(p_addr + aoff, 16, 1024),
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
        const uint32_t quarter = static_cast<uint32_t>(warp & 3);
        const int r = static_cast<int>(quarter) * 32 + lane;   // tile row == TMEM lane
        const int qi = r / G, g = r - (r / G) * G;
        const int64_t pos = p_lo + qi;
        const bool valid = pos >= q_offset && pos < q_offset + Lq;
        const bool warp_valid = __any_sync(0xffffffffu, valid) != 0;
        const uint32_t lane_base = (quarter * 32u) << 16;

        if (warp < 6) {
            // ------------------------------------------------ softmax (warps 2..5)
            const float sl2 = args.scale_log2;
            float m_run = -INFINITY, l_run = 0.0f;
            int64_t vis_end = args.causal ? pos + 1 : Lkv;   // keys [0, vis_end) visible
            if (vis_end > Lkv) vis_end = Lkv;
            for (int j = 0; j < nchunks; ++j) {
                const uint32_t sb = j & 1;
                if (!warp_wait(&sfull[sb], (j >> 1) & 1u, abort_flag)) break;
                tc_fence_after();
                int64_t lim64 = valid ? vis_end - static_cast<int64_t>(j) * SD_C : 0;
                const int lim = lim64 < 0 ? 0 : (lim64 > SD_C ? SD_C : static_cast<int>(lim64));
                const uint32_t s_addr = tmem_base + lane_base + sb * 128;
                float alpha = 1.0f;
                float m_new = m_run;
                if (warp_valid) {
                    // pass 1: running maximum of the scaled visible scores, c = 0..127
                    float mloc = -INFINITY;
#pragma unroll 1
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t sr[32];
                        tmem_ld32(s_addr + c4 * 32, sr);
                        tmem_wait_ld(sr);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int c = c4 * 32 + i;
                            const float x = c < lim ? __fmul_rn(__uint_as_float(sr[i]), sl2) : -INFINITY;
                            mloc = fmaxf(mloc, x);
                        }
                    }
                    m_new = fmaxf(m_run, mloc);
                    if (lim > 0) alpha = exp2f(__fsub_rn(m_run, m_new));
                }
                // P_j -> shared memory (K-major, 128-byte swizzle), after PV(j-1) has read P_{j-1}
                if (!warp_wait(pempty, (j & 1u) ^ 1u, abort_flag)) break;
                if (warp_valid) {
                    // pass 2: p = 2^(x - m'), running sum in c order, P rounded to T
                    float lsum = 0.0f;
#pragma unroll 1
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t sr[32];
                        tmem_ld32(s_addr + c4 * 32, sr);
                        tmem_wait_ld(sr);
                        float pv[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int c = c4 * 32 + i;
                            float e = 0.0f;
                            if (c < lim)
                                e = exp2f(__fsub_rn(__fmul_rn(__uint_as_float(sr[i]), sl2), m_new));
                            pv[i] = e;
                            lsum = __fadd_rn(lsum, e);
                        }
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8) {
                            const int cc = (c4 & 1) * 4 + q8;        // 16-byte chunk in the panel
                            const uint4 v = pack8<T>(pv + q8 * 8);
                            uint8_t *dst = sP + (c4 >> 1) * SD_PANEL + r * 128 + ((cc ^ (r & 7)) << 4);
                            *reinterpret_cast<uint4 *>(dst) = v;
                        }
                    }
                    if (lim > 0) {
                        l_run = __fadd_rn(__fmul_rn(l_run, alpha), lsum);
                        m_run = m_new;
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&sempty[sb]);
                    mbar_arrive(pfull);
                }
                // alpha_j -> correction warps
                if (!warp_wait(&aempty[sb], ((j >> 1) & 1u) ^ 1u, abort_flag)) break;
                alpha_s[sb * 128 + r] = alpha;
                __syncwarp();
                if (lane == 0) mbar_arrive(&afull[sb]);
            }
            lfin_s[r] = l_run;
            __syncwarp();
            if (lane == 0) mbar_arrive(lfull);
        } else {
            // ------------------------------------------------ correction (warps 6..13)
            constexpr int HD = SD_D / 2;                    // head-dim columns per thread
            const int col0 = ((warp - 6) >> 2) * HD;        // 0 or 64
            float acc[HD];
#pragma unroll
            for (int d = 0; d < HD; ++d) acc[d] = 0.0f;
            bool ok = true;
            for (int j = 0; j < nchunks; ++j) {
                const uint32_t ob = j & 1;
                if (!warp_wait(&afull[ob], (j >> 1) & 1u, abort_flag)) { ok = false; break; }
                const float alpha = alpha_s[ob * 128 + r];
                __syncwarp();
                if (lane == 0) mbar_arrive(&aempty[ob]);
                if (!warp_wait(&ofull[ob], (j >> 1) & 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                if (warp_valid) {
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tmem_base + lane_base + 256 + ob * 128 + col0 + c * 32, o);
                        tmem_wait_ld(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            acc[c * 32 + i] = __fmaf_rn(acc[c * 32 + i], alpha, __uint_as_float(o[i]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&oempty[ob]);
            }
            if (ok && warp_wait(lfull, 0, abort_flag) && valid) {
                const float l = lfin_s[r];
                const int h = kvh * G + g;
                T *orow = static_cast<T *>(args.o) + b * args.os[0] + h * args.os[1] +
                          (pos - q_offset) * args.os[2] + col0;
#pragma unroll
                for (int d8 = 0; d8 < HD / 8; ++d8) {
                    float v[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = __fdiv_rn(acc[d8 * 8 + i], l);
                    *reinterpret_cast<uint4 *>(orow + d8 * 8) = pack8<T>(v);
                }
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

template <typename T>
bi_status launch_sdpa_typed(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const SdpaArgs &args, cudaStream_t s) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_set[dev & 63]) {
        cudaError_t e = cudaFuncSetAttribute(sdpa_kernel<T>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(SD_SMEM_BYTES));
        if (e != cudaSuccess) return cuda_status(e);
        attr_set[dev & 63] = true;
    }
    const int64_t t_first = args.q_offset / args.qt;
    const int64_t t_last = (args.q_offset + args.Lq - 1) / args.qt;
    const int64_t tiles = t_last - t_first + 1;
    if (tiles > 0x7fffffff || args.Hkv > 65535 || args.B > 65535) return BI_ERR_UNSUPPORTED;
    dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(args.Hkv),
              static_cast<unsigned>(args.B));
    sdpa_kernel<T><<<grid, SD_THREADS, SD_SMEM_BYTES, s>>>(tq, tk, tv, args);
    count_launch();
    return cuda_status(cudaGetLastError());
}

}  // namespace

bi_status launch_sdpa(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                      const SdpaArgs &args, bi_dtype dt, cudaStream_t s) {
    if (dt == BI_BF16) return launch_sdpa_typed<__nv_bfloat16>(tq, tk, tv, args, s);
    if (dt == BI_F16) return launch_sdpa_typed<__half>(tq, tk, tv, args, s);
    return BI_ERR_UNSUPPORTED;
}

}  // namespace bi
