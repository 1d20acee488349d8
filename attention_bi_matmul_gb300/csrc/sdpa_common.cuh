// sdpa_common.cuh -- small device helpers shared by the attention kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace bi {
namespace {

// max(a, b, c) in one instruction (exact, like two fmaxf).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 8 fp32 -> 8 x 16-bit (16 bytes), converted two at a time (round to nearest even).
template <typename T> __device__ __forceinline__ uint32_t cvt2(float a, float b);
template <> __device__ __forceinline__ uint32_t cvt2<__nv_bfloat16>(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <> __device__ __forceinline__ uint32_t cvt2<__half>(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <typename T>
__device__ __forceinline__ uint4 pack8x2(const float *v) {
    return make_uint4(cvt2<T>(v[0], v[1]), cvt2<T>(v[2], v[3]), cvt2<T>(v[4], v[5]),
                      cvt2<T>(v[6], v[7]));
}

// 64 mask bytes (nonzero = visible) starting at p, of which the first `valid`
// exist (keys past the cache are never visible), as a bit word.
__device__ __forceinline__ uint64_t mask_bits64(const uint8_t *p, int64_t valid) {
    uint64_t bits = 0;
    if (valid >= 64 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 w = reinterpret_cast<const uint4 *>(p)[q];
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                // bytes -> 0/1 per byte -> 4 bits (byte b to bit b)
                const uint32_t ones = __vcmpne4(ws[t], 0u) & 0x01010101u;
                const uint32_t nib = ((ones * 0x01020408u) >> 24) & 0xFu;
                bits |= static_cast<uint64_t>(nib) << (16 * q + 4 * t);
            }
        }
    } else {
        const int n = valid < 0 ? 0 : (valid > 64 ? 64 : static_cast<int>(valid));
        for (int i = 0; i < n; ++i)
            if (p[i]) bits |= 1ull << i;
    }
    return bits;
}

// Named barrier shared by the two row warps of one TMEM lane quarter.
__device__ __forceinline__ void pair_sync(uint32_t quarter) {
    asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
}

__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap *m, int32_t c0, int32_t c1,
                                                int32_t c2, int32_t c3) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

// 32 mask bytes (nonzero = visible) starting at p, of which the first `valid` exist.
__device__ __forceinline__ uint32_t mask_bits32(const uint8_t *p, int64_t valid) {
    uint32_t bits = 0;
    if (valid >= 32 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint4 w = reinterpret_cast<const uint4 *>(p)[q];
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const uint32_t ones = __vcmpne4(ws[t], 0u) & 0x01010101u;
                const uint32_t nib = ((ones * 0x01020408u) >> 24) & 0xFu;
                bits |= nib << (16 * q + 4 * t);
            }
        }
    } else {
        const int n = valid < 0 ? 0 : (valid > 32 ? 32 : static_cast<int>(valid));
        for (int i = 0; i < n; ++i)
            if (p[i]) bits |= 1u << i;
    }
    return bits;
}

}  // namespace
}  // namespace bi
