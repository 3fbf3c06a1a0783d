// Shared device helpers of the ts library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define TS_LOG2E 1.4426950408889634f
#define TS_LN2 0.6931471805599453f

namespace ts {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 16-byte global -> shared async copy (cp.async.cg bypasses L1).
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
// Same, with zero fill when `valid` is false (src-size 0).
__device__ __forceinline__ void cp_async16_zfill(void *smem, const void *gmem, bool valid) {
    uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// 64-bit words per row of a batch mask: uint64 [T][mask_words(T)], at least 2.
__host__ __device__ __forceinline__ int mask_words(int T) { return T > 128 ? (T + 63) / 64 : 2; }

// Row visibility of batch token u for batch row t (mask is uint64 [T][mw]).
__device__ __forceinline__ bool mask_bit(const uint64_t *mask, int mw, int t, int u) {
    return (mask[(size_t)mw * t + (u >> 6)] >> (u & 63)) & 1ull;
}

}  // namespace ts
