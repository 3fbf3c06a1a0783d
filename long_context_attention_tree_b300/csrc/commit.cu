// Commit of the accepted path into the full KV cache: the kept draft tokens
// become the continuation of the sequence ("How it works" on the TokenSwift
// tool listing: the longest valid draft is kept and generation goes on from
// it).  The accepted batch rows move to the front of the batch region,
//     cache[g][N + i] = cache[g][N + path[i]],  i < L,
// for K and V of every KV head.  L and path come from the verification call
// on the device, so no host round trip sits between verify and commit.
//
// CTA = (KV head, K or V).  A destination row can be the source of a later
// path entry (path = 0, 2, 3 moves row 2 to slot 1 and row 3 to slot 2), so
// the CTA first stages the L source rows in shared memory and only then
// writes them back.
#include "internal.h"
#include "ts_common.cuh"

namespace ts {

namespace {
constexpr int CM_THREADS = 256;
constexpr int CM_ROUND = 128;  // path rows staged in shared memory at a time
}  // namespace

// Rows are moved in rounds of CM_ROUND path entries, each round read in full
// before it is written.  A round never overwrites a later round's source: the
// path is strictly increasing from >= 0, so entry j reads row path[j] >= j,
// while the rounds before it write rows i < j.
__global__ void __launch_bounds__(CM_THREADS) commit_path_kernel(__nv_bfloat16 *k, __nv_bfloat16 *v, int64_t ld_kv,
                                                                 int64_t N, int T, int d, int32_t *result,
                                                                 const int32_t *path) {
    extern __shared__ __align__(16) uint4 rows[];  // [CM_ROUND][d / 8]
    __shared__ int32_t s_path[TS_MAX_T];
    __shared__ int s_L, s_ok;
    const int g = blockIdx.x, tid = threadIdx.x;
    __nv_bfloat16 *base = (blockIdx.y == 0 ? k : v) + ((size_t)g * ld_kv + (size_t)N) * d;
    if (tid == 0) {
        const int L = result[0];
        s_L = L;
        s_ok = (L >= 0 && L <= T) ? 1 : 0;
    }
    __syncthreads();
    const int L = s_ok ? s_L : 0;
    for (int i = tid; i < L; i += CM_THREADS) {
        const int p = path[i];
        s_path[i] = p;
        // rows root..best of a topologically ordered forest: strictly increasing, inside the batch
        const bool bad = p < 0 || p >= T || (i > 0 && path[i - 1] >= p);
        if (bad) atomicAnd(&s_ok, 0);
    }
    __syncthreads();
    if (!s_ok) {
        if (g == 0 && blockIdx.y == 0 && tid == 0) result[3] = (int32_t)TS_ERR_DATA;
        return;
    }
    const int U = d / 8;  // 16-byte units per row
    for (int r0 = 0; r0 < L; r0 += CM_ROUND) {
        const int nr = L - r0 < CM_ROUND ? L - r0 : CM_ROUND;
        for (int e = tid; e < nr * U; e += CM_THREADS) {
            const int i = e / U, u = e % U;
            rows[e] = reinterpret_cast<const uint4 *>(base + (size_t)s_path[r0 + i] * d)[u];
        }
        __syncthreads();
        for (int e = tid; e < nr * U; e += CM_THREADS) {
            const int i = e / U, u = e % U;
            reinterpret_cast<uint4 *>(base + (size_t)(r0 + i) * d)[u] = rows[e];
        }
        __syncthreads();
    }
}

cudaError_t launch_commit_path(__nv_bfloat16 *k, __nv_bfloat16 *v, int64_t ld_kv, int64_t N, int T, int Hkv, int d,
                               int32_t *result, const int32_t *path, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    const size_t smem = (size_t)(T < CM_ROUND ? T : CM_ROUND) * d * 2;  // rows staged per round
    cudaError_t e = cudaFuncSetAttribute(commit_path_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    commit_path_kernel<<<dim3(Hkv, 2), CM_THREADS, smem, st>>>(k, v, ld_kv, N, T, d, result, path);
    return cudaGetLastError();
}

}  // namespace ts
