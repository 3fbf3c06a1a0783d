// Dynamic partial-KV-cache maintenance: chunk importance, top-k selection up
// to the retrieval budget, and the gather into the compact partial cache
// (TokenSwift ICML 2025 summary, "Approach": the drafting pass reads a partial
// KV cache that is refreshed every step from the chunks whose keys score
// highest against the current query; model card: retrieval budget 4096).
#include "internal.h"
#include "ts_common.cuh"

namespace ts {

constexpr int CHUNK = 64;

// ---------------------------------------------------------------------------
// Standalone chunk scoring: score[g][c] = max_{h in g} q_h . sum_{t in c} K[g][t].
// CTA = (CPB consecutive chunks, KV head).  128 threads: 16 lanes x 16 bytes
// cover one 128-dim bf16 row, 8 rows in flight; column sums reduce in smem.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128)
score_chunks_kernel(const __nv_bfloat16 *__restrict__ q_row, const __nv_bfloat16 *__restrict__ k,
                    int64_t ld_kv, int64_t N, int Hq, int G, int n_chunks, int c_begin, int cpb,
                    float *__restrict__ scores, int64_t ld_scores) {
    constexpr int LPR = D / 8;             // 16-byte lanes per row
    constexpr int RIF = 128 / LPR;         // rows in flight
    __shared__ float part[RIF][D];
    __shared__ float ksum[D];
    __shared__ float hmax[32];
    const int g = blockIdx.y;
    const int tid = threadIdx.x;
    const int lane16 = tid % LPR, rr = tid / LPR;
    const __nv_bfloat16 *kh = k + (size_t)g * ld_kv * D;
    for (int cc = 0; cc < cpb; ++cc) {
        const int c = c_begin + blockIdx.x * cpb + cc;
        if (c >= n_chunks) break;
        const int64_t t0 = (int64_t)c * CHUNK;
        const int64_t t1 = (t0 + CHUNK < N) ? t0 + CHUNK : N;
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int64_t t = t0 + rr; t < t1; t += RIF) {
            const uint4 w = *reinterpret_cast<const uint4 *>(kh + (size_t)t * D + lane16 * 8);
            acc[0] += bf16_lo(w.x); acc[1] += bf16_hi(w.x); acc[2] += bf16_lo(w.y); acc[3] += bf16_hi(w.y);
            acc[4] += bf16_lo(w.z); acc[5] += bf16_hi(w.z); acc[6] += bf16_lo(w.w); acc[7] += bf16_hi(w.w);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) part[rr][lane16 * 8 + e] = acc[e];
        __syncthreads();
        for (int e = tid; e < D; e += 128) {
            float s = 0.f;
#pragma unroll
            for (int r = 0; r < RIF; ++r) s += part[r][e];
            ksum[e] = s;
        }
        __syncthreads();
        // one warp per query head of the group (4 warps stride over G <= 32)
        const int warp = tid >> 5, lane = tid & 31;
        for (int j = warp; j < G; j += 4) {
            const __nv_bfloat16 *qh = q_row + (size_t)(g * G + j) * D;
            float dot = 0.f;
            for (int e = lane; e < D; e += 32) dot = fmaf(__bfloat162float(qh[e]), ksum[e], dot);
            dot = warp_sum(dot);
            if (lane == 0) hmax[j] = dot;
        }
        __syncthreads();
        if (tid == 0) {
            float best = hmax[0];
            for (int j = 1; j < G; ++j) best = fmaxf(best, hmax[j]);
            scores[(size_t)g * ld_scores + c] = best;
        }
        __syncthreads();
    }
}

cudaError_t launch_score_chunks(const __nv_bfloat16 *q_row, const __nv_bfloat16 *k, int64_t ld_kv, int64_t N,
                                int Hq, int Hkv, int d, float *scores, int64_t ld_scores, int c_begin,
                                cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    const int nc = (int)((N + CHUNK - 1) / CHUNK);
    if (nc - c_begin <= 0) return cudaSuccess;
    const int cpb = 4;
    dim3 grid((nc - c_begin + cpb - 1) / cpb, Hkv);
    const int G = Hq / Hkv;
    if (d == 128)
        score_chunks_kernel<128><<<grid, 128, 0, st>>>(q_row, k, ld_kv, N, Hq, G, nc, c_begin, cpb, scores,
                                                       ld_scores);
    else
        score_chunks_kernel<64><<<grid, 128, 0, st>>>(q_row, k, ld_kv, N, Hq, G, nc, c_begin, cpb, scores,
                                                      ld_scores);
    return cudaGetLastError();
}

// Scores of the chunks a commit did not touch carry over unchanged.
__global__ void __launch_bounds__(256) copy_scores_kernel(const float *__restrict__ old_s, int nc_old,
                                                          float *__restrict__ new_s, int nc_new, int c_keep) {
    const int g = blockIdx.y;
    for (int c = blockIdx.x * 256 + threadIdx.x; c < c_keep; c += gridDim.x * 256)
        new_s[(size_t)g * nc_new + c] = old_s[(size_t)g * nc_old + c];
}

cudaError_t launch_copy_scores(const float *scores_old, int nc_old, float *scores_new, int nc_new, int c_keep,
                               int Hkv, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    if (c_keep <= 0) return cudaSuccess;
    dim3 grid((c_keep + 255) / 256, Hkv);
    copy_scores_kernel<<<grid, 256, 0, st>>>(scores_old, nc_old, scores_new, nc_new, c_keep);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Top-k selection, then the gather.
// select_kernel: one CTA per KV head computes sel[g][.] and part_len[g] from
// composite keys (order key << 32 | ~chunk index), which are unique and order
// equal scores by lower index.  For k <= 256 every warp keeps a sorted list of
// its best L = 32R keys in registers (R per lane), merging in one batch of L
// keys at a time, and the 32 lists are merged pairwise through shared memory;
// larger k sort all keys in shared memory.
// gather_kernel: CTA = (selected chunk, KV head) copies the chunk's K and V
// rows.  The gather is launched as a programmatic dependent of the selection
// so its CTAs are resident and waiting when the selection finishes.
// ---------------------------------------------------------------------------
constexpr int SEL_THREADS = 1024;
constexpr int SEL_WARPS = SEL_THREADS / 32;
constexpr int GA_THREADS = 256;

__device__ __forceinline__ uint32_t order_key(float x) {
    x = x + 0.0f;  // -0 -> +0 (round-to-nearest), so equal values get equal keys
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The composite key of chunk c: always-kept chunks (the first n_sink, the
// last n_recent) take the largest order key, above every finite score's;
// padding (c >= n_chunks) is 0, below every key.
__device__ __forceinline__ uint64_t chunk_key(const float *sc, int c, int n_chunks, int n_sink, int n_recent) {
    if (c >= n_chunks) return 0ull;
    const uint32_t key = (c < n_sink || c >= n_chunks - n_recent) ? 0xffffffffu : order_key(sc[c]);
    return ((uint64_t)key << 32) | (uint32_t)~(uint32_t)c;
}

// One compare-exchange step of a bitonic network at distance j over a list of
// 32R keys held by one warp, element e = s*32 + lane in v[s].  Runs of length
// k end in descending order where (e & k) == 0 for DESC (ascending otherwise).
template <int R, typename K, bool DESC>
__device__ __forceinline__ void warp_cx(K (&v)[R], int k, int j, int lane) {
    if (j >= 32) {
        const int js = j >> 5;
#pragma unroll
        for (int s = 0; s < R; ++s) {
            if ((s & js) == 0) {
                const int e = s * 32 + lane;
                const bool desc = ((e & k) == 0) == DESC;
                const K a = v[s], b = v[s + js];
                const bool sw = desc ? (a < b) : (a > b);
                v[s] = sw ? b : a;
                v[s + js] = sw ? a : b;
            }
        }
    } else {
        const bool lower = (lane & j) == 0;
#pragma unroll
        for (int s = 0; s < R; ++s) {
            const int e = s * 32 + lane;
            const bool desc = ((e & k) == 0) == DESC;
            const K o = __shfl_xor_sync(0xffffffffu, v[s], j);
            v[s] = (lower == desc) ? (v[s] > o ? v[s] : o) : (v[s] < o ? v[s] : o);
        }
    }
}
template <int R, typename K, bool DESC>
__device__ __forceinline__ void warp_sort(K (&v)[R], int lane) {
#pragma unroll
    for (int k = 2; k <= 32 * R; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) warp_cx<R, K, DESC>(v, k, j, lane);
}
// v (descending) and b (ascending): v <- the 32R largest of both, descending.
// The element-wise maximum of a descending and an ascending list holds the
// largest half of their union as a bitonic sequence, which the half-cleaner
// stages then sort.
template <int R>
__device__ __forceinline__ void warp_merge_top(uint64_t (&v)[R], const uint64_t (&b)[R], int lane) {
#pragma unroll
    for (int s = 0; s < R; ++s) v[s] = v[s] > b[s] ? v[s] : b[s];
#pragma unroll
    for (int j = 16 * R; j > 0; j >>= 1) warp_cx<R, uint64_t, true>(v, 64 * R, j, lane);
}

template <int R>
__device__ void select_topk_warps(const float *sc, int n_chunks, int k_sel, int n_sink, int n_recent,
                                  uint64_t *lists, int32_t *sel_g, int *last_selected) {
    constexpr int L = 32 * R;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_batches = (n_chunks + L - 1) / L;
    uint64_t v[R];
#pragma unroll
    for (int s = 0; s < R; ++s) v[s] = 0ull;
    if (warp < n_batches) {
        // the warp's first batch, sorted descending, is its list
#pragma unroll
        for (int s = 0; s < R; ++s) v[s] = chunk_key(sc, warp * L + s * 32 + lane, n_chunks, n_sink, n_recent);
        warp_sort<R, uint64_t, true>(v, lane);
    }
    for (int bt = warp + SEL_WARPS; bt < n_batches; bt += SEL_WARPS) {
        uint64_t b[R];
#pragma unroll
        for (int s = 0; s < R; ++s) b[s] = chunk_key(sc, bt * L + s * 32 + lane, n_chunks, n_sink, n_recent);
        warp_sort<R, uint64_t, false>(b, lane);
        warp_merge_top<R>(v, b, lane);
    }
    // pairwise merge of the warps' lists: list w takes list w + act, reversed
    int act = 1;
    while (act < n_batches && act < SEL_WARPS) act <<= 1;
    for (act >>= 1; act >= 1; act >>= 1) {
        if (warp >= act && warp < 2 * act) {
#pragma unroll
            for (int s = 0; s < R; ++s) lists[(warp - act) * L + s * 32 + lane] = v[s];
        }
        __syncthreads();
        if (warp < act) {
            uint64_t b[R];
#pragma unroll
            for (int s = 0; s < R; ++s) b[s] = lists[warp * L + (L - 1 - (s * 32 + lane))];
            warp_merge_top<R>(v, b, lane);
        }
        __syncthreads();
    }
    if (warp == 0) {
        // the chosen chunk indices (padding: all ones)
        uint32_t c[R];
#pragma unroll
        for (int s = 0; s < R; ++s) c[s] = (s * 32 + lane < k_sel) ? ~(uint32_t)v[s] : 0xffffffffu;
        bool last = false;
#pragma unroll
        for (int s = 0; s < R; ++s) last |= (int)c[s] == n_chunks - 1;
        // ascending order by rank: the indices are distinct, and the padding
        // (all ones) is above every index, so a chosen index's rank is the
        // number of chosen indices below it
        int rank[R];
#pragma unroll
        for (int s = 0; s < R; ++s) rank[s] = 0;
#pragma unroll
        for (int t = 0; t < R; ++t)
#pragma unroll 8
            for (int src = 0; src < 32; ++src) {
                const uint32_t o = __shfl_sync(0xffffffffu, c[t], src);
#pragma unroll
                for (int s = 0; s < R; ++s) rank[s] += o < c[s] ? 1 : 0;
            }
#pragma unroll
        for (int s = 0; s < R; ++s)
            if (s * 32 + lane < k_sel) sel_g[rank[s]] = (int32_t)c[s];
        const bool any_last = __any_sync(0xffffffffu, last);
        if (lane == 0) *last_selected = any_last ? 1 : 0;
    }
}

// Bitonic sort of v[0, P) (P a power of two, at least 64) into descending
// (DESC) or ascending order by every thread of the CTA.  Stages whose stride
// is below 64 pair elements inside one warp's 64-element window, so only the
// wider stages need a block barrier.
template <typename K, bool DESC>
__device__ void bitonic_sort_block(K *v, int P) {
    const int nthr = blockDim.x;
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const int ls = __ffs(stride) - 1;
            for (int i = threadIdx.x; i < (P >> 1); i += nthr) {
                const int lo = ((i >> ls) << (ls + 1)) + (i & (stride - 1)), hi = lo + stride;
                const bool first = (lo & size) == 0;  // this run ends in the requested order
                const K a = v[lo], b = v[hi];
                if ((first == DESC) ? (a < b) : (a > b)) {
                    v[lo] = b;
                    v[hi] = a;
                }
            }
            if (stride > 32 || (P >> 1) > nthr) __syncthreads(); else __syncwarp();
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(SEL_THREADS)
select_kernel(const float *__restrict__ scores, int64_t N, int n_chunks, int k_sel, int n_sink, int n_recent,
              int32_t *__restrict__ sel, int32_t *__restrict__ part_len) {
    extern __shared__ __align__(16) uint64_t keys[];
    __shared__ int s_last;
    // the gather grid may launch now; it waits for this grid's results
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // this grid is itself a programmatic dependent: the scores are the previous
    // kernel's output
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int g = blockIdx.x, tid = threadIdx.x;
    const float *sc = scores + (size_t)g * n_chunks;
    int32_t *sel_g = sel + (size_t)g * k_sel;
    if (k_sel <= 64) {
        select_topk_warps<2>(sc, n_chunks, k_sel, n_sink, n_recent, keys, sel_g, &s_last);
    } else if (k_sel <= 128) {
        select_topk_warps<4>(sc, n_chunks, k_sel, n_sink, n_recent, keys, sel_g, &s_last);
    } else if (k_sel <= 256) {
        select_topk_warps<8>(sc, n_chunks, k_sel, n_sink, n_recent, keys, sel_g, &s_last);
    } else {
        // all keys sorted descending, then the first k_sel indices ascending
        int P = 64;
        while (P < n_chunks) P <<= 1;
        int PK = 64;
        while (PK < k_sel) PK <<= 1;
        uint32_t *idx = reinterpret_cast<uint32_t *>(keys + P);
        for (int c = tid; c < P; c += SEL_THREADS) keys[c] = chunk_key(sc, c, n_chunks, n_sink, n_recent);
        if (tid == 0) s_last = 0;
        __syncthreads();
        bitonic_sort_block<uint64_t, true>(keys, P);
        for (int i = tid; i < PK; i += SEL_THREADS) {
            uint32_t c = 0xffffffffu;  // padding sorts last
            if (i < k_sel) {
                c = ~(uint32_t)keys[i];
                if ((int)c == n_chunks - 1) s_last = 1;
            }
            idx[i] = c;
        }
        __syncthreads();
        bitonic_sort_block<uint32_t, false>(idx, PK);
        for (int i = tid; i < k_sel; i += SEL_THREADS) sel_g[i] = (int32_t)idx[i];
    }
    __syncthreads();
    // tokens gathered for this head: only the last chunk of the prefix can be
    // short, and being the largest index it is the last one selected
    if (tid == 0 && part_len != nullptr) {
        const int64_t tail = N - (int64_t)(n_chunks - 1) * CHUNK;  // tokens of the last chunk, 1..64
        part_len[g] = k_sel * CHUNK - (s_last ? (int)(CHUNK - tail) : 0);
    }
}

// One selected chunk of one KV head: its K and V rows (rows of the last chunk
// at or past N are neither read nor written), every load issued before the
// first store.
template <int D>
__global__ void __launch_bounds__(GA_THREADS)
gather_kernel(const int32_t *__restrict__ sel, int64_t N, int n_chunks, int k_sel,
              const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v, int64_t ld_kv,
              __nv_bfloat16 *__restrict__ k_part, __nv_bfloat16 *__restrict__ v_part, int64_t ld_part) {
    constexpr int U = D / 8;                     // 16-byte units per row
    constexpr int PER = CHUNK * U / GA_THREADS;  // units per thread per chunk (4 for D = 128)
    static_assert(CHUNK * U % GA_THREADS == 0, "chunk must split evenly over the threads");
    // wait until the selection grid has finished and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the next kernel (a programmatic dependent, e.g. the drafting attention) may launch
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int i = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
    const int c = min(max(sel[(size_t)g * k_sel + i], 0), n_chunks - 1);
    const int64_t left = N - (int64_t)c * CHUNK;
    const int rows = left < CHUNK ? (int)left : CHUNK;
    const __nv_bfloat16 *kh = k + ((size_t)g * ld_kv + (size_t)c * CHUNK) * D;
    const __nv_bfloat16 *vh = v + ((size_t)g * ld_kv + (size_t)c * CHUNK) * D;
    __nv_bfloat16 *kp = k_part + ((size_t)g * ld_part + (size_t)i * CHUNK) * D;
    __nv_bfloat16 *vp = v_part + ((size_t)g * ld_part + (size_t)i * CHUNK) * D;
    uint4 wk[PER], wv[PER];
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        const int e = tid + q * GA_THREADS, r = e / U, u = e % U;
        if (r < rows) {
            wk[q] = *reinterpret_cast<const uint4 *>(kh + (size_t)r * D + u * 8);
            wv[q] = *reinterpret_cast<const uint4 *>(vh + (size_t)r * D + u * 8);
        }
    }
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        const int e = tid + q * GA_THREADS, r = e / U, u = e % U;
        if (r < rows) {
            *reinterpret_cast<uint4 *>(kp + (size_t)r * D + u * 8) = wk[q];
            *reinterpret_cast<uint4 *>(vp + (size_t)r * D + u * 8) = wv[q];
        }
    }
}

cudaError_t launch_select(const float *scores, int Hkv, int64_t N, int n_chunks, int k_sel, int n_sink, int n_recent,
                          int32_t *sel, int32_t *part_len, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    if (k_sel <= 0 || n_chunks <= 0) return cudaSuccess;
    size_t smem;
    if (k_sel <= 256) {
        int R = 2;
        while (32 * R < k_sel) R <<= 1;
        smem = sizeof(uint64_t) * (size_t)(SEL_WARPS / 2) * 32 * R;  // the lists merged in the first round
    } else {
        int P = 64, PK = 64;
        while (P < n_chunks) P <<= 1;
        while (PK < k_sel) PK <<= 1;
        smem = sizeof(uint64_t) * (size_t)P + sizeof(uint32_t) * (size_t)PK;
    }
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // the selection as a programmatic dependent of the kernel that wrote the
    // scores (it waits for that grid before reading them)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(Hkv);
    cfg.blockDim = dim3(SEL_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, select_kernel, scores, N, n_chunks, k_sel, n_sink, n_recent, sel, part_len);
}

cudaError_t launch_gather(const int32_t *sel, int Hkv, int64_t N, int n_chunks, int k_sel,
                          const __nv_bfloat16 *k, const __nv_bfloat16 *v, int64_t ld_kv, int d,
                          __nv_bfloat16 *k_part, __nv_bfloat16 *v_part, int64_t ld_part, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    if (k_sel <= 0 || n_chunks <= 0) return cudaSuccess;
    // the gather as a programmatic dependent of the selection
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(k_sel, Hkv);
    cfg.blockDim = dim3(GA_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (d == 128)
        return cudaLaunchKernelEx(&cfg, gather_kernel<128>, sel, N, n_chunks, k_sel, k, v, ld_kv, k_part, v_part,
                                  ld_part);
    return cudaLaunchKernelEx(&cfg, gather_kernel<64>, sel, N, n_chunks, k_sel, k, v, ld_kv, k_part, v_part, ld_part);
}

}  // namespace ts
