// Dynamic partial-KV-cache maintenance: chunk importance, top-k selection up
// to the retrieval budget, and the gather into the compact partial cache
// (TokenSwift ICML 2025 summary, "Approach": the drafting pass reads a partial
// KV cache that is refreshed every step from the chunks whose keys score
// highest against the current query; model card: retrieval budget 4096).
#include "internal.h"
#include "topk_radix.cuh"
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
// select_kernel: one CTA per KV head computes sel[g][.] and part_len[g] with
// the radix select of topk_radix.cuh.
// gather_kernel: CTA = (selected chunk, KV head) copies the chunk's K and V
// rows.  The gather is launched as a programmatic dependent of the selection
// so its CTAs are resident and waiting when the selection finishes.
// ---------------------------------------------------------------------------
constexpr int SEL_THREADS = 512;
constexpr int GA_THREADS = 256;

__global__ void __launch_bounds__(SEL_THREADS)
select_kernel(const float *__restrict__ scores, int64_t N, int n_chunks, int k_sel, int n_sink, int n_recent,
              int32_t *__restrict__ sel, int32_t *__restrict__ part_len) {
    extern __shared__ __align__(16) uint32_t keys[];  // [n_chunks]
    __shared__ TopkSmem sm;
    // the gather grid may launch now; it waits for this grid's results
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // this grid is itself a programmatic dependent: the scores are the previous
    // kernel's output
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int g = blockIdx.x;
    int32_t *sel_g = sel + (size_t)g * k_sel;
    const bool last_taken = radix_topk_ascending<SEL_THREADS>(
        scores + (size_t)g * n_chunks, n_chunks, k_sel, n_sink, n_recent, keys, sm,
        [&](int pos, int c) { sel_g[pos] = c; });
    // tokens gathered for this head: only the last chunk of the prefix can be
    // short, and being the largest index it is the last one chosen (the
    // thread whose range holds that chunk knows whether it was chosen)
    const int per = (n_chunks + SEL_THREADS - 1) / SEL_THREADS;
    if (part_len != nullptr && (int)threadIdx.x == (n_chunks - 1) / per) {
        const int64_t tail = N - (int64_t)(n_chunks - 1) * CHUNK;  // tokens of the last chunk, 1..64
        part_len[g] = k_sel * CHUNK - (last_taken ? (int)(CHUNK - tail) : 0);
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
    const size_t smem = sizeof(uint32_t) * (size_t)n_chunks;
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
