// n-gram table of the generated text and top-k 4-gram retrieval (TokenSwift
// tool listing, "How it works": the top-k candidate 4-grams form draft tokens
// and the n-gram table is updated after every step; model card command line:
// --ngram_topk 20, --gamma 4).
//
// Table: open addressing with linear probing over C slots (a power of two);
// a slot holds a 4-gram key (four int32, all ones when empty), its count and
// the start position of its first occurrence.  The home slot is a hash of all
// four tokens, so probe runs stay short whatever the token frequencies.
//
// Update: one thread per new window; a plain read of the slot first, a
// 128-bit compare-and-swap only to claim an empty one; the count goes up with
// an atomic add and the first position with an atomic min.  Probing is
// bounded by C; a full table or a negative id sets the caller's status word
// to TS_ERR_DATA.
//
// Top-k: one CTA scans the sequence for the anchor.  An occurrence starting at
// q contributes its 4-gram only when q is that 4-gram's first occurrence in
// the table, so every distinct 4-gram is taken exactly once, with its count
// from the table.  Candidates (count, tail) gather in shared memory; a bitonic
// sort (count descending, then (w1, w2, w3) ascending) keeps the best k,
// and cuts the buffer to k whenever the next block of the scan might not fit.
#include "internal.h"
#include "ts_common.cuh"

namespace ts {

namespace {
constexpr uint32_t NG_EMPTY = 0xffffffffu;
constexpr int NG_THREADS = 1024;
constexpr int NG_SCAN = 4 * NG_THREADS;     // sequence positions per scan block
constexpr int NG_CAP = NG_SCAN + 1024;      // shared-memory candidates (80 KB): k <= 1024 plus one block

// MurmurHash3's 32-bit finalizer (Appleby): an invertible avalanche mix.
__device__ __forceinline__ uint32_t mix32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x85ebca6bu;
    x ^= x >> 13;
    x *= 0xc2b2ae35u;
    x ^= x >> 16;
    return x;
}
__device__ __forceinline__ uint32_t home_of(int4 w, uint32_t C) {
    uint32_t h = mix32((uint32_t)w.x + 0x9e3779b9u);
    h = mix32(h ^ (uint32_t)w.y);
    h = mix32(h ^ (uint32_t)w.z);
    h = mix32(h ^ (uint32_t)w.w);
    return h & (C - 1u);
}

__device__ __forceinline__ bool same(int4 a, int4 b) { return a.x == b.x && a.y == b.y && a.z == b.z && a.w == b.w; }
__device__ __forceinline__ bool is_empty(int4 a) { return (a.x & a.y & a.z & a.w) == (int)NG_EMPTY; }

// 128-bit compare-and-swap on a global slot (PTX atom.cas.b128, sm_90 and
// later); returns the slot's previous content.
__device__ __forceinline__ int4 cas128(int4 *addr, int4 cmp, int4 val) {
    const uint64_t cl = ((uint64_t)(uint32_t)cmp.y << 32) | (uint32_t)cmp.x;
    const uint64_t ch = ((uint64_t)(uint32_t)cmp.w << 32) | (uint32_t)cmp.z;
    const uint64_t vl = ((uint64_t)(uint32_t)val.y << 32) | (uint32_t)val.x;
    const uint64_t vh = ((uint64_t)(uint32_t)val.w << 32) | (uint32_t)val.z;
    uint64_t ol, oh;
    asm volatile(
        "{\n\t.reg .b128 c, v, o;\n\t"
        "mov.b128 c, {%2, %3};\n\t"
        "mov.b128 v, {%4, %5};\n\t"
        "atom.relaxed.gpu.global.cas.b128 o, [%6], c, v;\n\t"
        "mov.b128 {%0, %1}, o;\n\t}"
        : "=l"(ol), "=l"(oh)
        : "l"(cl), "l"(ch), "l"(vl), "l"(vh), "l"(addr)
        : "memory");
    return make_int4((int)(uint32_t)ol, (int)(uint32_t)(ol >> 32), (int)(uint32_t)oh, (int)(uint32_t)(oh >> 32));
}

// Candidate order: larger count first, then the tail (w1, w2, w3) ascending.
// x = count, y z w = tail; an entry with count < 0 is padding (worst).
__device__ __forceinline__ bool before(int4 a, int4 b) {
    if (a.x != b.x) return a.x > b.x;
    if (a.y != b.y) return a.y < b.y;
    if (a.z != b.z) return a.z < b.z;
    return a.w < b.w;
}

// Sort cand[0, n) into `before` order and keep the first min(n, k); returns
// the new count.  Bitonic network over the next power of two (padding worst).
// Every thread of the CTA calls it with the same n.
__device__ int sort_and_cut(int4 *cand, int n, int k) {
    int P = 1;
    while (P < n) P <<= 1;
    for (int i = n + threadIdx.x; i < P; i += blockDim.x) cand[i] = make_int4(-1, 0, 0, 0);
    __syncthreads();
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < (P >> 1); i += blockDim.x) {
                const int lo = 2 * stride * (i / stride) + (i % stride), hi = lo + stride;
                const bool up = (lo & size) == 0;  // this run ends up in `before` order
                const int4 a = cand[lo], b = cand[hi];
                if (up ? before(b, a) : before(a, b)) {
                    cand[lo] = b;
                    cand[hi] = a;
                }
            }
            __syncthreads();
        }
    }
    return n < k ? n : k;
}
}  // namespace

__global__ void __launch_bounds__(256) ngram_reset_kernel(int4 *keys, int32_t *counts, int32_t *first, uint32_t C) {
    for (uint32_t i = blockIdx.x * 256 + threadIdx.x; i < C; i += gridDim.x * 256) {
        keys[i] = make_int4(-1, -1, -1, -1);
        counts[i] = 0;
        first[i] = 0x7fffffff;
    }
}

__global__ void __launch_bounds__(256) ngram_update_kernel(int4 *keys, int32_t *counts, int32_t *first, uint32_t C,
                                                           const int32_t *__restrict__ seq, int64_t p0, int64_t p1,
                                                           int32_t *status) {
    const int4 empty = make_int4(-1, -1, -1, -1);
    for (int64_t p = p0 + blockIdx.x * 256 + threadIdx.x; p < p1; p += (int64_t)gridDim.x * 256) {
        const int4 w = make_int4(seq[p - 3], seq[p - 2], seq[p - 1], seq[p]);
        if (w.x < 0 || w.y < 0 || w.z < 0 || w.w < 0) {
            atomicExch(status, (int)TS_ERR_DATA);
            continue;
        }
        uint32_t s = home_of(w, C);
        bool placed = false;
        for (uint32_t probe = 0; probe < C && !placed; ++probe, s = (s + 1u) & (C - 1u)) {
            int4 cur = __ldcg(&keys[s]);  // L2-coherent read
            if (is_empty(cur)) cur = cas128(&keys[s], empty, w);  // claim it (or see who did)
            if (is_empty(cur) || same(cur, w)) {
                atomicAdd(&counts[s], 1);
                atomicMin(&first[s], (int)(p - 3));
                placed = true;
            }
        }
        if (!placed) atomicExch(status, (int)TS_ERR_DATA);  // table full
    }
}

__global__ void __launch_bounds__(NG_THREADS) ngram_topk_kernel(const int4 *__restrict__ keys,
                                                                const int32_t *__restrict__ counts,
                                                                const int32_t *__restrict__ first, uint32_t C,
                                                                const int32_t *__restrict__ seq, int64_t n,
                                                                const int32_t *anchor_p, int k, int32_t *chains,
                                                                int32_t *out_counts, int32_t *found) {
    extern __shared__ int4 cand[];  // [NG_CAP]
    __shared__ int s_n;
    const int tid = threadIdx.x;
    const int32_t a = *anchor_p;
    int nc = 0;
    if (a >= 0 && n >= 4) {
        const int64_t last = n - 4;  // last start position of a 4-gram
        for (int64_t base = 0; base <= last; base += NG_SCAN) {
            if (nc + NG_SCAN > NG_CAP) nc = sort_and_cut(cand, nc, k);
            __syncthreads();  // the previous block's reads of s_n are done
            if (tid == 0) s_n = nc;
            int32_t tok[NG_SCAN / NG_THREADS];
#pragma unroll
            for (int j = 0; j < NG_SCAN / NG_THREADS; ++j) {
                const int64_t q = base + tid + (int64_t)j * NG_THREADS;
                tok[j] = q <= last ? seq[q] : -1;
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < NG_SCAN / NG_THREADS; ++j) {
                if (tok[j] != a) continue;
                const int64_t q = base + tid + (int64_t)j * NG_THREADS;
                const int4 w = make_int4(a, seq[q + 1], seq[q + 2], seq[q + 3]);
                uint32_t s = home_of(w, C);
                for (uint32_t probe = 0; probe < C; ++probe, s = (s + 1u) & (C - 1u)) {
                    const int4 cur = keys[s];
                    if (is_empty(cur)) break;  // not in the table
                    if (same(cur, w)) {
                        if (first[s] == (int)q) cand[atomicAdd(&s_n, 1)] = make_int4(counts[s], w.y, w.z, w.w);
                        break;
                    }
                }
            }
            __syncthreads();
            nc = s_n;
        }
        nc = sort_and_cut(cand, nc, k);
    }
    for (int i = tid; i < k; i += NG_THREADS) {
        if (i < nc) {
            const int4 c = cand[i];
            chains[4 * i] = a;
            chains[4 * i + 1] = c.y;
            chains[4 * i + 2] = c.z;
            chains[4 * i + 3] = c.w;
            out_counts[i] = c.x;
        } else {
            chains[4 * i] = chains[4 * i + 1] = chains[4 * i + 2] = chains[4 * i + 3] = -1;
            out_counts[i] = 0;
        }
    }
    if (tid == 0) *found = nc;
}

namespace {
struct TableView {
    int4 *keys;
    int32_t *counts, *first;
};
TableView view_of(void *table, uint32_t C) {
    int4 *keys = static_cast<int4 *>(table);
    int32_t *counts = reinterpret_cast<int32_t *>(keys + C);
    return {keys, counts, counts + C};
}
}  // namespace

cudaError_t launch_ngram_reset(void *table, uint32_t C, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    const TableView t = view_of(table, C);
    const uint32_t blocks = (C + 255) / 256 < 4096 ? (C + 255) / 256 : 4096;
    ngram_reset_kernel<<<blocks, 256, 0, st>>>(t.keys, t.counts, t.first, C);
    return cudaGetLastError();
}

cudaError_t launch_ngram_update(void *table, uint32_t C, const int32_t *seq, int64_t n_old, int64_t n_new,
                                int32_t *status, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    const int64_t p0 = n_old > 3 ? n_old : 3;
    if (n_new <= p0) return cudaSuccess;
    const TableView t = view_of(table, C);
    const int64_t blocks = (n_new - p0 + 255) / 256 < 4096 ? (n_new - p0 + 255) / 256 : 4096;
    ngram_update_kernel<<<(unsigned)blocks, 256, 0, st>>>(t.keys, t.counts, t.first, C, seq, p0, n_new, status);
    return cudaGetLastError();
}

cudaError_t launch_ngram_topk(const void *table, uint32_t C, const int32_t *seq, int64_t n, const int32_t *anchor,
                              int k, int32_t *chains, int32_t *counts, int32_t *found, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    const TableView t = view_of(const_cast<void *>(table), C);
    const size_t smem = sizeof(int4) * NG_CAP;
    cudaError_t e = cudaFuncSetAttribute(ngram_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ngram_topk_kernel<<<1, NG_THREADS, smem, st>>>(t.keys, t.counts, t.first, C, seq, n, anchor, k, chains, counts,
                                                   found);
    return cudaGetLastError();
}

}  // namespace ts
