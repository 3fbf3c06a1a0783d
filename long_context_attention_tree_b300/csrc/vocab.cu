// Vocabulary side of one TokenSwift verification step: windowed contextual
// penalty, temperature, min-p, greedy target, and exact-match acceptance
// along the draft tree / n-gram paths.
//   model card, "Example using TokenSwift command line": --penalty 1.2
//     --penalty_length 1024 --min_p 0.1 --temperature 1.0;
//   tool listing, "How it works": drafts are accepted when they exactly match
//     the target tokens, and a longest accepted draft is kept.
//
// Row pass: one thread-block cluster of VOCAB_CLUSTER CTAs per batch row; each
// CTA owns a contiguous slice of the vocabulary (76 KB for 152064 ids), which
// one bulk copy (TMA) moves into shared memory while the CTA builds its
// window bitmap.  Pass 1 over shared memory (four logits per 16-byte read)
// writes the penalised logits back, keeps each thread's per-slot maxima in
// registers and gives the slice's maximum; eight remote reads per CTA give
// the row maximum; pass 2 visits only the slots whose maximum reaches the
// min-p threshold (a few per row), counts the kept ids, finds the lowest id
// attaining the row maximum (the greedy target) and draws the Gumbel maximum
// when sampling.  The logits are read from HBM once, by the copy
// engine, with no chain of dependent loads per thread.
#include <cooperative_groups.h>

#include "internal.h"
#include "tc_ptx.cuh"
#include "ts_common.cuh"

namespace cg = cooperative_groups;

namespace ts {

constexpr int VOCAB_CLUSTER = 8;
constexpr int VOCAB_THREADS = 512;
constexpr int VOCAB_MAX_SLICE = 20480;              // V <= 8 * 20480 = 163840 (80 KB of shared memory)
constexpr int VOCAB_BITMAP_WORDS = VOCAB_MAX_SLICE / 32;

struct ArgMax {
    float v;
    int i;
};
__device__ __forceinline__ ArgMax better(ArgMax a, ArgMax b) {
    // larger value wins; equal values: lower index wins; index -1 = empty
    if (a.i < 0) return b;
    if (b.i < 0) return a;
    if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
    return a;
}

// ---- min-p sampling (model card: --min_p 0.1 --temperature 1.0 sample the
// target).  Gumbel-max over the kept set: target = argmax_{l_v >= threshold}
// (l_v + G_v), G_v = -ln(-ln U_v), which draws v with probability
// proportional to exp(l_v) over the kept ids.  U_v comes from Philox4x64-10
// (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
// SC 2011) at counter (v / 4, row, offset, 0) under key (seed, 0), word v % 4:
// U = (2 (x >> 41) + 1) 2^-24, exact in fp32 and inside (0, 1).
__device__ __forceinline__ uint64_t philox_word(uint64_t c0, uint64_t c1, uint64_t c2, uint64_t c3, uint64_t k0,
                                                uint64_t k1, int word) {
    constexpr uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    constexpr uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += W0;
            k1 += W1;
        }
        const uint64_t hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
        const uint64_t hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
        const uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return word == 0 ? c0 : word == 1 ? c1 : word == 2 ? c2 : c3;
}
// Natural logarithm for normal x > 0 as a fixed sequence of IEEE fp32
// operations (explicitly rounded, never contracted), so that every platform
// computing the same steps gets the same bits: x = 2^e m with m in
// [sqrt(1/2), sqrt(2)), ln m = 2 atanh(s) = 2s (1 + s^2/3 + ... + s^10/11)
// with s = (m - 1)/(m + 1), |s| <= 0.1716; ln x = e ln 2 + ln m.
__device__ __forceinline__ float ln_f32(float x) {
    const uint32_t b = __float_as_uint(x);
    int e = (int)((b >> 23) & 0xffu) - 127;
    float m = __uint_as_float((b & 0x7fffffu) | 0x3f800000u);
    if (m > 0x1.6a09e6p+0f) {
        m = __fmul_rn(m, 0.5f);
        e += 1;
    }
    const float s = __fdiv_rn(__fsub_rn(m, 1.0f), __fadd_rn(m, 1.0f));
    const float z = __fmul_rn(s, s);
    float p = __fmaf_rn(z, 0x1.745d18p-4f, 0x1.c71c72p-4f);
    p = __fmaf_rn(z, p, 0x1.24924ap-3f);
    p = __fmaf_rn(z, p, 0x1.99999ap-3f);
    p = __fmaf_rn(z, p, 0x1.555556p-2f);
    p = __fmaf_rn(z, p, 1.0f);
    const float lm = __fmul_rn(__fmul_rn(2.0f, s), p);
    return __fmaf_rn(__int2float_rn(e), 0x1.62e430p-1f, lm);
}
// (not inlined: the row pass calls it from several unrolled sites)
__device__ __noinline__ float gumbel(int v, int row, const VocabArgs &a) {
    const uint64_t x = philox_word((uint64_t)(v >> 2), (uint64_t)row, a.offset, 0ull, a.seed, 0ull, v & 3);
    const float u = __fmul_rn(__uint2float_rn(2u * (uint32_t)(x >> 41) + 1u), 0x1p-24f);
    return -ln_f32(-ln_f32(u));
}

// Reductions of (value, index) pairs and counts over one CTA; every thread
// receives the result.  `red` holds one slot per warp.
__device__ __forceinline__ ArgMax block_best(ArgMax b, ArgMax *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ArgMax other{__shfl_xor_sync(0xffffffffu, b.v, o), __shfl_xor_sync(0xffffffffu, b.i, o)};
        b = better(b, other);
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = b;
    __syncthreads();
    ArgMax r = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = better(r, red[w]);
    return r;
}

// Bulk copy (TMA, no tensor map) of `bytes` from global to this CTA's shared
// memory, completing on `bar` (address and size multiples of 16 bytes).
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            tc::smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(tc::smem_u32(bar))
        : "memory");
}

template <bool SAMPLE>
__global__ void __cluster_dims__(VOCAB_CLUSTER, 1, 1) __launch_bounds__(VOCAB_THREADS)
penalty_minp_kernel(const VocabArgs a, int slice) {
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ __align__(16) float xs[];  // this CTA's slice of the row's logits
    __shared__ uint32_t bitmap[VOCAB_BITMAP_WORDS];
    __shared__ ArgMax red[VOCAB_THREADS / 32];
    __shared__ float red_max[VOCAB_THREADS / 32];
    __shared__ float cta_max;
    __shared__ int warp_cnt[VOCAB_THREADS / 32], warp_arg[VOCAB_THREADS / 32];
    __shared__ int cta_cnt, cta_arg;
    __shared__ ArgMax cta_samp;
    __shared__ float row_max;
    __shared__ __align__(8) uint64_t bar;

    const int row = blockIdx.y;
    const unsigned rank = cluster.block_rank();
    const int v0 = (int)rank * slice;
    const int v1 = min(a.V, v0 + slice);
    const int n = max(0, v1 - v0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *lrow = a.logits + (size_t)row * a.V;
    // the slice's whole 16-byte units go by one bulk copy; a ragged end (rows
    // whose start is not 16-byte aligned, or a length not a multiple of 4)
    // by plain loads
    const bool aligned = (((uintptr_t)(lrow + v0)) & 15u) == 0;
    const int n_bulk = aligned ? (n & ~3) : 0;
    if (tid == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
        if (n_bulk > 0) {
            tc::mbar_arrive_expect_tx(&bar, (uint32_t)n_bulk * 4u);
            bulk_g2s(xs, lrow + v0, (uint32_t)n_bulk * 4u, &bar);
        } else {
            tc::mbar_arrive(&bar);
        }
    }
    for (int i = n_bulk + tid; i < n; i += VOCAB_THREADS) xs[i] = lrow[v0 + i];

    // window bitmap restricted to this slice (ids outside [0, V) are ignored
    // here; the acceptance kernel reports them).  With the path-aware window,
    // row i's window is the last W tokens of history ++ the drafts on its
    // path root..i: history[min(d, W)..W) and the path's last min(d, W) drafts.
    for (int w = tid; w < VOCAB_BITMAP_WORDS; w += VOCAB_THREADS) bitmap[w] = 0u;
    int depth = 0;
    if (a.path_window) {
        // the walk stops at a parent that is not below its child (a bad parent
        // array, which the acceptance kernel reports)
        for (int j = row; j >= 0;) {
            ++depth;
            const int p = a.parent[j];
            j = (p < j && p >= -1) ? p : -1;
        }
    }
    const int take = depth < a.W ? depth : a.W;  // path drafts inside the window
    __syncthreads();
    for (int w = take + tid; w < a.W; w += VOCAB_THREADS) {
        const int id = a.history[w];
        if (id >= v0 && id < v1) atomicOr(&bitmap[(id - v0) >> 5], 1u << ((id - v0) & 31));
    }
    if (a.path_window && tid == 0) {
        int pos = depth;  // 1-based position of j on the path
        for (int j = row; j >= 0 && pos > depth - take; --pos) {
            const int id = a.draft[j];
            if (id >= v0 && id < v1) atomicOr(&bitmap[(id - v0) >> 5], 1u << ((id - v0) & 31));
            const int p = a.parent[j];
            j = (p < j && p >= -1) ? p : -1;
        }
    }
    // the slice has landed (bounded wait; a copy that never lands leaves the
    // row's target undefined, kept = -1, and the acceptance kernel reports
    // TS_ERR_TIMEOUT in result[3])
    const bool landed = tc::mbar_wait(&bar, 0, nullptr);
    __syncthreads();

    // penalised, tempered logits of slice elements 4q..4q+3 (dividing by a
    // temperature of 1 is exact, so that division is skipped)
    const bool tempered = a.temperature != 1.0f;
    const int n4 = n >> 2;
    const float4 *xs4 = reinterpret_cast<const float4 *>(xs);
    auto final4 = [&](int q, float (&l)[4]) {
        const float4 x = xs4[q];
        l[0] = x.x; l[1] = x.y; l[2] = x.z; l[3] = x.w;
        const uint32_t bits = (bitmap[q >> 3] >> ((q & 7) * 4)) & 0xfu;
        if (bits) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if ((bits >> e) & 1u) l[e] = l[e] > 0.f ? __fdiv_rn(l[e], a.theta) : __fmul_rn(l[e], a.theta);
        }
        if (tempered) {
#pragma unroll
            for (int e = 0; e < 4; ++e) l[e] = __fdiv_rn(l[e], a.temperature);
        }
    };
    auto final1 = [&](int i) {
        float l = xs[i];
        if ((bitmap[i >> 5] >> (i & 31)) & 1u) l = l > 0.f ? __fdiv_rn(l, a.theta) : __fmul_rn(l, a.theta);
        return tempered ? __fdiv_rn(l, a.temperature) : l;
    };

    // ---- pass 1: the penalised logits written back in place, each 16-byte
    // slot's maximum kept in a register, and the slice's maximum
    constexpr int SLOTS = VOCAB_MAX_SLICE / 4 / VOCAB_THREADS;  // 10
    float m4[SLOTS];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < SLOTS; ++i) {
        const int q = i * VOCAB_THREADS + tid;
        m4[i] = -INFINITY;
        if (q < n4) {
            float l[4];
            final4(q, l);
            reinterpret_cast<float4 *>(xs)[q] = make_float4(l[0], l[1], l[2], l[3]);
            m4[i] = fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3]));
            mx = fmaxf(mx, m4[i]);
        }
    }
    for (int i = 4 * n4 + tid; i < n; i += VOCAB_THREADS) {
        xs[i] = final1(i);
        mx = fmaxf(mx, xs[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red_max[warp] = mx;
    __syncthreads();
    if (tid == 0) {
        float b = red_max[0];
        for (int w = 1; w < VOCAB_THREADS / 32; ++w) b = fmaxf(b, red_max[w]);
        cta_max = b;
    }
    cluster.sync();
    // the row maximum: lanes 0..7 of warp 0 read one CTA's slice maximum each
    // (eight remote reads per CTA, not eight per thread)
    if (warp == 0) {
        float v = lane < VOCAB_CLUSTER ? *cluster.map_shared_rank(&cta_max, lane) : -INFINITY;
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) row_max = v;
    }
    __syncthreads();
    const float m = row_max;
    // min-p threshold: smallest fp32 >= m + ln(min_p) (exact comparison)
    const float f = __double2float_ru((double)m + a.log_min_p);

    // ---- pass 2: min-p count, the lowest id attaining the maximum, and the
    // Gumbel-max draw over the kept ids
    int cnt = 0, arg = 0x7fffffff;
    ArgMax sb{-INFINITY, -1};
    auto visit = [&](float l, int v) {
        if (l >= f) {
            ++cnt;
            if (l == m && v < arg) arg = v;
            if constexpr (SAMPLE) sb = better(sb, ArgMax{__fadd_rn(l, gumbel(v, row, a)), v});
        }
    };
    // only slots whose maximum reaches the threshold are visited element by
    // element (a few per row at min-p 0.1)
#pragma unroll
    for (int i = 0; i < SLOTS; ++i) {
        const int q = i * VOCAB_THREADS + tid;
        if (q < n4 && m4[i] >= f) {
            const float4 l = reinterpret_cast<const float4 *>(xs)[q];
            visit(l.x, v0 + 4 * q + 0);
            visit(l.y, v0 + 4 * q + 1);
            visit(l.z, v0 + 4 * q + 2);
            visit(l.w, v0 + 4 * q + 3);
        }
    }
    for (int i = 4 * n4 + tid; i < n; i += VOCAB_THREADS) visit(xs[i], v0 + i);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        arg = min(arg, __shfl_xor_sync(0xffffffffu, arg, o));
    }
    if (lane == 0) {
        warp_cnt[warp] = cnt;
        warp_arg[warp] = arg;
    }
    if constexpr (SAMPLE) {
        sb = block_best(sb, red);
        if (tid == 0) cta_samp = sb;
    }
    __syncthreads();
    if (tid == 0) {
        int c = 0, ar = 0x7fffffff;
        for (int w = 0; w < VOCAB_THREADS / 32; ++w) {
            c += warp_cnt[w];
            ar = min(ar, warp_arg[w]);
        }
        cta_cnt = landed ? c : -1;  // -1: this CTA's slice never landed
        cta_arg = ar;
    }
    cluster.sync();
    if (rank == 0 && warp == 0) {
        // lane r < 8 reads CTA r's results (remote reads in parallel)
        int c = 0, ar = 0x7fffffff;
        ArgMax sbest{-INFINITY, -1};
        if (lane < VOCAB_CLUSTER) {
            c = *cluster.map_shared_rank(&cta_cnt, lane);
            ar = *cluster.map_shared_rank(&cta_arg, lane);
            if constexpr (SAMPLE) sbest = *cluster.map_shared_rank(&cta_samp, lane);
        }
        const bool lost = __any_sync(0xffffffffu, c < 0);
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) {
            c += __shfl_xor_sync(0xffffffffu, c, o);
            ar = min(ar, __shfl_xor_sync(0xffffffffu, ar, o));
            if constexpr (SAMPLE) {
                const ArgMax other{__shfl_xor_sync(0xffffffffu, sbest.v, o), __shfl_xor_sync(0xffffffffu, sbest.i, o)};
                sbest = better(sbest, other);
            }
        }
        if (lane == 0) {
            a.target[row] = SAMPLE ? sbest.i : ar;
            a.kept[row] = lost ? -1 : c;
        }
    }
    cluster.sync();  // keep every CTA's shared memory alive until rank 0 has read it
}

// Acceptance: one CTA, one thread per batch row walking its (short) ancestor
// chain; the longest accepted depth wins.  Greedy targets keep the lowest of
// the longest rows; sampled targets draw one of them uniformly ("How it
// works": a random longest accepted draft is kept): with S the
// m longest accepted rows in ascending order, the kept row is
// S[floor(x m / 2^64)], x = word 0 of Philox4x64-10 at counter
// (0, 0, offset, 1) under key (seed, 0).
__global__ void __launch_bounds__(1024) accept_kernel(const VocabArgs a) {
    __shared__ int s_parent[1024];
    __shared__ int s_target[1024];
    __shared__ int s_draft[1024];
    __shared__ int s_depth[1024];  // depth of an accepted row, 0 otherwise
    __shared__ int s_bad;
    __shared__ int s_key;
    __shared__ int s_pick;
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_bad = 0;
        s_key = -1;
    }
    __syncthreads();
    for (int i = tid; i < a.T; i += blockDim.x) {
        const int p = a.parent[i];
        s_parent[i] = p;
        s_target[i] = a.target[i];
        s_draft[i] = a.draft[i];
        if (p < -1 || p >= i) atomicOr(&s_bad, 1);
        if (a.kept[i] < 0) atomicOr(&s_bad, 4);  // the row pass's copy never landed
        a.path[i] = -1;
    }
    for (int w = tid; w < a.W; w += blockDim.x) {
        const int id = a.history[w];
        if (id < 0 || id >= a.V) atomicOr(&s_bad, 2);
    }
    __syncthreads();
    if (s_bad & 1) {  // a bad parent array: report, accept nothing
        if (tid == 0) {
            a.result[0] = 0; a.result[1] = -1; a.result[2] = a.anchor; a.result[3] = 5;  // TS_ERR_DATA
        }
        return;
    }
    for (int i = tid; i < a.T; i += blockDim.x) {
        bool ok = true;
        int depth = 0;
        // parent[n] < n strictly, so the walk ends within i+1 steps
        for (int n = i; n >= 0; n = s_parent[n]) {
            const int pn = s_parent[n];
            const int expected = pn >= 0 ? s_target[pn] : a.anchor;
            ok = ok && (s_draft[n] == expected);
            ++depth;
        }
        s_depth[i] = ok ? depth : 0;
        if (ok) atomicMax(&s_key, (depth << 16) | (0xffff - i));
    }
    __syncthreads();
    const int L_all = s_key < 0 ? 0 : (s_key >> 16);
    if (a.sample && L_all > 0 && tid < 32) {
        // warp 0: m = #longest rows, then the j-th of them in row order
        int m = 0;
        for (int b = 0; b < a.T; b += 32) {
            const int i = b + tid;
            m += __popc(__ballot_sync(0xffffffffu, i < a.T && s_depth[i] == L_all));
        }
        const uint64_t x = philox_word(0ull, 0ull, a.offset, 1ull, a.seed, 0ull, 0);
        int j = (int)__umul64hi(x, (uint64_t)m);
        for (int b = 0; b < a.T; b += 32) {
            const int i = b + tid;
            const unsigned bal = __ballot_sync(0xffffffffu, i < a.T && s_depth[i] == L_all);
            const int c = __popc(bal);
            if (j < c) {
                unsigned rest = bal;
                for (int q = 0; q < j; ++q) rest &= rest - 1;  // drop the j lowest set bits
                if (tid == 0) s_pick = b + __ffs(rest) - 1;
                break;
            }
            j -= c;
        }
    }
    __syncthreads();
    if (tid == 0) {
        const int key = s_key;
        const int L = key < 0 ? 0 : (key >> 16);
        const int best = key < 0 ? -1 : (a.sample ? s_pick : 0xffff - (key & 0xffff));
        a.result[0] = L;
        a.result[1] = best;
        a.result[2] = L > 0 ? s_target[best] : a.anchor;
        a.result[3] = (s_bad & 4) ? (int)TS_ERR_TIMEOUT : ((s_bad & 2) ? (int)TS_ERR_DATA : 0);
        int pos = L - 1;
        for (int n = best; n >= 0 && pos >= 0; n = s_parent[n], --pos) a.path[pos] = n;
    }
}

cudaError_t launch_vocab(const VocabArgs &a, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    int slice = (a.V + VOCAB_CLUSTER - 1) / VOCAB_CLUSTER;
    slice = (slice + 31) & ~31;
    if (slice > VOCAB_MAX_SLICE) return cudaErrorInvalidValue;
    dim3 grid(VOCAB_CLUSTER, a.T);
    const size_t smem = (size_t)slice * sizeof(float);
    cudaError_t e0;
    if (a.sample) {
        e0 = cudaFuncSetAttribute(penalty_minp_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e0 != cudaSuccess) return e0;
        penalty_minp_kernel<true><<<grid, VOCAB_THREADS, smem, st>>>(a, slice);
    } else {
        e0 = cudaFuncSetAttribute(penalty_minp_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e0 != cudaSuccess) return e0;
        penalty_minp_kernel<false><<<grid, VOCAB_THREADS, smem, st>>>(a, slice);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    accept_kernel<<<1, 1024, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ts
