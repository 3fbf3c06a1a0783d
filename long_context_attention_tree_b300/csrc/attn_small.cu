// Split-KV tree-masked GQA attention on the CUDA cores for small batches:
// at most 24 (batch row, query head) pairs per KV head, head dim 128.  This
// is the shape of the TokenSwift self-drafting pass ("How it works": the
// target model with a partial KV cache drafts the next tokens), e.g. 4 chain
// rows x 5 query heads over a 4096-token partial cache.
//
// CTA = (KV head g, 256-token KV range), 512 threads.  Rows r = (t, j)
// t-major, R = T*G, padded to RP = 4*R4.
//   S:  thread = (token, half of the head dim); each thread streams its half
//       K row (128 B) from global memory and forms all R partial dot products
//       with Q held in shared memory as [d][RP] fp32 (one broadcast 16-byte
//       read feeds four rows), packed fp32x2 FMAs; the two halves are added
//       through shared memory.
//   softmax over the CTA's 256 tokens per row: warp shuffles, then shared
//       memory across the 8 warps; P = 2^(s*c - m) goes to shared memory as
//       [token][RP].
//   O:  lane = 4 dims, warp = 16 tokens; each lane reads V[token][4 dims]
//       (coalesced 256 B per token) and accumulates R x 4 outputs; the
//       sixteen warps' partial sums are added through shared memory.
// The partial (O, m, l) of each range goes to the split workspace and the
// log-sum-exp merge kernel combines the ranges (a single range writes the
// normalised output directly).  The chunk importance of the scoring row can
// be produced by the same pass.
#include "internal.h"
#include "ts_common.cuh"

namespace ts {

namespace {
constexpr int SM_THREADS = 512;
constexpr int SM_TOKENS = 256;  // tokens per CTA (two threads each in the S phase)
constexpr int D = 128;

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
}  // namespace

template <int R4>
__global__ void __launch_bounds__(SM_THREADS, 1) tree_attn_small_kernel(const AttnArgs a, int n_splits) {
    constexpr int RP = 4 * R4;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *qs = reinterpret_cast<float *>(smem_raw);   // [D][RP]
    float *ps = qs + D * RP;                            // [SM_TOKENS][RP]
    float *xs = ps + SM_TOKENS * RP;                    // [SM_TOKENS][RP] upper-half partial S
    float *ob = xs + SM_TOKENS * RP;                    // [8 warps][RP][D] partial O
    float *red = ob + 8 * RP * D;                       // [8 warps][RP] partial max, then partial sum
    float *fin = red + 8 * RP;                          // [RP] final max, then [RP] final sum
    float *scs = fin + 2 * RP;                          // [8 warps][32] score partials

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, g = blockIdx.y;
    const int G = a.G, R = a.T * G;
    const int64_t L = a.N + a.T;
    const int64_t t0 = (int64_t)split * SM_TOKENS;

    // ---- Q of the group -> shared memory, transposed to [d][row] (zero padding rows)
    for (int e = tid; e < RP * (D / 8); e += SM_THREADS) {
        const int r = e / (D / 8), c8 = (e % (D / 8)) * 8;
        float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (r < R) {
            const int t = r / G, j = r % G;
            const uint4 w = *reinterpret_cast<const uint4 *>(a.q + ((size_t)t * a.Hq + g * G + j) * D + c8);
            f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
            f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) qs[(c8 + i) * RP + r] = f[i];
    }
    __syncthreads();

    // ---- S: this thread's token and half of the head dim, against every row
    const int hd = tid >> 8;                 // head-dim half (warp-uniform)
    const int tl = tid & (SM_TOKENS - 1);    // token inside the range
    const int64_t tok = t0 + tl;
    const bool in_range = tok < L;
    float2 s[R4][2];
#pragma unroll
    for (int i = 0; i < R4; ++i) s[i][0] = s[i][1] = make_float2(0.f, 0.f);
    if (in_range) {
        const uint4 *krow = reinterpret_cast<const uint4 *>(a.k + ((size_t)g * a.ld_kv + (size_t)tok) * D) + hd * 8;
        uint4 kw[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) kw[c] = krow[c];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint32_t wv[4] = {kw[c].x, kw[c].y, kw[c].z, kw[c].w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float kv = (e & 1) ? bf16_hi(wv[e >> 1]) : bf16_lo(wv[e >> 1]);
                const float2 k2 = make_float2(kv, kv);
                const float4 *q4 = reinterpret_cast<const float4 *>(qs + (hd * 64 + c * 8 + e) * RP);
#pragma unroll
                for (int i = 0; i < R4; ++i) {
                    const float4 q = q4[i];
                    s[i][0] = ffma2(make_float2(q.x, q.y), k2, s[i][0]);
                    s[i][1] = ffma2(make_float2(q.z, q.w), k2, s[i][1]);
                }
            }
        }
    }
    if (hd == 1) {
#pragma unroll
        for (int i = 0; i < R4; ++i)
            reinterpret_cast<float4 *>(xs + tl * RP)[i] = make_float4(s[i][0].x, s[i][0].y, s[i][1].x, s[i][1].y);
    }
    __syncthreads();
    float sv[RP];
#pragma unroll
    for (int i = 0; i < R4; ++i) {
        const float4 u = reinterpret_cast<const float4 *>(xs + tl * RP)[i];
        sv[4 * i + 0] = s[i][0].x + u.x; sv[4 * i + 1] = s[i][0].y + u.y;
        sv[4 * i + 2] = s[i][1].x + u.z; sv[4 * i + 3] = s[i][1].y + u.w;
    }

    // ---- fused chunk importance of the scoring row (raw q.k over tokens < N);
    // a 64-token chunk is two warps of this CTA
    if (hd == 0 && a.chunk_scores != nullptr && a.score_row >= 0 && a.score_row < a.T) {
        const int r0 = a.score_row * G;
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            if (r >= r0 && r < r0 + G) {
                float x = (tok < a.N) ? sv[r] : 0.f;
                x = warp_sum(x);
                if (lane == 0) scs[warp * 32 + (r - r0)] = x;
            }
        }
    }

    // ---- visibility: prefix tokens for every row, batch tokens by ancestry
    const float c = a.scale_log2;
#pragma unroll
    for (int r = 0; r < RP; ++r) {
        bool vis = false;
        if (in_range && r < R) {
            if (tok < a.N) {
                vis = true;
            } else {
                const int t = r / G;
                vis = mask_bit(a.mask, t, (int)(tok - a.N));
            }
        }
        sv[r] = vis ? sv[r] * c : -INFINITY;
    }

    // ---- row max over the CTA's tokens (warps 0-7 own one token per lane)
    if (hd == 0) {
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            const float m = warp_max(sv[r]);
            if (lane == 0) red[warp * RP + r] = m;
        }
    }
    __syncthreads();
    if (a.chunk_scores != nullptr && a.score_row >= 0 && a.score_row < a.T && tid < 4) {
        // chunk (2 warps) tid of this CTA: max over the group's heads
        const int64_t ch_tok0 = t0 + 64 * tid;
        if (ch_tok0 < a.N) {
            float best = -INFINITY;
            for (int j = 0; j < G; ++j) best = fmaxf(best, scs[(2 * tid) * 32 + j] + scs[(2 * tid + 1) * 32 + j]);
            a.chunk_scores[(size_t)g * a.n_chunks + (size_t)(ch_tok0 / 64)] = best;
        }
    }
    if (tid < RP) {
        float m = -INFINITY;
#pragma unroll
        for (int w = 0; w < 8; ++w) m = fmaxf(m, red[w * RP + tid]);
        fin[tid] = m;
    }
    __syncthreads();

    // ---- P -> shared memory [token][row], partial row sums
    if (hd == 0) {
        float pv[RP];
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            const float m = fin[r];
            pv[r] = (m == -INFINITY) ? 0.f : exp2f(sv[r] - m);
        }
#pragma unroll
        for (int i = 0; i < R4; ++i)
            reinterpret_cast<float4 *>(ps + tl * RP)[i] =
                make_float4(pv[4 * i], pv[4 * i + 1], pv[4 * i + 2], pv[4 * i + 3]);
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            const float l = warp_sum(pv[r]);
            if (lane == 0) red[warp * RP + r] = l;
        }
    }
    __syncthreads();
    if (tid < RP) {
        float l = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) l += red[w * RP + tid];
        fin[RP + tid] = l;
    }

    // ---- O: lane = dims [4 lane, 4 lane + 4), warp = tokens [16 warp, 16 warp + 16)
    float2 o[RP][2];
#pragma unroll
    for (int r = 0; r < RP; ++r) o[r][0] = o[r][1] = make_float2(0.f, 0.f);
    const int64_t wt0 = t0 + 16 * warp;
    const int n_tok = (int)max((int64_t)0, min((int64_t)16, L - wt0));
    const uint2 *vcol = reinterpret_cast<const uint2 *>(a.v + ((size_t)g * a.ld_kv + (size_t)wt0) * D) + lane;
    for (int i0 = 0; i0 < n_tok; i0 += 8) {
        uint2 vw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) vw[i] = (i0 + i < n_tok) ? vcol[(size_t)(i0 + i) * (D / 4)] : make_uint2(0u, 0u);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 v01 = make_float2(bf16_lo(vw[i].x), bf16_hi(vw[i].x));
            const float2 v23 = make_float2(bf16_lo(vw[i].y), bf16_hi(vw[i].y));
            const float4 *p4 = reinterpret_cast<const float4 *>(ps + (16 * warp + i0 + i) * RP);
#pragma unroll
            for (int q = 0; q < R4; ++q) {
                const float4 p = p4[q];  // zero past the range: tokens beyond L have P = 0
                const float pr[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 pp = make_float2(pr[e], pr[e]);
                    o[4 * q + e][0] = ffma2(pp, v01, o[4 * q + e][0]);
                    o[4 * q + e][1] = ffma2(pp, v23, o[4 * q + e][1]);
                }
            }
        }
    }
    // ---- add the sixteen warps' partial O: 16 -> 8 -> 4 -> 2 -> 1
#pragma unroll
    for (int step = 8; step >= 1; step >>= 1) {
        if (warp >= step && warp < 2 * step) {
            float4 *dst = reinterpret_cast<float4 *>(ob + (size_t)(warp - step) * RP * D) + lane;
#pragma unroll
            for (int r = 0; r < RP; ++r)
                dst[r * (D / 4)] = make_float4(o[r][0].x, o[r][0].y, o[r][1].x, o[r][1].y);
        }
        __syncthreads();
        if (warp < step) {
            const float4 *src = reinterpret_cast<const float4 *>(ob + (size_t)warp * RP * D) + lane;
#pragma unroll
            for (int r = 0; r < RP; ++r) {
                const float4 x = src[r * (D / 4)];
                o[r][0].x += x.x; o[r][0].y += x.y; o[r][1].x += x.z; o[r][1].y += x.w;
            }
        }
        __syncthreads();
    }
    if (warp == 0) {
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            if (r >= R) break;
            const int t = r / G, j = r % G;
            const size_t row = (size_t)t * a.Hq + g * G + j;
            const float m = fin[r], l = fin[RP + r];
            if (n_splits == 1) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
                __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(a.out + row * D) + 2 * lane;
                dst[0] = __floats2bfloat162_rn(o[r][0].x * inv, o[r][0].y * inv);
                dst[1] = __floats2bfloat162_rn(o[r][1].x * inv, o[r][1].y * inv);
                if (a.lse != nullptr && lane == 0) a.lse[row] = (m + log2f(l)) * TS_LN2;
            } else {
                float4 *dst = reinterpret_cast<float4 *>(a.ws_o + ((size_t)split * a.T * a.Hq + row) * D) + lane;
                *dst = make_float4(o[r][0].x, o[r][0].y, o[r][1].x, o[r][1].y);
                if (lane == 0)
                    reinterpret_cast<float2 *>(a.ws_ml)[(size_t)split * a.T * a.Hq + row] = make_float2(m, l);
            }
        }
    }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
bool small_ok(int T, int Hq, int Hkv, int d) { return d == 128 && T >= 1 && T * (Hq / Hkv) <= 24; }

int small_splits(int T, int64_t N) { return (int)((N + T + SM_TOKENS - 1) / SM_TOKENS); }

template <int R4>
static size_t small_smem() {
    constexpr int RP = 4 * R4;
    return sizeof(float) * ((size_t)D * RP + 2 * (size_t)SM_TOKENS * RP + 8 * (size_t)RP * D + 8 * RP + 2 * RP + 8 * 32);
}

template <int R4>
static cudaError_t launch_small_t(const AttnArgs &a, int splits, cudaStream_t st) {
    const size_t smem = small_smem<R4>();
    cudaError_t e = cudaFuncSetAttribute(tree_attn_small_kernel<R4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(splits, a.Hkv);
    tree_attn_small_kernel<R4><<<grid, SM_THREADS, smem, st>>>(a, splits);
    return cudaGetLastError();
}

cudaError_t launch_tree_attn_small(const AttnArgs &a, int splits, cudaStream_t st) {
    const int r4 = (a.T * a.G + 3) / 4;
    switch (r4) {
        case 1: return launch_small_t<1>(a, splits, st);
        case 2: return launch_small_t<2>(a, splits, st);
        case 3: return launch_small_t<3>(a, splits, st);
        case 4: return launch_small_t<4>(a, splits, st);
        case 5: return launch_small_t<5>(a, splits, st);
        case 6: return launch_small_t<6>(a, splits, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ts
