// Split-KV tree-masked GQA attention on the CUDA cores for small batches:
// at most 24 (batch row, query head) pairs per KV head, head dim 128.  This
// is the shape of the TokenSwift self-drafting pass ("How it works": the
// target model with a partial KV cache drafts the next tokens), e.g. 4 chain
// rows x 5 query heads over a 4096-token partial cache.
//
// CTA = (KV head g, 128-token KV range); rows r = (t, j) t-major, R = T*G,
// in groups of four.  The range's K and V (32 KB each) are copied into
// shared memory with 16-byte cp.async at the start, so every byte of the
// range is in flight at once (K rows XOR-swizzled by 16-byte chunk so that
// lanes reading different rows hit different banks).  Two warps own each
// group of four rows, one per 64-token half of the range, so a CTA runs
// 2 x ceil(R/4) warps and the latencies of one warp's chain hide behind the
// others':
//   S:  lane l of half h takes tokens 64h + l and 64h + l + 32, 8 dims at a
//       time; Q sits in shared memory as [d][row][2] fp32 (each value twice),
//       so one broadcast 16-byte read gives two rows as pairs and the products
//       are packed fp32x2 FMAs over the token pair.
//   softmax over the range: row max per half by warp shuffles, the two halves
//       combined through shared memory; P goes to the warp's own slab as
//       [token][row][2]; row sums per half, added at the end.
//   O:  lane l owns dims 4l..4l+3; per token one 8-byte V read (the warp
//       reads the whole 256-byte row) and two broadcast reads of P feed 16
//       FMAs; half 1 hands its partial O to half 0 through shared memory.
// The partial (O, m, l) of each range goes to the split workspace and the
// log-sum-exp merge kernel combines the ranges (a single range writes the
// normalised output directly).  The chunk importance of the scoring row can
// be produced by the same pass (a range is two 64-token chunks).
#include "internal.h"
#include "ts_common.cuh"

namespace ts {

namespace {
constexpr int SM_TOKENS = 128;  // tokens per CTA: 4 per lane
constexpr int D = 128;

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
}  // namespace

template <int R4>
__global__ void __launch_bounds__(R4 * 64) tree_attn_small_kernel(const AttnArgs a, int n_splits) {
    constexpr int RP = 4 * R4;
    constexpr int NT = R4 * 64;                        // threads: two warps per row group
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char *sk = smem_raw;                      // [SM_TOKENS][D] bf16, 16-byte chunks swizzled
    unsigned char *sv = sk + SM_TOKENS * D * 2;        // [SM_TOKENS][D] bf16
    float *qs = reinterpret_cast<float *>(sv + SM_TOKENS * D * 2);  // [D][RP][2]
    float *ps = qs + D * RP * 2;                       // [2 R4 warps][64 tokens][4][2]
    float *oc = reinterpret_cast<float *>(sk);         // [R4][4 rows][D]: half 1's P.V partial (K is dead by then)
    __shared__ float scs[2][32];                       // chunk sums of the scoring rows, [chunk][head]
    __shared__ float red_m[2][RP], red_l[2][RP];       // per half: row max and row sum

    // a programmatic dependent: the previous kernel (e.g. the gather of the
    // partial cache) has completed and its writes are visible past this point
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int half = warp / R4, rg = warp % R4;        // tokens [64 half, 64 half + 64), rows 4 rg .. 4 rg + 3
    const int split = blockIdx.x, g = blockIdx.y;
    const int G = a.G, R = a.T * G;
    const int64_t L = a.N + a.T;
    const int64_t t0 = (int64_t)split * SM_TOKENS;
    const int n_tok = (int)max((int64_t)0, min((int64_t)SM_TOKENS, L - t0));

    // ---- Q of the group: global loads first (they must not queue behind the
    // range's K/V copies); rows vary fastest across the threads so that the
    // transposed shared-memory stores do not collide in one bank
    constexpr int QITER = (RP * (D / 8) + NT - 1) / NT;
    uint4 qw[QITER];
#pragma unroll
    for (int u = 0; u < QITER; ++u) {
        const int e = threadIdx.x + u * NT;
        const int r = e % RP, c8 = (e / RP) * 8;
        qw[u] = make_uint4(0u, 0u, 0u, 0u);
        if (e < RP * (D / 8) && r < R) {
            const int t = r / G, j = r % G;
            qw[u] = *reinterpret_cast<const uint4 *>(a.q + ((size_t)t * a.Hq + g * G + j) * D + c8);
        }
    }

    // ---- the range's K (group 0) and V (group 1) -> shared memory; rows past
    // the range are zero-filled
    {
        const __nv_bfloat16 *kg = a.k + ((size_t)g * a.ld_kv + (size_t)t0) * D;
        const __nv_bfloat16 *vg = a.v + ((size_t)g * a.ld_kv + (size_t)t0) * D;
        for (int e = threadIdx.x; e < SM_TOKENS * (D / 8); e += NT) {
            const int row = e / (D / 8), c = e % (D / 8);
            const bool ok = row < n_tok;
            cp_async16_zfill(sk + row * (D * 2) + ((c ^ (row & 7)) * 16), kg + (ok ? (size_t)row * D + c * 8 : 0), ok);
        }
        cp_async_commit();
        for (int e = threadIdx.x; e < SM_TOKENS * (D / 8); e += NT) {
            const int row = e / (D / 8), c = e % (D / 8);
            const bool ok = row < n_tok;
            cp_async16_zfill(sv + row * (D * 2) + c * 16, vg + (ok ? (size_t)row * D + c * 8 : 0), ok);
        }
        cp_async_commit();
    }

    // ---- Q -> shared memory as [d][row][2] (padding rows zero)
#pragma unroll
    for (int u = 0; u < QITER; ++u) {
        const int e = threadIdx.x + u * NT;
        if (e < RP * (D / 8)) {
            const int r = e % RP, c8 = (e / RP) * 8;
            const uint4 w = qw[u];
            const float f[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                                bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
            for (int i = 0; i < 8; ++i)
                *reinterpret_cast<float2 *>(qs + ((c8 + i) * RP + r) * 2) = make_float2(f[i], f[i]);
        }
    }
    cp_async_wait<1>();  // K has landed
    __syncthreads();

    // ---- S for tokens tok[i] = t0 + 64 half + lane + 32 i (i = 0, 1) and rows
    // 4 rg + jr: acc[jr] = (token 0, token 1)
    int64_t tok[2];
    bool in_range[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        tok[i] = t0 + 64 * half + lane + 32 * i;
        in_range[i] = tok[i] < L;
    }
    float2 acc[4];
#pragma unroll
    for (int jr = 0; jr < 4; ++jr) acc[jr] = make_float2(0.f, 0.f);
    {
        const float4 *q4 = reinterpret_cast<const float4 *>(qs) + rg * 2;             // rows 4rg..4rg+3 of dim 0
        const unsigned char *krow = sk + (64 * half + lane) * (D * 2);               // token 64 half + lane; + 32 i
        const int sw = lane & 7;                                                     // (64 half + lane + 32 i) & 7
#pragma unroll 4
        for (int c = 0; c < D / 8; ++c) {
            const uint4 k0 = *reinterpret_cast<const uint4 *>(krow + ((c ^ sw) * 16));
            const uint4 k1 = *reinterpret_cast<const uint4 *>(krow + 32 * (D * 2) + ((c ^ sw) * 16));
            const uint32_t w0[4] = {k0.x, k0.y, k0.z, k0.w}, w1[4] = {k1.x, k1.y, k1.z, k1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float4 qa = q4[(c * 8 + e) * (RP / 2)];      // (q0, q0, q1, q1)
                const float4 qb = q4[(c * 8 + e) * (RP / 2) + 1];  // (q2, q2, q3, q3)
                const float2 kk = (e & 1) ? make_float2(bf16_hi(w0[e >> 1]), bf16_hi(w1[e >> 1]))
                                          : make_float2(bf16_lo(w0[e >> 1]), bf16_lo(w1[e >> 1]));
                acc[0] = ffma2(kk, make_float2(qa.x, qa.y), acc[0]);
                acc[1] = ffma2(kk, make_float2(qa.z, qa.w), acc[1]);
                acc[2] = ffma2(kk, make_float2(qb.x, qb.y), acc[2]);
                acc[3] = ffma2(kk, make_float2(qb.z, qb.w), acc[3]);
            }
        }
    }
    float s[2][4];  // [token i][row jr], raw q.k
#pragma unroll
    for (int jr = 0; jr < 4; ++jr) {
        s[0][jr] = acc[jr].x;
        s[1][jr] = acc[jr].y;
    }

    // ---- fused chunk importance of the scoring row (raw q.k over tokens < N):
    // half h covers chunk 2 split + h
    if (a.chunk_scores != nullptr) {
#pragma unroll
        for (int jr = 0; jr < 4; ++jr) {
            const int r = 4 * rg + jr;
            if (r < R && r / G == a.score_row) {  // warp-uniform
                float x = (tok[0] < a.N ? s[0][jr] : 0.f) + (tok[1] < a.N ? s[1][jr] : 0.f);
                x = warp_sum(x);
                if (lane == 0) scs[half][r % G] = x;
            }
        }
    }

    // ---- visibility: the head's prefix tokens for every row, batch tokens by ancestry
    const float c = a.scale_log2;
    const int64_t plen = prefix_of(a, g);
    float mh[4];
#pragma unroll
    for (int jr = 0; jr < 4; ++jr) {
        const int r = 4 * rg + jr;
        const int t = r < R ? r / G : 0;
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            bool vis = in_range[i] && r < R;
            if (vis) vis = tok[i] < a.N ? tok[i] < plen : mask_bit(a.mask, a.mw, t, (int)(tok[i] - a.N));
            s[i][jr] = vis ? s[i][jr] * c : -INFINITY;
            mx = fmaxf(mx, s[i][jr]);
        }
        mh[jr] = warp_max(mx);
        if (lane == 0) red_m[half][4 * rg + jr] = mh[jr];
    }
    __syncthreads();
    if (a.chunk_scores != nullptr && threadIdx.x < 2) {
        const int64_t ch0 = t0 + 64 * threadIdx.x;
        if (ch0 < a.N) {
            float best = -INFINITY;
            for (int j = 0; j < G; ++j) best = fmaxf(best, scs[threadIdx.x][j]);
            a.chunk_scores[(size_t)g * a.n_chunks + (size_t)(ch0 / 64)] = best;
        }
    }
    // ---- P = 2^(s*c - m) with the range's row max into this warp's slab
    // [token][row][2]; row sums per half
    float m[4];
#pragma unroll
    for (int jr = 0; jr < 4; ++jr) m[jr] = fmaxf(red_m[0][4 * rg + jr], red_m[1][4 * rg + jr]);
    float *pw = ps + (size_t)warp * 64 * 8;
    float lh[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float p[4];
#pragma unroll
        for (int jr = 0; jr < 4; ++jr) {
            p[jr] = (m[jr] == -INFINITY) ? 0.f : exp2f(s[i][jr] - m[jr]);
            lh[jr] += p[jr];
        }
        float4 *dst = reinterpret_cast<float4 *>(pw + (lane + 32 * i) * 8);
        dst[0] = make_float4(p[0], p[0], p[1], p[1]);
        dst[1] = make_float4(p[2], p[2], p[3], p[3]);
    }
#pragma unroll
    for (int jr = 0; jr < 4; ++jr) {
        lh[jr] = warp_sum(lh[jr]);
        if (lane == 0) red_l[half][4 * rg + jr] = lh[jr];
    }
    cp_async_wait<0>();  // V has landed (this thread's copies) ...
    __syncthreads();     // ... and every thread's; P of this warp is visible too

    // ---- O: lane = dims [4 lane, 4 lane + 4), the 64 tokens of this half
    float2 o[4][2];
#pragma unroll
    for (int jr = 0; jr < 4; ++jr) o[jr][0] = o[jr][1] = make_float2(0.f, 0.f);
    const uint2 *vcol = reinterpret_cast<const uint2 *>(sv) + (size_t)64 * half * (D / 4) + lane;
    const int n_half = max(0, min(64, n_tok - 64 * half));
    for (int i0 = 0; i0 < n_half; i0 += 16) {
        uint2 vw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) vw[i] = vcol[(i0 + i) * (D / 4)];  // zero past the range
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float2 v01 = make_float2(bf16_lo(vw[i].x), bf16_hi(vw[i].x));
            const float2 v23 = make_float2(bf16_lo(vw[i].y), bf16_hi(vw[i].y));
            const float4 *p4 = reinterpret_cast<const float4 *>(pw + (i0 + i) * 8);
            const float4 pa = p4[0], pb = p4[1];  // zero past the range
            o[0][0] = ffma2(make_float2(pa.x, pa.y), v01, o[0][0]);
            o[0][1] = ffma2(make_float2(pa.x, pa.y), v23, o[0][1]);
            o[1][0] = ffma2(make_float2(pa.z, pa.w), v01, o[1][0]);
            o[1][1] = ffma2(make_float2(pa.z, pa.w), v23, o[1][1]);
            o[2][0] = ffma2(make_float2(pb.x, pb.y), v01, o[2][0]);
            o[2][1] = ffma2(make_float2(pb.x, pb.y), v23, o[2][1]);
            o[3][0] = ffma2(make_float2(pb.z, pb.w), v01, o[3][0]);
            o[3][1] = ffma2(make_float2(pb.z, pb.w), v23, o[3][1]);
        }
    }
    // the split merge, a programmatic dependent, may start launching now
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // ---- half 1 hands its partial to half 0 (through the dead K buffer)
    if (half == 1) {
#pragma unroll
        for (int jr = 0; jr < 4; ++jr)
            *reinterpret_cast<float4 *>(oc + ((size_t)rg * 4 + jr) * D + 4 * lane) =
                make_float4(o[jr][0].x, o[jr][0].y, o[jr][1].x, o[jr][1].y);
    }
    __syncthreads();
    if (half == 1) return;

    // ---- this range's result for the warp's rows
#pragma unroll
    for (int jr = 0; jr < 4; ++jr) {
        const int r = 4 * rg + jr;
        if (r >= R) break;
        const float4 q1 = *reinterpret_cast<const float4 *>(oc + ((size_t)rg * 4 + jr) * D + 4 * lane);
        o[jr][0].x += q1.x; o[jr][0].y += q1.y; o[jr][1].x += q1.z; o[jr][1].y += q1.w;
        const float l = red_l[0][r] + red_l[1][r];
        const int t = r / G, j = r % G;
        const size_t row = (size_t)t * a.Hq + g * G + j;
        if (n_splits == 1) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(a.out + row * D) + 2 * lane;
            dst[0] = __floats2bfloat162_rn(o[jr][0].x * inv, o[jr][0].y * inv);
            dst[1] = __floats2bfloat162_rn(o[jr][1].x * inv, o[jr][1].y * inv);
            if (a.lse != nullptr && lane == 0) a.lse[row] = (m[jr] + log2f(l)) * TS_LN2;
        } else {
            float4 *dst = reinterpret_cast<float4 *>(a.ws_o + ((size_t)split * a.T * a.Hq + row) * D) + lane;
            *dst = make_float4(o[jr][0].x, o[jr][0].y, o[jr][1].x, o[jr][1].y);
            if (lane == 0)
                reinterpret_cast<float2 *>(a.ws_ml)[(size_t)split * a.T * a.Hq + row] = make_float2(m[jr], l);
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
    // K, V; Q as fp32 pairs; a 64-token P slab per warp (2 R4 warps)
    return 2 * (size_t)SM_TOKENS * D * 2 + sizeof(float) * ((size_t)D * RP * 2 + (size_t)2 * R4 * 64 * 8);
}

template <int R4>
static cudaError_t launch_small_t(const AttnArgs &a, int splits, cudaStream_t st) {
    const size_t smem = small_smem<R4>();
    cudaError_t e = cudaFuncSetAttribute(tree_attn_small_kernel<R4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(splits, a.Hkv);
    cfg.blockDim = dim3(R4 * 64);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tree_attn_small_kernel<R4>, a, splits);
}

cudaError_t launch_tree_attn_small(const AttnArgs &a, int splits, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
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
