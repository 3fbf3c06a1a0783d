// Split-KV tree-masked GQA attention on the CUDA cores, and the log-sum-exp
// merge of split partials.
//
// Used for batches with fewer than 64 query rows (the 4-row self-drafting pass
// over the partial cache of the TokenSwift "How it works" loop, small trees),
// for head_dim 64, and as an independent cross-check of the tensor-core path.
//
// Work decomposition: CTA = (row block, KV head g, KV split).  A row block is
// `tpb` whole batch rows t times all G query heads of the group, so the K/V
// tile staged in shared memory is reused by every query head that reads it.
// KV tiles are 64 tokens (= one scoring chunk), double-buffered with cp.async.
// Scores are kept in the log2 domain (scale * log2 e folded in) so the softmax
// uses exp2.
#include "internal.h"
#include "ts_common.cuh"

namespace ts {

constexpr int SIMT_TILE = 64;
constexpr int SIMT_THREADS = 128;

template <int D>
struct SimtSmem {
    static constexpr int KSTRIDE = D + 8;  // bf16 elements; 16 B pad -> conflict-free 16 B reads
};

template <int D, int RB>
__global__ void __launch_bounds__(SIMT_THREADS)
tree_attn_simt_kernel(const AttnArgs a) {
    constexpr int KS = SimtSmem<D>::KSTRIDE;
    constexpr int SS = SIMT_TILE + 4;        // fp32 row stride of the score tile
    constexpr int RPT = RB / 8;              // rows per thread (S and PV phases)
    constexpr int DPT = D / 16;              // output dims per thread (PV phase)
    constexpr int TPR = SIMT_THREADS / RB;   // softmax threads per row
    constexpr int CPR = SIMT_TILE / TPR;     // softmax columns per thread

    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *sQ = reinterpret_cast<float *>(smem_raw);                       // [RB][D]
    __nv_bfloat16 *sK = reinterpret_cast<__nv_bfloat16 *>(sQ + RB * D);   // [2][64][KS]
    __nv_bfloat16 *sV = sK + 2 * SIMT_TILE * KS;                            // [2][64][KS]
    float *sS = reinterpret_cast<float *>(sV + 2 * SIMT_TILE * KS);        // [RB][SS]
    float *sAlpha = sS + RB * SS;                                           // [RB]
    float *sM = sAlpha + RB;                                                // [RB]
    float *sL = sM + RB;                                                    // [RB]
    float *sScore = sL + RB;                                                // [RB]

    const int tid = threadIdx.x;
    const int rb = blockIdx.x, g = blockIdx.y, split = blockIdx.z;
    const int G = a.G;
    const int t0 = rb * a.tpb;
    const int rows_here = a.tpb * G;
    const int64_t L = a.N + a.T;
    const int tile_begin = split * a.tiles_per_split;
    const int tile_end = min(a.n_tiles, tile_begin + a.tiles_per_split);

    const __nv_bfloat16 *kh = a.k + (size_t)g * a.ld_kv * D;
    const __nv_bfloat16 *vh = a.v + (size_t)g * a.ld_kv * D;

    // --- Q block -> fp32 smem (rows past the batch are zero and never written back)
    for (int e = tid; e < RB * (D / 8); e += SIMT_THREADS) {
        const int lr = e / (D / 8), c8 = (e % (D / 8)) * 8;
        const int t = t0 + lr / G, j = lr % G;
        float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (lr < rows_here && t < a.T) {
            const uint4 w = *reinterpret_cast<const uint4 *>(a.q + ((size_t)t * a.Hq + g * G + j) * D + c8);
            f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
            f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) sQ[lr * D + c8 + i] = f[i];
    }

    auto load_tile = [&](int it, int buf) {
        const int64_t tok0 = (int64_t)it * SIMT_TILE;
        for (int e = tid; e < SIMT_TILE * (D / 8); e += SIMT_THREADS) {
            const int r = e / (D / 8), c8 = (e % (D / 8)) * 8;
            const int64_t tok = tok0 + r;
            const bool ok = tok < L;
            const size_t off = (size_t)(ok ? tok : 0) * D + c8;
            cp_async16_zfill(sK + ((size_t)buf * SIMT_TILE + r) * KS + c8, kh + off, ok);
            cp_async16_zfill(sV + ((size_t)buf * SIMT_TILE + r) * KS + c8, vh + off, ok);
        }
        cp_async_commit();
    };

    // softmax state, owned by the TPR threads of each row
    const int srow = tid / TPR, spart = tid % TPR;
    const int s_t = t0 + srow / G;
    const bool srow_valid = srow < rows_here && s_t < a.T;
    float m_run = -INFINITY, l_run = 0.f;
    const bool score_block = a.chunk_scores != nullptr && a.score_row >= t0 && a.score_row < t0 + a.tpb &&
                             a.score_row < a.T;
    const int64_t plen = prefix_of(a, g);

    // PV ownership
    const int tx = tid & 15, ty = tid >> 4;
    float o[RPT][DPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i)
#pragma unroll
        for (int c = 0; c < DPT; ++c) o[i][c] = 0.f;

    if (tile_begin < tile_end) load_tile(tile_begin, 0);

    for (int it = tile_begin; it < tile_end; ++it) {
        const int buf = (it - tile_begin) & 1;
        if (it + 1 < tile_end) {
            load_tile(it + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        const __nv_bfloat16 *cK = sK + (size_t)buf * SIMT_TILE * KS;
        const __nv_bfloat16 *cV = sV + (size_t)buf * SIMT_TILE * KS;

        // --- S = Q K^T (raw, unscaled): rows ty+8i, tokens tx+16j
        {
            float acc[RPT][4];
#pragma unroll
            for (int i = 0; i < RPT; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 2
            for (int c = 0; c < D; c += 8) {
                float kf[4][8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(cK + (size_t)(tx + 16 * j) * KS + c);
                    kf[j][0] = bf16_lo(w.x); kf[j][1] = bf16_hi(w.x); kf[j][2] = bf16_lo(w.y);
                    kf[j][3] = bf16_hi(w.y); kf[j][4] = bf16_lo(w.z); kf[j][5] = bf16_hi(w.z);
                    kf[j][6] = bf16_lo(w.w); kf[j][7] = bf16_hi(w.w);
                }
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    const float4 qa = *reinterpret_cast<const float4 *>(sQ + (ty + 8 * i) * D + c);
                    const float4 qb = *reinterpret_cast<const float4 *>(sQ + (ty + 8 * i) * D + c + 4);
                    const float qf[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[i][j] = fmaf(qf[e], kf[j][e], acc[i][j]);
                }
            }
#pragma unroll
            for (int i = 0; i < RPT; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) sS[(ty + 8 * i) * SS + tx + 16 * j] = acc[i][j];
        }
        __syncthreads();

        // --- online softmax (log2 domain) + fused chunk score of the scoring row
        {
            const int64_t tok0 = (int64_t)it * SIMT_TILE;
            float x[CPR];
            float tmax = -INFINITY;
            float raw_sum = 0.f;
#pragma unroll
            for (int i = 0; i < CPR; ++i) {
                const int col = spart + TPR * i;
                const int64_t tok = tok0 + col;
                const float s = sS[srow * SS + col];
                bool vis = false;
                if (srow_valid) {
                    if (tok < a.N) {
                        vis = tok < plen;
                        raw_sum += s;
                    } else if (tok < L) {
                        vis = mask_bit(a.mask, a.mw, s_t, (int)(tok - a.N));
                    }
                }
                x[i] = vis ? s * a.scale_log2 : -INFINITY;
                tmax = fmaxf(tmax, x[i]);
            }
#pragma unroll
            for (int o2 = TPR / 2; o2 > 0; o2 >>= 1) {
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o2));
                raw_sum += __shfl_xor_sync(0xffffffffu, raw_sum, o2);
            }
            const float m_new = fmaxf(m_run, tmax);
            const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
            float psum = 0.f;
#pragma unroll
            for (int i = 0; i < CPR; ++i) {
                const float p = (m_new == -INFINITY) ? 0.f : exp2f(x[i] - m_new);
                psum += p;
                sS[srow * SS + spart + TPR * i] = p;
            }
#pragma unroll
            for (int o2 = TPR / 2; o2 > 0; o2 >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o2);
            l_run = l_run * alpha + psum;
            m_run = m_new;
            if (spart == 0) {
                sAlpha[srow] = alpha;
                if (score_block) sScore[srow] = raw_sum;
            }
        }
        __syncthreads();
        if (score_block && tid == 0 && (int64_t)it * SIMT_TILE < a.N) {
            const int base = (a.score_row - t0) * G;
            float best = sScore[base];
            for (int j = 1; j < G; ++j) best = fmaxf(best, sScore[base + j]);
            a.chunk_scores[(size_t)g * a.n_chunks + it] = best;
        }

        // --- O = alpha * O + P V : rows ty+8i, dims tx*DPT + [0, DPT)
        {
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const float al = sAlpha[ty + 8 * i];
#pragma unroll
                for (int c = 0; c < DPT; ++c) o[i][c] *= al;
            }
#pragma unroll 4
            for (int r = 0; r < SIMT_TILE; ++r) {
                float vf[DPT];
                if constexpr (DPT == 8) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(cV + (size_t)r * KS + tx * 8);
                    vf[0] = bf16_lo(w.x); vf[1] = bf16_hi(w.x); vf[2] = bf16_lo(w.y); vf[3] = bf16_hi(w.y);
                    vf[4] = bf16_lo(w.z); vf[5] = bf16_hi(w.z); vf[6] = bf16_lo(w.w); vf[7] = bf16_hi(w.w);
                } else {
                    const uint2 w = *reinterpret_cast<const uint2 *>(cV + (size_t)r * KS + tx * 4);
                    vf[0] = bf16_lo(w.x); vf[1] = bf16_hi(w.x); vf[2] = bf16_lo(w.y); vf[3] = bf16_hi(w.y);
                }
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    const float p = sS[(ty + 8 * i) * SS + r];
#pragma unroll
                    for (int c = 0; c < DPT; ++c) o[i][c] = fmaf(p, vf[c], o[i][c]);
                }
            }
        }
        __syncthreads();
    }

    // --- epilogue: publish m, l; write final output or split partials
    // (the split merge, a programmatic dependent, may start launching now)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (spart == 0) {
        sM[srow] = m_run;
        sL[srow] = l_run;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int lr = ty + 8 * i;
        const int t = t0 + lr / G, j = lr % G;
        if (lr >= rows_here || t >= a.T) continue;
        const int h = g * G + j;
        const size_t row = (size_t)t * a.Hq + h;
        const float m = sM[lr], l = sL[lr];
        if (a.splits == 1) {
            const float inv = 1.f / l;
            __nv_bfloat16 *dst = a.out + row * D + tx * DPT;
#pragma unroll
            for (int c = 0; c < DPT; c += 2) {
                __nv_bfloat162 pr = __floats2bfloat162_rn(o[i][c] * inv, o[i][c + 1] * inv);
                *reinterpret_cast<__nv_bfloat162 *>(dst + c) = pr;
            }
            if (a.lse != nullptr && tx == 0) a.lse[row] = (m + log2f(l)) * TS_LN2;
        } else {
            float *dst = a.ws_o + ((size_t)split * a.T * a.Hq + row) * D + tx * DPT;
#pragma unroll
            for (int c = 0; c < DPT; c += 4)
                *reinterpret_cast<float4 *>(dst + c) = make_float4(o[i][c], o[i][c + 1], o[i][c + 2], o[i][c + 3]);
            if (tx == 0) {
                float2 *ml = reinterpret_cast<float2 *>(a.ws_ml) + (size_t)split * a.T * a.Hq + row;
                *ml = make_float2(m, l);
            }
        }
    }
}

// Log-sum-exp merge over splits (log2 domain partials).  WPR warps per
// (t, h) row (1 when there are many rows, 4 when there are few): each warp
// issues its first eight partial-output loads, reads the splits' (m, l)
// pairs side by side (two per lane) and reduces max and normaliser with
// shuffles while those loads are in flight; warp w then accumulates splits
// w, w+WPR, ... with eight loads in flight per lane, and the row's warps add
// their sums through shared memory.  A row costs about two dependent memory
// round trips.
template <int D, int WPR>
__global__ void __launch_bounds__(128) lse_merge_kernel(const MergeArgs a) {
    constexpr int DPL = D / 32;  // dims per lane
    constexpr int BATCH = 8;     // splits in flight per warp
    constexpr int RPC = 4 / WPR; // rows per CTA
    __shared__ __align__(16) float part[4][D];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row = blockIdx.x * RPC + warp / WPR, sub = warp % WPR;
    const int rows = a.T * a.Hq;
    const bool live = row < rows;  // uniform per CTA when WPR == 4
    const size_t stride = (size_t)rows;
    const int n_split = !live ? 0 : ((row / a.Hq) < a.t_split ? a.splits : a.splits_hi);
    const float2 *ml = reinterpret_cast<const float2 *>(a.ws_ml) + row;
    const float *src0 = a.ws_o + (size_t)row * D + lane * DPL;
    // the partials are the attention kernel's output (this grid may start early)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the next kernel (a programmatic dependent, e.g. the chunk selection) may launch
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    float v[BATCH][DPL];
    auto load_batch = [&](int s0) {
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
            const int s = s0 + WPR * i;
#pragma unroll
            for (int c = 0; c < DPL; ++c) v[i][c] = 0.f;
            if (s < n_split) {
                const float *src = src0 + (size_t)s * stride * D;
                if constexpr (DPL == 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(src);
                    v[i][0] = x.x; v[i][1] = x.y; v[i][2] = x.z; v[i][3] = x.w;
                } else {
                    const float2 x = *reinterpret_cast<const float2 *>(src);
                    v[i][0] = x.x; v[i][1] = x.y;
                }
            }
        }
    };
    load_batch(sub);

    // (m, l) of splits lane and lane + 32 in registers, the rest re-read
    const float2 none = make_float2(-INFINITY, 0.f);
    const float2 p0 = lane < n_split ? ml[(size_t)lane * stride] : none;
    const float2 p1 = lane + 32 < n_split ? ml[(size_t)(lane + 32) * stride] : none;
    float m = fmaxf(p0.x, p1.x);
    for (int s = lane + 64; s < n_split; s += 32) m = fmaxf(m, ml[(size_t)s * stride].x);
    m = warp_max(m);
    // -inf: the split saw no visible key
    const float w0 = p0.x == -INFINITY ? 0.f : exp2f(p0.x - m);
    const float w1 = p1.x == -INFINITY ? 0.f : exp2f(p1.x - m);
    float l = p0.y * w0 + p1.y * w1;
    for (int s = lane + 64; s < n_split; s += 32) {
        const float2 p = ml[(size_t)s * stride];
        if (p.x != -INFINITY) l = fmaf(p.y, exp2f(p.x - m), l);
    }
    l = warp_sum(l);

    float acc[DPL];
#pragma unroll
    for (int c = 0; c < DPL; ++c) acc[c] = 0.f;
    for (int s0 = sub; s0 < n_split; s0 += WPR * BATCH) {
        if (s0 != sub) load_batch(s0);
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
            const int s = s0 + WPR * i;  // warp-uniform
            float w;
            if (s < 32) {
                w = __shfl_sync(0xffffffffu, w0, s);
            } else if (s < 64) {
                w = __shfl_sync(0xffffffffu, w1, s - 32);
            } else {
                const float mx = s < n_split ? ml[(size_t)s * stride].x : -INFINITY;
                w = mx == -INFINITY ? 0.f : exp2f(mx - m);
            }
#pragma unroll
            for (int c = 0; c < DPL; ++c) acc[c] = fmaf(v[i][c], w, acc[c]);
        }
    }
    if constexpr (WPR > 1) {
#pragma unroll
        for (int c = 0; c < DPL; ++c) part[warp][lane * DPL + c] = acc[c];
        __syncthreads();
        if (warp != 0) return;
#pragma unroll
        for (int c = 0; c < DPL; ++c) {
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < WPR; ++w) t += part[w][lane * DPL + c];
            acc[c] = t;
        }
    }
    if (!live) return;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16 *dst = a.out + (size_t)row * D + lane * DPL;
#pragma unroll
    for (int c = 0; c < DPL; c += 2)
        *reinterpret_cast<__nv_bfloat162 *>(dst + c) = __floats2bfloat162_rn(acc[c] * inv, acc[c + 1] * inv);
    if (a.lse != nullptr && lane == 0) a.lse[row] = (m + log2f(l)) * TS_LN2;
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
static int simt_rb(int T, int G) { return (T * G <= 16 && G <= 16) ? 16 : 32; }

template <int D, int RB>
static size_t simt_smem_bytes() {
    constexpr int KS = SimtSmem<D>::KSTRIDE;
    return sizeof(float) * RB * D + 2 * 2 * SIMT_TILE * KS * sizeof(__nv_bfloat16) +
           sizeof(float) * RB * (SIMT_TILE + 4) + 4 * sizeof(float) * RB;
}

SimtPlan simt_plan(int T, int Hq, int Hkv, int d, int64_t N, int num_sms) {
    SimtPlan p{};
    const int G = Hq / Hkv;
    p.rb = simt_rb(T, G);
    p.tpb = p.rb / G;
    p.n_rb = (T + p.tpb - 1) / p.tpb;
    const int64_t L = N + T;
    p.n_tiles = (int)((L + SIMT_TILE - 1) / SIMT_TILE);
    const int64_t base = (int64_t)p.n_rb * Hkv;
    const int64_t want = (2 * (int64_t)num_sms + base - 1) / base;  // about two CTAs per SM
    int64_t splits = want;
    const int64_t max_by_tiles = (p.n_tiles + 1) / 2;                 // at least ~2 tiles per split
    if (splits > max_by_tiles) splits = max_by_tiles;
    if (splits > 64) splits = 64;
    if (splits < 1) splits = 1;
    p.tiles_per_split = (int)((p.n_tiles + splits - 1) / splits);
    p.splits = (p.n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    if (p.splits < 1) p.splits = 1;
    (void)d;
    return p;
}

template <int D, int RB>
static cudaError_t launch_simt_t(const AttnArgs &a, const SimtPlan &p, cudaStream_t st) {
    const size_t smem = simt_smem_bytes<D, RB>();
    cudaError_t e = cudaFuncSetAttribute(tree_attn_simt_kernel<D, RB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_rb, a.Hkv, p.splits);
    tree_attn_simt_kernel<D, RB><<<grid, SIMT_THREADS, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_tree_attn_simt(const AttnArgs &a, const SimtPlan &p, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    if (a.d == 128) return p.rb == 16 ? launch_simt_t<128, 16>(a, p, st) : launch_simt_t<128, 32>(a, p, st);
    return p.rb == 16 ? launch_simt_t<64, 16>(a, p, st) : launch_simt_t<64, 32>(a, p, st);
}

cudaError_t launch_lse_merge(const MergeArgs &m, int d, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    const int rows = m.T * m.Hq;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // few rows: four warps share a row's splits; many rows: a warp per row
    const bool few = (int64_t)rows * 4 <= (int64_t)sms * 32;
    const int blocks = few ? rows : (rows + 3) / 4;
    // a programmatic dependent of the attention kernel: its CTAs launch while
    // the attention kernel's last CTAs finish, then wait for its results
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(128);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (d == 128)
        return few ? cudaLaunchKernelEx(&cfg, lse_merge_kernel<128, 4>, m) : cudaLaunchKernelEx(&cfg, lse_merge_kernel<128, 1>, m);
    return few ? cudaLaunchKernelEx(&cfg, lse_merge_kernel<64, 4>, m) : cudaLaunchKernelEx(&cfg, lse_merge_kernel<64, 1>, m);
}

}  // namespace ts
