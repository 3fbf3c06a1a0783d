// Split-KV tree-masked GQA attention on the CUDA cores for small batches:
// at most 24 (batch row, query head) pairs per KV head, head dim 128.  This
// is the shape of the TokenSwift self-drafting pass ("How it works": the
// target model with a partial KV cache drafts the next tokens), e.g. 4 chain
// rows x 5 query heads over a 4096-token partial cache.
//
// The work is fp32 FMAs (about 1 FMA per 1.5 bytes of K/V), so the kernel is
// built to keep the FMA pipe busy with packed fp32x2 FMAs and few other
// instructions per FMA.
//
// CTA = (KV head g, 128-token KV range), four warps; warp w owns the range's
// tokens 32w .. 32w+31 from the load to its partial result, so the warps
// never wait for one another until the final combine.  Rows r = (t, j)
// t-major, R = T*G, padded to 4 RG (RG = ceil(R/4)).
//   load:  each warp copies its 32 K rows and 32 V rows into shared memory
//          with 16-byte cp.async (K XOR-swizzled by 16-byte chunk so that a
//          quarter-warp reading one chunk of eight rows hits eight banks);
//          rows that are out of range or not gathered are zero-filled.
//   S:     lane (rg, tg) = (lane / 8, lane % 8) takes rows rg*RG .. +RG-1 and
//          tokens tg + 8i (i < 4): per 8 dims it reads four K chunks and 2 RG
//          Q quads (Q is fp32 in shared memory, [dim/4][row slot][4]), and
//          issues 16 RG fp32x2 FMAs over dimension pairs.
//   softmax: the warp's own row max and sum (shuffles over the eight token
//          lanes); P goes to the warp's slab as (p, p) pairs.
//   O:     lane (rh, dg) = (lane / 16, lane % 16) takes rows rh*2RG .. +2RG-1
//          and dims 8dg .. 8dg+7: per token one 16-byte V read, RG 16-byte P
//          reads and 8 RG fp32x2 FMAs.
//   combine: the four warp partials (m, l, O) are merged through shared
//          memory (over the dead K/V buffers) into the range's partial, which
//          goes to the split workspace for the log-sum-exp merge kernel (a
//          single range writes the normalised output directly).
// The chunk importance of the scoring row can be produced by the same pass
// (a warp holds half a 64-token chunk).
//
// Gather variant: the prefix rows are not read from a compact cache but from
// the chunks of the full cache that the top-k selection chose (position p of
// the compact cache is row sel[g][p/64]*64 + p%64 of the full cache); each
// warp also writes its gathered rows into the compact cache, so the refresh
// of the partial cache (selection, gather) and the drafting pass over it read
// the selected K/V bytes from HBM once.
#include "internal.h"
#include "ts_common.cuh"

namespace ts {

namespace {
constexpr int D = 128;
constexpr int WT = 32;              // tokens per warp
constexpr int NWARP = 4;
constexpr int NTHR = NWARP * 32;
constexpr int RANGE = NWARP * WT;   // tokens per CTA: two 64-token chunks
constexpr int ROWB = D * 2;         // bytes of one K/V row

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// The two bf16 halves of a word as an fp32 pair (low half first), by byte
// permutes: each half moves to the upper 16 bits of a zeroed word.
__device__ __forceinline__ float2 bf16x2_f2(uint32_t w) {
    uint32_t lo, hi;
    asm("prmt.b32 %0, %1, %2, 0x1044;" : "=r"(lo) : "r"(w), "r"(0u));
    asm("prmt.b32 %0, %1, %2, 0x3244;" : "=r"(hi) : "r"(w), "r"(0u));
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}

template <int RG>
struct SmallCfg {
    static constexpr int RP = 4 * RG;                  // rows incl. padding
    static constexpr int QS = (RG & 1) ? RG : RG + 1;  // Q slots per row group: odd, so the four groups'
                                                       // 16-byte reads fall in four different bank groups
    static constexpr int QSLOTS = 4 * QS;
    static constexpr int PP = RP + 2;                  // (p, p) pairs per token in a P slab
    static constexpr size_t K_OFF = 0;
    static constexpr size_t V_OFF = (size_t)RANGE * ROWB;
    static constexpr size_t Q_OFF = 2 * (size_t)RANGE * ROWB;
    static constexpr size_t P_OFF = Q_OFF + (size_t)(D / 4) * QSLOTS * 16;
    static constexpr size_t SMEM = P_OFF + (size_t)NWARP * WT * PP * 8;
    static_assert((size_t)NWARP * RP * D * 4 <= 2 * (size_t)RANGE * ROWB, "warp partials must fit the K/V buffers");
};
}  // namespace

template <int RG, bool GATHER>
__global__ void __launch_bounds__(NTHR) tree_attn_small_kernel(const AttnArgs a, const SmallGather gs, int n_splits) {
    using C = SmallCfg<RG>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char *sK = smem_raw + C::K_OFF;
    unsigned char *sV = smem_raw + C::V_OFF;
    float *sQ = reinterpret_cast<float *>(smem_raw + C::Q_OFF);
    float *sP = reinterpret_cast<float *>(smem_raw + C::P_OFF);
    __shared__ float red_m[NWARP][C::RP], red_l[NWARP][C::RP];  // per warp: row max and row sum
    __shared__ float row_m[C::RP], row_l[C::RP];                // the range's
    __shared__ float sc_part[NWARP][32];                        // scoring row: half-chunk sums per head

    // a programmatic dependent: the previous kernel (the selection, the gather
    // of the partial cache) has completed and its writes are visible past here
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int split = blockIdx.x, g = blockIdx.y;
    const int G = a.G, R = a.T * G;
    const int64_t Np = a.N, L = Np + a.T;            // prefix positions, all positions
    const int64_t t0 = (int64_t)split * RANGE;
    const int64_t wb = t0 + (int64_t)w * WT;          // first position of this warp's block
    const bool active = wb < L;
    const int64_t plen = GATHER ? Np : prefix_of(a, g);
    // gather: the full-cache chunk behind this warp's block (a block lies in
    // one chunk: Np is a multiple of 64 there)
    int64_t src_base = 0;
    if (GATHER && wb < Np) {
        const int c = min(max(gs.sel[(size_t)g * gs.k_sel + (int)(wb >> 6)], 0), gs.n_chunks - 1);
        src_base = (int64_t)c * 64 + (wb & 63);
    }
    sc_part[w][lane] = 0.f;

    // ---- Q of the group: global loads first (they must not queue behind the
    // K/V copies)
    constexpr int QITER = (C::RP * 16 + NTHR - 1) / NTHR;
    uint4 qw[QITER];
#pragma unroll
    for (int u = 0; u < QITER; ++u) {
        const int e = threadIdx.x + u * NTHR, r = e >> 4, c8 = e & 15;
        qw[u] = make_uint4(0u, 0u, 0u, 0u);
        if (r < R) {
            const int t = r / G, j = r % G;
            qw[u] = *reinterpret_cast<const uint4 *>(a.q + ((size_t)t * a.Hq + g * G + j) * D + c8 * 8);
        }
    }

    // ---- this warp's 32 K rows (group 0) and V rows (group 1) -> shared memory
    // lane: 16-byte chunk lane % 16 of rows lane / 16 + 2u
    {
        const int c = lane & 15;
        const __nv_bfloat16 *kbase = GATHER ? gs.k : a.k, *vbase = GATHER ? gs.v : a.v;
        size_t off[16];
        bool ok[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int rl = (lane >> 4) + 2 * u;
            const int64_t p = wb + rl;
            ok[u] = false;
            off[u] = 0;
            if (p < Np) {
                if (GATHER) {
                    const int64_t src = src_base + rl;
                    ok[u] = src < gs.N;
                    off[u] = ((size_t)g * gs.ld + (size_t)src) * D + c * 8;
                } else {
                    ok[u] = p < plen;
                    off[u] = ((size_t)g * a.ld_kv + (size_t)p) * D + c * 8;
                }
            } else if (p < L) {
                ok[u] = true;
                off[u] = ((size_t)g * a.ld_kv + (size_t)p) * D + c * 8;
            }
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int rho = w * WT + (lane >> 4) + 2 * u;
            const __nv_bfloat16 *src = (GATHER && wb < Np) ? kbase : a.k;
            cp_async16_zfill(sK + rho * ROWB + ((c ^ (rho & 7)) << 4), src + (ok[u] ? off[u] : 0), ok[u]);
        }
        cp_async_commit();
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int rho = w * WT + (lane >> 4) + 2 * u;
            const __nv_bfloat16 *src = (GATHER && wb < Np) ? vbase : a.v;
            cp_async16_zfill(sV + rho * ROWB + (c << 4), src + (ok[u] ? off[u] : 0), ok[u]);
        }
        cp_async_commit();
    }

    // ---- Q -> shared memory as fp32 [dim/4][slot][4]; row r in slot
    // (r / RG) * QS + r % RG (padding rows zero)
#pragma unroll
    for (int u = 0; u < QITER; ++u) {
        const int e = threadIdx.x + u * NTHR, r = e >> 4, c8 = e & 15;
        if (r < C::RP) {
            const uint4 x = qw[u];
            const int slot = (r / RG) * C::QS + r % RG;
            float4 *dst = reinterpret_cast<float4 *>(sQ);
            dst[(2 * c8) * C::QSLOTS + slot] = make_float4(bf16_lo(x.x), bf16_hi(x.x), bf16_lo(x.y), bf16_hi(x.y));
            dst[(2 * c8 + 1) * C::QSLOTS + slot] =
                make_float4(bf16_lo(x.z), bf16_hi(x.z), bf16_lo(x.w), bf16_hi(x.w));
        }
    }
    __syncthreads();  // Q and the zeroed score slots are visible

    cp_async_wait<1>();  // this lane's K copies have landed ...
    __syncwarp();        // ... and every lane's of the warp

    // gather: the warp's K rows into the compact cache (rows that exist)
    if (GATHER && wb < Np) {
        const int c = lane & 15;
#pragma unroll 4
        for (int u = 0; u < 16; ++u) {
            const int rl = (lane >> 4) + 2 * u, rho = w * WT + rl;
            if (src_base + rl < gs.N) {
                const uint4 x = *reinterpret_cast<const uint4 *>(sK + rho * ROWB + ((c ^ (rho & 7)) << 4));
                *reinterpret_cast<uint4 *>(gs.k_dst + ((size_t)g * a.ld_kv + (size_t)(wb + rl)) * D + c * 8) = x;
            }
        }
    }

    const int rg = lane >> 3, tg = lane & 7;
    float m[RG], l[RG];
#pragma unroll
    for (int i = 0; i < RG; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
    }
    float *pw = sP + (size_t)w * WT * C::PP * 2;  // this warp's P slab [token][row][(p, p)]
    if (active) {
        // ---- S for rows rg*RG + i, tokens tg + 8j of the block: acc[i][j] holds
        // the even- and odd-dimension partial sums
        float2 acc[RG][4];
#pragma unroll
        for (int i = 0; i < RG; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.f, 0.f);
        const unsigned char *kb = sK + (w * WT + tg) * ROWB;  // token tg; + 8j rows (same swizzle: row & 7 = tg)
        const float4 *qb = reinterpret_cast<const float4 *>(sQ) + rg * C::QS;
#pragma unroll 2
        for (int c = 0; c < D / 8; ++c) {
            uint4 kw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) kw[j] = *reinterpret_cast<const uint4 *>(kb + j * 8 * ROWB + ((c ^ tg) << 4));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float4 q4[RG];
#pragma unroll
                for (int i = 0; i < RG; ++i) q4[i] = qb[(2 * c + h) * C::QSLOTS + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 k0 = bf16x2_f2(h ? kw[j].z : kw[j].x);  // dims 8c + 4h, +1
                    const float2 k1 = bf16x2_f2(h ? kw[j].w : kw[j].y);  // dims 8c + 4h + 2, +3
#pragma unroll
                    for (int i = 0; i < RG; ++i) {
                        acc[i][j] = ffma2(k0, make_float2(q4[i].x, q4[i].y), acc[i][j]);
                        acc[i][j] = ffma2(k1, make_float2(q4[i].z, q4[i].w), acc[i][j]);
                    }
                }
            }
        }
        float s[RG][4];
#pragma unroll
        for (int i = 0; i < RG; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[i][j] = acc[i][j].x + acc[i][j].y;

        // ---- fused chunk importance of the scoring row (raw q.k over the
        // prefix): this warp's half-chunk sum per head
        if (a.chunk_scores != nullptr) {
#pragma unroll
            for (int i = 0; i < RG; ++i) {
                float x = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) x += (wb + tg + 8 * j < Np) ? s[i][j] : 0.f;
                x += __shfl_xor_sync(0xffffffffu, x, 1);
                x += __shfl_xor_sync(0xffffffffu, x, 2);
                x += __shfl_xor_sync(0xffffffffu, x, 4);
                const int r = rg * RG + i;
                if (tg == 0 && r < R && r / G == a.score_row) sc_part[w][r % G] = x;
            }
        }

        // ---- visibility, scale, the warp's row max
        const float cs = a.scale_log2;
#pragma unroll
        for (int i = 0; i < RG; ++i) {
            const int r = rg * RG + i;
            const int t = r < R ? r / G : 0;
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t p = wb + tg + 8 * j;
                bool vis = r < R && p < L;
                if (vis) {
                    if (p < Np)
                        vis = GATHER ? (src_base + tg + 8 * j < gs.N) : (p < plen);
                    else
                        vis = mask_bit(a.mask, a.mw, t, (int)(p - Np));
                }
                s[i][j] = vis ? s[i][j] * cs : -INFINITY;
                mx = fmaxf(mx, s[i][j]);
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            m[i] = mx;
        }
        // ---- P = 2^(s*c - m) into the slab as (p, p); the warp's row sums
#pragma unroll
        for (int i = 0; i < RG; ++i) {
            float ls = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float pv = (m[i] == -INFINITY) ? 0.f : exp2f(s[i][j] - m[i]);
                ls += pv;
                *reinterpret_cast<float2 *>(pw + ((size_t)(tg + 8 * j) * C::PP + rg * RG + i) * 2) =
                    make_float2(pv, pv);
            }
            ls += __shfl_xor_sync(0xffffffffu, ls, 1);
            ls += __shfl_xor_sync(0xffffffffu, ls, 2);
            ls += __shfl_xor_sync(0xffffffffu, ls, 4);
            l[i] = ls;
        }
    }
    if (tg == 0) {
#pragma unroll
        for (int i = 0; i < RG; ++i) {
            red_m[w][rg * RG + i] = m[i];
            red_l[w][rg * RG + i] = l[i];
        }
    }

    cp_async_wait<0>();  // V has landed (this lane's copies) ...
    __syncwarp();        // ... and every lane's; this warp's P is visible too

    if (GATHER && wb < Np) {
        const int c = lane & 15;
#pragma unroll 4
        for (int u = 0; u < 16; ++u) {
            const int rl = (lane >> 4) + 2 * u, rho = w * WT + rl;
            if (src_base + rl < gs.N) {
                const uint4 x = *reinterpret_cast<const uint4 *>(sV + rho * ROWB + (c << 4));
                *reinterpret_cast<uint4 *>(gs.v_dst + ((size_t)g * a.ld_kv + (size_t)(wb + rl)) * D + c * 8) = x;
            }
        }
    }

    // ---- O over the warp's 32 tokens: rows rh*2RG + i2, dims 8dg .. 8dg+7
    const int rh = lane >> 4, dg = lane & 15;
    float2 o[2 * RG][4];
#pragma unroll
    for (int i = 0; i < 2 * RG; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) o[i][k] = make_float2(0.f, 0.f);
    if (active) {
        const unsigned char *vb = sV + (w * WT) * ROWB + dg * 16;
        const float *pb = pw + rh * 2 * RG * 2;
#pragma unroll 4
        for (int tw = 0; tw < WT; ++tw) {
            const uint4 vw = *reinterpret_cast<const uint4 *>(vb + tw * ROWB);
            const float2 v0 = bf16x2_f2(vw.x), v1 = bf16x2_f2(vw.y), v2 = bf16x2_f2(vw.z), v3 = bf16x2_f2(vw.w);
#pragma unroll
            for (int i = 0; i < RG; ++i) {
                const float4 pp = *reinterpret_cast<const float4 *>(pb + ((size_t)tw * C::PP + 2 * i) * 2);
                const float2 pa = make_float2(pp.x, pp.y), pc = make_float2(pp.z, pp.w);
                o[2 * i][0] = ffma2(pa, v0, o[2 * i][0]);
                o[2 * i][1] = ffma2(pa, v1, o[2 * i][1]);
                o[2 * i][2] = ffma2(pa, v2, o[2 * i][2]);
                o[2 * i][3] = ffma2(pa, v3, o[2 * i][3]);
                o[2 * i + 1][0] = ffma2(pc, v0, o[2 * i + 1][0]);
                o[2 * i + 1][1] = ffma2(pc, v1, o[2 * i + 1][1]);
                o[2 * i + 1][2] = ffma2(pc, v2, o[2 * i + 1][2]);
                o[2 * i + 1][3] = ffma2(pc, v3, o[2 * i + 1][3]);
            }
        }
    }
    __syncthreads();  // every warp's (m, l) and score sums are written; K and V are dead

    if (a.chunk_scores != nullptr && threadIdx.x < 2) {
        const int64_t ch0 = t0 + 64 * threadIdx.x;
        if (ch0 < Np) {
            float best = -INFINITY;
            for (int j = 0; j < G; ++j) best = fmaxf(best, sc_part[2 * threadIdx.x][j] + sc_part[2 * threadIdx.x + 1][j]);
            a.chunk_scores[(size_t)g * a.n_chunks + (size_t)(ch0 / 64)] = best;
        }
    }

    // ---- combine the four warp partials: each warp scales its O by
    // 2^(m_w - M) and parks it over the K/V buffers as fp32 [warp][row][dim]
    float *sO = reinterpret_cast<float *>(smem_raw);
#pragma unroll
    for (int i2 = 0; i2 < 2 * RG; ++i2) {
        const int r = rh * 2 * RG + i2;
        float M = red_m[0][r];
#pragma unroll
        for (int x = 1; x < NWARP; ++x) M = fmaxf(M, red_m[x][r]);
        const float mw = red_m[w][r];
        const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
        float4 *dst = reinterpret_cast<float4 *>(sO + ((size_t)w * C::RP + r) * D + dg * 8);
        dst[0] = make_float4(o[i2][0].x * f, o[i2][0].y * f, o[i2][1].x * f, o[i2][1].y * f);
        dst[1] = make_float4(o[i2][2].x * f, o[i2][2].y * f, o[i2][3].x * f, o[i2][3].y * f);
        if (w == 0 && dg == 0) {
            float Ls = 0.f;
#pragma unroll
            for (int x = 0; x < NWARP; ++x)
                if (red_m[x][r] != -INFINITY) Ls += exp2f(red_m[x][r] - M) * red_l[x][r];
            row_m[r] = M;
            row_l[r] = Ls;
        }
    }
    // the split merge, a programmatic dependent, may start launching now
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();

    // ---- the range's result: (row, 4 dims) per thread
    for (int e = threadIdx.x; e < R * (D / 4); e += NTHR) {
        const int r = e >> 5, q4 = e & 31;
        float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int x = 0; x < NWARP; ++x) {
            const float4 y = *reinterpret_cast<const float4 *>(sO + ((size_t)x * C::RP + r) * D + 4 * q4);
            acc4.x += y.x; acc4.y += y.y; acc4.z += y.z; acc4.w += y.w;
        }
        const int t = r / G, j = r % G;
        const size_t row = (size_t)t * a.Hq + g * G + j;
        const float M = row_m[r], Ls = row_l[r];
        if (n_splits == 1) {
            const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
            __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(a.out + row * D + 4 * q4);
            dst[0] = __floats2bfloat162_rn(acc4.x * inv, acc4.y * inv);
            dst[1] = __floats2bfloat162_rn(acc4.z * inv, acc4.w * inv);
            if (a.lse != nullptr && q4 == 0) a.lse[row] = (M + log2f(Ls)) * TS_LN2;
        } else {
            *reinterpret_cast<float4 *>(a.ws_o + ((size_t)split * a.T * a.Hq + row) * D + 4 * q4) = acc4;
            if (q4 == 0) reinterpret_cast<float2 *>(a.ws_ml)[(size_t)split * a.T * a.Hq + row] = make_float2(M, Ls);
        }
    }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
bool small_ok(int T, int Hq, int Hkv, int d) { return d == 128 && T >= 1 && T * (Hq / Hkv) <= 24; }

int small_splits(int T, int64_t N) { return (int)((N + T + RANGE - 1) / RANGE); }

template <int RG, bool GATHER>
static cudaError_t launch_small_t(const AttnArgs &a, const SmallGather &gs, int splits, cudaStream_t st) {
    const size_t smem = SmallCfg<RG>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(tree_attn_small_kernel<RG, GATHER>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(splits, a.Hkv);
    cfg.blockDim = dim3(NTHR);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tree_attn_small_kernel<RG, GATHER>, a, gs, splits);
}

template <bool GATHER>
static cudaError_t launch_small_g(const AttnArgs &a, const SmallGather &gs, int splits, cudaStream_t st) {
    switch ((a.T * a.G + 3) / 4) {
        case 1: return launch_small_t<1, GATHER>(a, gs, splits, st);
        case 2: return launch_small_t<2, GATHER>(a, gs, splits, st);
        case 3: return launch_small_t<3, GATHER>(a, gs, splits, st);
        case 4: return launch_small_t<4, GATHER>(a, gs, splits, st);
        case 5: return launch_small_t<5, GATHER>(a, gs, splits, st);
        case 6: return launch_small_t<6, GATHER>(a, gs, splits, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tree_attn_small(const AttnArgs &a, const SmallGather *gs, int splits, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    if (gs != nullptr) return launch_small_g<true>(a, *gs, splits, st);
    return launch_small_g<false>(a, SmallGather{}, splits, st);
}

}  // namespace ts
