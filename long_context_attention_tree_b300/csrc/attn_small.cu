// Split-KV tree-masked GQA attention on the CUDA cores for small batches:
// at most 24 (batch row, query head) pairs per KV head, head dim 128.  This
// is the shape of the TokenSwift self-drafting pass ("How it works": the
// target model with a partial KV cache drafts the next tokens), e.g. 4 chain
// rows x 5 query heads over a 4096-token partial cache.
//
// The work is fp32 FMAs (about 1 FMA per 1.5 bytes of K/V), so the kernel is
// built to keep the FMA pipe busy with packed fp32x2 FMAs and few other
// instructions per FMA, with four warps per scheduler to hide latencies.
//
// CTA = (KV head g, 256-token KV range) = eight 32-token blocks, sixteen
// warps, one CTA per SM (a range's K/V fill 128 KB of shared memory; half as
// many ranges as with 128-token CTAs, two per SM, which leaves the split
// merge half the partials at the same kernel time):
// warp (b, h) = (w / 2, w % 2) owns dims 64h .. 64h+63 of block b from the
// load to its partial result.  Rows r = (t, j) t-major, R = T*G, padded to
// 4 RG (RG = ceil(R/4)).
//   load:  each warp copies its half of the block's 32 K rows and 32 V rows
//          into shared memory with 16-byte cp.async (K XOR-swizzled by
//          16-byte chunk within each 128-byte half row, so that a quarter-warp
//          reading one chunk of eight rows hits eight banks); rows out of range
//          or not gathered are zero-filled.  Q comes first (prefetched into L2
//          before the kernel waits for its predecessor, then its own copy
//          group, waited for before the K/V copies go out) and is converted to
//          fp32 [dim/4][row slot][4].
//   S:     lane (rg, tg) = (lane / 8, lane % 8) takes rows rg*RG .. +RG-1 and
//          tokens tg + 8i (i < 4) of the block: per 8 dims of its half it reads
//          four K chunks and 2 RG Q quads and issues 16 RG fp32x2 FMAs over
//          dimension pairs.  The two warps of a block swap their half sums
//          through shared memory (a 64-thread named barrier), so both hold S.
//   softmax: both warps compute the block's row max, P and row sum (the same
//          arithmetic, so the same values); each writes half of the rows' P to
//          the block's slab as (p, p) pairs.
//   O:     lane (rh, dg) = (lane / 16, lane % 16) takes rows rh*2RG .. +2RG-1
//          and dims 64h + 4dg .. +3: per token one 8-byte V read, RG 16-byte P
//          reads and 4 RG fp32x2 FMAs.
//   combine: the eight blocks' partials (m, l, O) are merged through shared
//          memory (over the dead K/V buffers) into the range's partial, which
//          goes to the split workspace for the log-sum-exp merge kernel (a
//          single range writes the normalised output directly).
// The chunk importance of the scoring row can be produced by the same pass
// (a block holds half a 64-token chunk).
//
// Gather variant: the prefix rows are not read from a compact cache but from
// the chunks of the full cache that the top-k selection chose (position p of
// the compact cache is row sel[g][p/64]*64 + p%64 of the full cache); each
// warp also writes its gathered half rows into the compact cache, so the
// refresh of the partial cache (selection, gather) and the drafting pass over
// it read the selected K/V bytes from HBM once.
#include "internal.h"
#include "topk_radix.cuh"
#include "ts_common.cuh"

namespace ts {

namespace {
constexpr int D = 128;
constexpr int WT = 32;              // tokens per block
constexpr int NBLK = 8;             // blocks per CTA
constexpr int NWARP = 2 * NBLK;     // two warps (dimension halves) per block
constexpr int NTHR = NWARP * 32;
constexpr int RANGE = NBLK * WT;    // tokens per CTA: four 64-token chunks
constexpr int CPR = NBLK / 2;       // chunks per range
constexpr int ROWB = D * 2;         // bytes of one K/V row
constexpr int HALFB = ROWB / 2;     // bytes of one half row (64 dims)

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// The two bf16 halves of a word as an fp32 pair (low half first), by byte
// permutes: each half moves to the upper 16 bits of a zeroed word.
__device__ __forceinline__ float2 bf16x2_f2(uint32_t w) {
    uint32_t lo, hi;
    asm("prmt.b32 %0, %1, %2, 0x1044;" : "=r"(lo) : "r"(w), "r"(0u));
    asm("prmt.b32 %0, %1, %2, 0x3244;" : "=r"(hi) : "r"(w), "r"(0u));
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}

// 2^x on the special-function unit (ex2.approx: relative error about 2^-22;
// subnormal results flush to zero)
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The two warps of block b (named barrier 1 + b, 64 threads).
__device__ __forceinline__ void pair_sync(int b) { asm volatile("bar.sync %0, 64;" ::"r"(1 + b) : "memory"); }

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
    static constexpr size_t SMEM = P_OFF + (size_t)NBLK * WT * PP * 8;
    static_assert((size_t)NBLK * RP * D * 4 <= 2 * (size_t)RANGE * ROWB, "block partials must fit the K/V buffers");
    static_assert((size_t)RG * 32 * 16 <= (size_t)WT * HALFB, "half sums must fit a warp's K half");
    static_assert((size_t)RP * ROWB <= (size_t)NBLK * WT * PP * 8, "Q staging must fit the P slabs");
};
}  // namespace

template <int RG, bool GATHER, bool SELECT>
__global__ void __launch_bounds__(NTHR, 1) tree_attn_small_kernel(const AttnArgs a, const SmallGather gs, int n_splits) {
    using C = SmallCfg<RG>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char *sK = smem_raw + C::K_OFF;
    unsigned char *sV = smem_raw + C::V_OFF;
    float *sQ = reinterpret_cast<float *>(smem_raw + C::Q_OFF);
    float *sP = reinterpret_cast<float *>(smem_raw + C::P_OFF);
    __shared__ float red_m[NBLK][C::RP], red_l[NBLK][C::RP];  // per block: row max and row sum
    __shared__ float row_m[C::RP], row_l[C::RP];              // the range's
    __shared__ float sc_part[NBLK][32];                       // scoring row: half-chunk sums per head
    __shared__ uint64_t s_mask[24];                           // batch rows' mask words

    // Q into L2 while the previous kernel finishes (a prefetch is only a hint:
    // a line that a later write replaces is replaced in L2 too)
    for (int e = threadIdx.x; e < 2 * a.T * a.G; e += NTHR) {
        const int r = e >> 1;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a.q + ((size_t)(r / a.G) * a.Hq + blockIdx.y * a.G + r % a.G) * D +
                                                      (e & 1) * 64));
    }
    // a programmatic dependent: the previous kernel (the selection, the gather
    // of the partial cache) has completed and its writes are visible past here
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int b = w >> 1, hd = w & 1;                  // block, dimension half
    const int split = blockIdx.x, g = blockIdx.y;
    const int G = a.G, R = a.T * G;
    const int64_t Np = a.N, L = Np + a.T;            // prefix positions, all positions
    const int64_t t0 = (int64_t)split * RANGE;
    const int64_t wb = t0 + (int64_t)b * WT;          // first position of this warp's block
    const bool active = wb < L;                       // the same for both warps of a block
    const int64_t plen = GATHER ? Np : prefix_of(a, g);
    // gather: the full-cache chunk behind this block (a block lies in one
    // chunk: Np is a multiple of 64 there)
    int64_t src_base = 0;
    if (GATHER && !SELECT && wb < Np) {
        const int c = min(max(gs.sel[(size_t)g * gs.k_sel + (int)(wb >> 6)], 0), gs.n_chunks - 1);
        src_base = (int64_t)c * 64 + (wb & 63);
    }
    if (threadIdx.x < NBLK * 32) sc_part[threadIdx.x >> 5][lane] = 0.f;

    // ---- the batch rows' mask words (T <= 24 rows and tail tokens: word 0)
    // and Q of the group (copy group 0, staged as bf16 in the P slabs) ahead
    // of the K/V copies
    uint64_t mword = 0;
    if (threadIdx.x < a.T) mword = a.mask[(size_t)threadIdx.x * a.mw];
    unsigned char *sQb = reinterpret_cast<unsigned char *>(sP);  // [RP][256 B] until S starts
    for (int e = threadIdx.x; e < C::RP * 16; e += NTHR) {
        const int r = e >> 4, c8 = e & 15;
        size_t off = 0;
        if (r < R) off = ((size_t)(r / G) * a.Hq + g * G + r % G) * D + c8 * 8;
        cp_async16_zfill(sQb + r * ROWB + c8 * 16, a.q + off, r < R);
    }
    cp_async_commit();
    if (SELECT) {
        // this head's top-k chunks (the keys over the K/V buffers, which no
        // copy has touched yet): the range's four chunks, and the full list
        // and gathered length from the CTAs of the first range
        __shared__ TopkSmem tsm;
        __shared__ int s_chunk[CPR];
        const int pos0 = CPR * split;
        const bool last_taken = radix_topk_ascending<NTHR>(
            gs.scores + (size_t)g * gs.n_chunks, gs.n_chunks, gs.k_sel, gs.n_sink, gs.n_recent,
            reinterpret_cast<uint32_t *>(sK), tsm, [&](int pos, int c) {
                if (split == 0) gs.sel_out[(size_t)g * gs.k_sel + pos] = c;
                if (pos >= pos0 && pos < pos0 + CPR) s_chunk[pos - pos0] = c;
            });
        const int per = (gs.n_chunks + NTHR - 1) / NTHR;
        if (split == 0 && gs.part_len_out != nullptr && (int)threadIdx.x == (gs.n_chunks - 1) / per) {
            const int64_t tail = gs.N - (int64_t)(gs.n_chunks - 1) * 64;  // tokens of the last chunk, 1..64
            gs.part_len_out[g] = gs.k_sel * 64 - (last_taken ? (int)(64 - tail) : 0);
        }
        __syncthreads();  // the range's chunks are known; the keys are dead
        if (wb < Np) src_base = (int64_t)s_chunk[b >> 1] * 64 + (wb & 63);
    }
    // Q is waited for before the K/V copies go out: behind them it would land
    // only when most of the grid's K/V has (the whole grid asks for its K/V at
    // once), and no warp can start before Q is in place
    if (threadIdx.x < a.T) s_mask[threadIdx.x] = mword;
    cp_async_wait<0>();
    __syncthreads();

    // ---- this warp's half of its block's K rows (group 1) and V rows (group 2)
    // lane: 16-byte chunk lane % 8 of the half, rows lane / 8 + 4u
    {
        const int c = lane & 7;
        size_t off[8];
        bool ok[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int rl = (lane >> 3) + 4 * u;
            const int64_t p = wb + rl;
            ok[u] = false;
            off[u] = 0;
            if (p < Np) {
                if (GATHER) {
                    const int64_t src = src_base + rl;
                    ok[u] = src < gs.N;
                    off[u] = ((size_t)g * gs.ld + (size_t)src) * D + hd * 64 + c * 8;
                } else {
                    ok[u] = p < plen;
                    off[u] = ((size_t)g * a.ld_kv + (size_t)p) * D + hd * 64 + c * 8;
                }
            } else if (p < L) {
                ok[u] = true;
                off[u] = ((size_t)g * a.ld_kv + (size_t)p) * D + hd * 64 + c * 8;
            }
        }
        const __nv_bfloat16 *ksrc = (GATHER && wb < Np) ? gs.k : a.k;
        const __nv_bfloat16 *vsrc = (GATHER && wb < Np) ? gs.v : a.v;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int rho = b * WT + (lane >> 3) + 4 * u;
            cp_async16_zfill(sK + rho * ROWB + hd * HALFB + ((c ^ (rho & 7)) << 4), ksrc + (ok[u] ? off[u] : 0),
                             ok[u]);
        }
        cp_async_commit();
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int rho = b * WT + (lane >> 3) + 4 * u;
            cp_async16_zfill(sV + rho * ROWB + hd * HALFB + (c << 4), vsrc + (ok[u] ? off[u] : 0), ok[u]);
        }
        cp_async_commit();
    }

    // ---- Q -> fp32 [dim/4][slot][4]; row r in slot (r / RG) * QS + r % RG
    // (padding rows zero)
    for (int e = threadIdx.x; e < C::RP * 16; e += NTHR) {
        const int r = e >> 4, c8 = e & 15;
        const uint4 x = *reinterpret_cast<const uint4 *>(sQb + r * ROWB + c8 * 16);
        const int slot = (r / RG) * C::QS + r % RG;
        float4 *dst = reinterpret_cast<float4 *>(sQ);
        dst[(2 * c8) * C::QSLOTS + slot] = make_float4(bf16_lo(x.x), bf16_hi(x.x), bf16_lo(x.y), bf16_hi(x.y));
        dst[(2 * c8 + 1) * C::QSLOTS + slot] = make_float4(bf16_lo(x.z), bf16_hi(x.z), bf16_lo(x.w), bf16_hi(x.w));
    }
    __syncthreads();  // Q and the zeroed score slots are visible; the staging is dead

    cp_async_wait<1>();  // this lane's K copies have landed ...
    __syncwarp();        // ... and every lane's of the warp

    // gather: the warp's K half rows into the compact cache (rows that exist)
    if (GATHER && wb < Np) {
        const int c = lane & 7;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int rl = (lane >> 3) + 4 * u, rho = b * WT + rl;
            if (src_base + rl < gs.N) {
                const uint4 x = *reinterpret_cast<const uint4 *>(sK + rho * ROWB + hd * HALFB + ((c ^ (rho & 7)) << 4));
                *reinterpret_cast<uint4 *>(gs.k_dst + ((size_t)g * a.ld_kv + (size_t)(wb + rl)) * D + hd * 64 + c * 8) = x;
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
    float *pw = sP + (size_t)b * WT * C::PP * 2;  // the block's P slab [token][row][(p, p)]
    if (active) {
        // ---- S over this warp's 64 dims for rows rg*RG + i, tokens tg + 8j:
        // acc[i][j] holds the even- and odd-dimension partial sums
        float2 acc[RG][4];
#pragma unroll
        for (int i = 0; i < RG; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.f, 0.f);
        unsigned char *kb = sK + (b * WT + tg) * ROWB + hd * HALFB;  // token tg; + 8j rows (row & 7 = tg)
        const float4 *qb = reinterpret_cast<const float4 *>(sQ) + (size_t)(16 * hd) * C::QSLOTS + rg * C::QS;
#pragma unroll 2
        for (int c = 0; c < 8; ++c) {
            uint4 kw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) kw[j] = *reinterpret_cast<const uint4 *>(kb + j * 8 * ROWB + ((c ^ tg) << 4));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float4 q4[RG];
#pragma unroll
                for (int i = 0; i < RG; ++i) q4[i] = qb[(2 * c + h) * C::QSLOTS + i];
                float2 k0[4], k1[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    k0[j] = bf16x2_f2(h ? kw[j].z : kw[j].x);  // dims 8c + 4h, +1 of the half
                    k1[j] = bf16x2_f2(h ? kw[j].w : kw[j].y);  // dims 8c + 4h + 2, +3
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int i = 0; i < RG; ++i) acc[i][j] = ffma2(k0[j], make_float2(q4[i].x, q4[i].y), acc[i][j]);
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int i = 0; i < RG; ++i) acc[i][j] = ffma2(k1[j], make_float2(q4[i].z, q4[i].w), acc[i][j]);
            }
        }
        // ---- swap half sums with the block's other warp through this warp's
        // (consumed) K half rows: slot-major [RG][lane][4 tokens]
        float s[RG][4];
        float4 *xs_mine = reinterpret_cast<float4 *>(kb - tg * ROWB);  // the warp's K half, row 0 of the block
#pragma unroll
        for (int i = 0; i < RG; ++i) {
            const float4 v4 = make_float4(acc[i][0].x + acc[i][0].y, acc[i][1].x + acc[i][1].y,
                                          acc[i][2].x + acc[i][2].y, acc[i][3].x + acc[i][3].y);
            s[i][0] = v4.x; s[i][1] = v4.y; s[i][2] = v4.z; s[i][3] = v4.w;
        }
        // the swap area of a warp: WT rows of HALFB bytes at stride ROWB, i.e. 8
        // float4 per row; slot q lies in row q / 8, float4 q % 8
        __syncwarp();  // every lane's K reads are done
#pragma unroll
        for (int i = 0; i < RG; ++i) {
            const int q = i * 32 + lane;
            xs_mine[(q >> 3) * (ROWB / 16) + (q & 7)] = make_float4(s[i][0], s[i][1], s[i][2], s[i][3]);
        }
        pair_sync(b);
        const float4 *xs_other = reinterpret_cast<const float4 *>(sK + (b * WT) * ROWB + (hd ^ 1) * HALFB);
        // the sum in a fixed order (half 0 + half 1), so both warps hold the same S
#pragma unroll
        for (int i = 0; i < RG; ++i) {
            const int q = i * 32 + lane;
            const float4 o4 = xs_other[(q >> 3) * (ROWB / 16) + (q & 7)];
            if (hd == 0) {
                s[i][0] += o4.x; s[i][1] += o4.y; s[i][2] += o4.z; s[i][3] += o4.w;
            } else {
                s[i][0] = o4.x + s[i][0]; s[i][1] = o4.y + s[i][1]; s[i][2] = o4.z + s[i][2]; s[i][3] = o4.w + s[i][3];
            }
        }

        // ---- fused chunk importance of the scoring row (raw q.k over the
        // prefix): the block's half-chunk sum per head
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
                if (hd == 0 && tg == 0 && r < R && r / G == a.score_row) sc_part[b][r % G] = x;
            }
        }

        // ---- visibility, scale, the block's row max.  A prefix token's
        // visibility is the same for every row; a batch token's (tail block
        // only) is the row's mask bit.
        const float cs = a.scale_log2;
        const bool tail_block = wb + WT > Np;  // the block reaches the batch's own tokens
        bool tok_ok[4];
        int tail_u[4];                         // batch token index, or -1 past the batch
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t p = wb + tg + 8 * j;
            tok_ok[j] = p < Np && (GATHER ? (src_base + tg + 8 * j < gs.N) : (p < plen));
            tail_u[j] = (p >= Np && p < L) ? (int)(p - Np) : -1;
        }
#pragma unroll
        for (int i = 0; i < RG; ++i) {
            const int r = rg * RG + i;
            const bool row_ok = r < R;
            const uint64_t mrow = (tail_block && row_ok) ? s_mask[r / G] : 0ull;
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                bool vis = row_ok && tok_ok[j];
                if (tail_block) vis = vis || (tail_u[j] >= 0 && ((mrow >> tail_u[j]) & 1ull));
                s[i][j] = vis ? s[i][j] * cs : -INFINITY;
                mx = fmaxf(mx, s[i][j]);
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            m[i] = mx;
        }
        // ---- P = 2^(s*c - m); this warp writes row groups 2hd, 2hd + 1 of the
        // block's slab as (p, p); the block's row sums
        const bool writer = (rg >> 1) == hd;
#pragma unroll
        for (int i = 0; i < RG; ++i) {
            float ls = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float pv = (m[i] == -INFINITY) ? 0.f : fast_exp2(s[i][j] - m[i]);
                ls += pv;
                if (writer)
                    *reinterpret_cast<float2 *>(pw + ((size_t)(tg + 8 * j) * C::PP + rg * RG + i) * 2) =
                        make_float2(pv, pv);
            }
            ls += __shfl_xor_sync(0xffffffffu, ls, 1);
            ls += __shfl_xor_sync(0xffffffffu, ls, 2);
            ls += __shfl_xor_sync(0xffffffffu, ls, 4);
            l[i] = ls;
        }
    }
    if (hd == 0 && tg == 0) {
#pragma unroll
        for (int i = 0; i < RG; ++i) {
            red_m[b][rg * RG + i] = m[i];
            red_l[b][rg * RG + i] = l[i];
        }
    }

    cp_async_wait<0>();  // V has landed (this lane's copies) ...
    __syncwarp();        // ... and every lane's

    if (GATHER && wb < Np) {
        const int c = lane & 7;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int rl = (lane >> 3) + 4 * u, rho = b * WT + rl;
            if (src_base + rl < gs.N) {
                const uint4 x = *reinterpret_cast<const uint4 *>(sV + rho * ROWB + hd * HALFB + (c << 4));
                *reinterpret_cast<uint4 *>(gs.v_dst + ((size_t)g * a.ld_kv + (size_t)(wb + rl)) * D + hd * 64 + c * 8) = x;
            }
        }
    }

    // ---- O over the block's 32 tokens: rows rh*2RG + i2, dims 64hd + 4dg .. +3
    const int rh = lane >> 4, dg = lane & 15;
    float2 o[2 * RG][2];
#pragma unroll
    for (int i = 0; i < 2 * RG; ++i) o[i][0] = o[i][1] = make_float2(0.f, 0.f);
    if (active) {
        pair_sync(b);  // the block's P (both warps' rows) is visible
        const unsigned char *vb = sV + (b * WT) * ROWB + hd * HALFB + dg * 8;
        const float *pb = pw + rh * 2 * RG * 2;
#pragma unroll 4
        for (int tw = 0; tw < WT; ++tw) {
            const uint2 vw = *reinterpret_cast<const uint2 *>(vb + tw * ROWB);
            const float2 v0 = bf16x2_f2(vw.x), v1 = bf16x2_f2(vw.y);
#pragma unroll
            for (int i = 0; i < RG; ++i) {
                const float4 pp = *reinterpret_cast<const float4 *>(pb + ((size_t)tw * C::PP + 2 * i) * 2);
                const float2 pa = make_float2(pp.x, pp.y), pc = make_float2(pp.z, pp.w);
                o[2 * i][0] = ffma2(pa, v0, o[2 * i][0]);
                o[2 * i][1] = ffma2(pa, v1, o[2 * i][1]);
                o[2 * i + 1][0] = ffma2(pc, v0, o[2 * i + 1][0]);
                o[2 * i + 1][1] = ffma2(pc, v1, o[2 * i + 1][1]);
            }
        }
    }
    __syncthreads();  // every block's (m, l) and score sums are written; K and V are dead

    if (a.chunk_scores != nullptr && threadIdx.x < CPR) {
        const int64_t ch0 = t0 + 64 * threadIdx.x;
        if (ch0 < Np) {
            float best = -INFINITY;
            for (int j = 0; j < G; ++j) best = fmaxf(best, sc_part[2 * threadIdx.x][j] + sc_part[2 * threadIdx.x + 1][j]);
            a.chunk_scores[(size_t)g * a.n_chunks + (size_t)(ch0 / 64)] = best;
        }
    }

    // ---- combine the eight block partials: each warp scales its O by
    // 2^(m_b - M) and parks it over the K/V buffers as fp32 [block][row][dim]
    float *sO = reinterpret_cast<float *>(smem_raw);
#pragma unroll
    for (int i2 = 0; i2 < 2 * RG; ++i2) {
        const int r = rh * 2 * RG + i2;
        float M = red_m[0][r];
#pragma unroll
        for (int x = 1; x < NBLK; ++x) M = fmaxf(M, red_m[x][r]);
        const float mb = red_m[b][r];
        const float f = (mb == -INFINITY) ? 0.f : fast_exp2(mb - M);
        *reinterpret_cast<float4 *>(sO + ((size_t)b * C::RP + r) * D + hd * 64 + dg * 4) =
            make_float4(o[i2][0].x * f, o[i2][0].y * f, o[i2][1].x * f, o[i2][1].y * f);
        if (w == 0 && dg == 0) {
            float Ls = 0.f;
#pragma unroll
            for (int x = 0; x < NBLK; ++x)
                if (red_m[x][r] != -INFINITY) Ls += fast_exp2(red_m[x][r] - M) * red_l[x][r];
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
        for (int x = 0; x < NBLK; ++x) {
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

template <int RG, bool GATHER, bool SELECT>
static cudaError_t launch_small_t(const AttnArgs &a, const SmallGather &gs, int splits, cudaStream_t st) {
    const size_t smem = SmallCfg<RG>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(tree_attn_small_kernel<RG, GATHER, SELECT>,
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
    return cudaLaunchKernelEx(&cfg, tree_attn_small_kernel<RG, GATHER, SELECT>, a, gs, splits);
}

template <bool GATHER, bool SELECT>
static cudaError_t launch_small_g(const AttnArgs &a, const SmallGather &gs, int splits, cudaStream_t st) {
    switch ((a.T * a.G + 3) / 4) {
        case 1: return launch_small_t<1, GATHER, SELECT>(a, gs, splits, st);
        case 2: return launch_small_t<2, GATHER, SELECT>(a, gs, splits, st);
        case 3: return launch_small_t<3, GATHER, SELECT>(a, gs, splits, st);
        case 4: return launch_small_t<4, GATHER, SELECT>(a, gs, splits, st);
        case 5: return launch_small_t<5, GATHER, SELECT>(a, gs, splits, st);
        case 6: return launch_small_t<6, GATHER, SELECT>(a, gs, splits, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tree_attn_small(const AttnArgs &a, const SmallGather *gs, int splits, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    if (gs != nullptr && gs->scores != nullptr) return launch_small_g<true, true>(a, *gs, splits, st);
    if (gs != nullptr) return launch_small_g<true, false>(a, *gs, splits, st);
    return launch_small_g<false, false>(a, SmallGather{}, splits, st);
}

}  // namespace ts
