// Split-KV tree-masked GQA attention on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators, TMA), for the TokenSwift verify pass: a batch
// of T >= 64 speculative rows (draft tree + n-gram chains) against the full
// bf16 KV cache ("fed into the LLM with a full KV cache", "How it works").
//
// Rows of one KV head g are the T x G pairs (t, j), t-major; an M-tile is
// tpb = floor(128/G) whole batch rows times the G query heads of the group,
// so every K/V byte staged in shared memory serves all G heads.  A CTA owns
// two M-tiles (256 rows) of one KV head and a contiguous range of 128-token
// KV tiles; the grid is (splits, M-tile pairs, Hkv) and the split partials
// are merged by the log-sum-exp merge kernel.
//
// Warp roles (320 threads):
//   warp 0      TMA producer: Q once, then K/V tiles into a 2-stage ring;
//   warp 1      owns TMEM (512 columns) and issues every tcgen05.mma from one
//               thread: S_m = Q_m K^T (SS, K-major), O_m += P_m V (TS, P from
//               TMEM, V MN-major);
//   warps 2-5   softmax warpgroup of M-tile 0 (thread = row);
//   warps 6-9   softmax warpgroup of M-tile 1.
// TMEM columns: S_0 [0,128) S_1 [128,256) O_0 [256,384) O_1 [384,512); P_m
// (bf16, two per column) overwrites the first 64 columns of S_m.
// The running max is updated lazily: O and l are rescaled only when a row's
// max grows by more than 2^8, which keeps every P below 256 and makes the
// (TMEM round-trip) rescale rare.  Every wait is bounded (see tc_ptx.cuh).
#include "internal.h"
#include "tc_ptx.cuh"
#include "ts_common.cuh"

namespace ts {

__device__ int g_device_error = 0;

namespace {

constexpr int TC_THREADS = 320;
constexpr int KV_TILE = 128;
constexpr int NSTAGE = 2;
constexpr int TILE_BYTES = 128 * 128 * 2;  // one 128 x 128 bf16 tile (two 64-column swizzled halves)
constexpr int HALF_BYTES = TILE_BYTES / 2;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units

struct __align__(8) TcSmemTail {
    uint64_t q_full;
    uint64_t k_full[NSTAGE], k_empty[NSTAGE];
    uint64_t v_full[NSTAGE], v_empty[NSTAGE];
    uint64_t s_full[2], p_full[2], o_done[2];
    uint64_t mma_done;
    uint64_t score_bar[2];       // G score rows arrive once per tile (by tile parity)
    uint32_t tmem_base;
    int abort_flag;
    float score_part[2][32][2];  // [tile parity][head j][chunk half]
};

constexpr size_t TC_SMEM_BYTES = 1024 /*alignment slack*/ + 2 * TILE_BYTES /*Q*/ + 2 * NSTAGE * TILE_BYTES /*K,V*/ +
                                 sizeof(TcSmemTail);

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void raise_abort(TcSmemTail *tl) {
    *(volatile int *)&tl->abort_flag = 1;
    atomicExch(&g_device_error, (int)TS_ERR_TIMEOUT);
}

}  // namespace

__global__ void __launch_bounds__(TC_THREADS, 1)
tree_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnArgs a, const int n_mtiles) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *sQ = base;                           // [2][TILE_BYTES]
    unsigned char *sK = sQ + 2 * TILE_BYTES;            // [NSTAGE][TILE_BYTES]
    unsigned char *sV = sK + NSTAGE * TILE_BYTES;       // [NSTAGE][TILE_BYTES]
    TcSmemTail *tl = reinterpret_cast<TcSmemTail *>(sV + NSTAGE * TILE_BYTES);
    volatile int *abort_flag = &tl->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, mp = blockIdx.y, g = blockIdx.z;
    const int G = a.G, tpb = a.tpb;
    const int mt0 = 2 * mp;
    const int nm = min(2, n_mtiles - mt0);  // M-tiles owned (1 or 2)
    const int tile_begin = split * a.tiles_per_split;
    const int n_my = min(a.n_tiles, tile_begin + a.tiles_per_split) - tile_begin;

    if (threadIdx.x == 0) {
        tc::mbar_init(&tl->q_full, 1);
        for (int s = 0; s < NSTAGE; ++s) {
            tc::mbar_init(&tl->k_full[s], 1);
            tc::mbar_init(&tl->k_empty[s], 1);
            tc::mbar_init(&tl->v_full[s], 1);
            tc::mbar_init(&tl->v_empty[s], 1);
        }
        for (int m = 0; m < 2; ++m) {
            tc::mbar_init(&tl->s_full[m], 1);
            tc::mbar_init(&tl->p_full[m], 128);
            tc::mbar_init(&tl->o_done[m], 1);
        }
        tc::mbar_init(&tl->mma_done, 1);
        tc::mbar_init(&tl->score_bar[0], (uint32_t)a.G);
        tc::mbar_init(&tl->score_bar[1], (uint32_t)a.G);
        tl->abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&tl->tmem_base, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = tl->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n_my > 0) {
            tc::prefetch_tmap(&tm_q);
            tc::prefetch_tmap(&tm_k);
            tc::prefetch_tmap(&tm_v);
            const uint32_t qbytes = (uint32_t)(2 * 128 * G * tpb);  // two 64-column halves of tpb*G rows
            tc::mbar_arrive_expect_tx(&tl->q_full, qbytes * nm);
            for (int m = 0; m < nm; ++m)
                for (int h = 0; h < 2; ++h)
                    tc::tma_load_3d(sQ + m * TILE_BYTES + h * HALF_BYTES, &tm_q, &tl->q_full, h * 64, g * G,
                                    (mt0 + m) * tpb);
            int nk = 0, nv = 0;  // K and V tiles issued
            for (int it = 0; it < n_my; ++it) {
                const int st = it % NSTAGE;
                const uint32_t ph = (uint32_t)(it / NSTAGE) & 1u;
                const int tok0 = (tile_begin + it) * KV_TILE;
                if (it >= NSTAGE && !tc::mbar_wait(&tl->k_empty[st], ph ^ 1u, abort_flag)) { raise_abort(tl); break; }
                tc::mbar_arrive_expect_tx(&tl->k_full[st], TILE_BYTES);
                for (int h = 0; h < 2; ++h)
                    tc::tma_load_3d(sK + st * TILE_BYTES + h * HALF_BYTES, &tm_k, &tl->k_full[st], h * 64, tok0, g);
                nk = it + 1;
                if (it >= NSTAGE && !tc::mbar_wait(&tl->v_empty[st], ph ^ 1u, abort_flag)) { raise_abort(tl); break; }
                tc::mbar_arrive_expect_tx(&tl->v_full[st], TILE_BYTES);
                for (int h = 0; h < 2; ++h)
                    tc::tma_load_3d(sV + st * TILE_BYTES + h * HALF_BYTES, &tm_v, &tl->v_full[st], h * 64, tok0, g);
                nv = it + 1;
            }
            // never leave with a copy in flight into this CTA's shared memory
            tc::mbar_wait(&tl->q_full, 0, nullptr);
            for (int it = max(0, nk - NSTAGE); it < nk; ++it)
                tc::mbar_wait(&tl->k_full[it % NSTAGE], (uint32_t)(it / NSTAGE) & 1u, nullptr);
            for (int it = max(0, nv - NSTAGE); it < nv; ++it)
                tc::mbar_wait(&tl->v_full[it % NSTAGE], (uint32_t)(it / NSTAGE) & 1u, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_my > 0) {
            const uint32_t id_s = tc::idesc_bf16_f32(128, 128, false);
            const uint32_t id_o = tc::idesc_bf16_f32(128, 128, true);
            bool ok = tc::mbar_wait(&tl->q_full, 0, abort_flag);
            for (int it = 0; ok && it < n_my; ++it) {
                const int st = it % NSTAGE;
                const uint32_t ph = (uint32_t)(it / NSTAGE) & 1u;
                if (!(ok = tc::mbar_wait(&tl->k_full[st], ph, abort_flag))) break;
                tc::fence_after_sync();
                const uint32_t kbase = tc::smem_u32(sK + st * TILE_BYTES);
                for (int m = 0; m < nm; ++m) {
                    const uint32_t qbase = tc::smem_u32(sQ + m * TILE_BYTES);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t off = (uint32_t)((k >> 2) * HALF_BYTES + (k & 3) * 32);
                        tc::mma_ss(tbase + m * 128, tc::smem_desc_sw128(qbase + off, 16, 1024),
                                   tc::smem_desc_sw128(kbase + off, 16, 1024), id_s, k > 0);
                    }
                    tc::mma_commit(&tl->s_full[m]);
                }
                tc::mma_commit(&tl->k_empty[st]);
                if (!(ok = tc::mbar_wait(&tl->v_full[st], ph, abort_flag))) break;
                const uint32_t vbase = tc::smem_u32(sV + st * TILE_BYTES);
                for (int m = 0; m < nm; ++m) {
                    if (!(ok = tc::mbar_wait(&tl->p_full[m], (uint32_t)it & 1u, abort_flag))) break;
                    tc::fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma_ts(tbase + 256 + m * 128, tbase + m * 128 + kk * 8,
                                   tc::smem_desc_sw128(vbase + kk * 2048, HALF_BYTES, 1024), id_o, (it > 0 || kk > 0));
                    tc::mma_commit(&tl->o_done[m]);
                }
                if (!ok) break;
                tc::mma_commit(&tl->v_empty[st]);
            }
            if (!ok) raise_abort(tl);
            // drain: every issued MMA completes before TMEM is released
            tc::mma_commit(&tl->mma_done);
            tc::mbar_wait(&tl->mma_done, 0, nullptr);
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        const int wg = (warp - 2) >> 2;          // 0 or 1: M-tile owned
        const int quad = warp & 3;               // TMEM lane quadrant this warp may access
        const int r = quad * 32 + lane;          // row inside the M-tile
        const uint32_t lane_addr = tbase + ((uint32_t)(quad * 32) << 16);
        const uint32_t s_col = (uint32_t)wg * 128, o_col = 256 + (uint32_t)wg * 128;
        if (wg < nm && n_my > 0) {
            const int mt = mt0 + wg;
            const int t = mt * tpb + r / G;
            const int j = r % G;
            const bool row_valid = r < tpb * G && t < a.T;
            uint64_t mk0 = 0, mk1 = 0;
            if (row_valid) {
                mk0 = a.mask[2 * t];
                mk1 = a.mask[2 * t + 1];
            }
            const bool score_wg = a.chunk_scores != nullptr && a.score_row / tpb == mt;
            const bool is_score_row = score_wg && row_valid && t == a.score_row;
            const bool is_score_reducer = score_wg && r == (a.score_row % tpb) * G;
            const float c = a.scale_log2;
            float m_run = -INFINITY, l_run = 0.f;
            bool ok = true;
            for (int it = 0; it < n_my; ++it) {
                const int tile = tile_begin + it;
                const int64_t tok0 = (int64_t)tile * KV_TILE;
                ok = tc::mbar_wait(&tl->s_full[wg], (uint32_t)it & 1u, abort_flag);
                if (!(ok = __all_sync(0xffffffffu, ok))) break;
                tc::fence_after_sync();
                // Tiles wholly inside the prefix need no mask; others test each token.
                const bool full_tile = tok0 + KV_TILE <= a.N;
                auto visible = [&](int64_t tok) -> bool {
                    if (tok < a.N) return true;
                    if (tok >= a.N + a.T) return false;
                    const int u = (int)(tok - a.N);
                    return ((u < 64 ? (mk0 >> u) : (mk1 >> (u - 64))) & 1ull) != 0;
                };
                // ---- pass 1: row max (raw q.k) and the fused chunk sums of the scoring row
                float mx = -INFINITY, s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t v[32];
                    tc::tmem_ld32(lane_addr + s_col + cc * 32, v);
                    tc::tmem_wait_ld();
                    if (row_valid) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float xv = __uint_as_float(v[i]);
                            const int64_t tok = tok0 + cc * 32 + i;
                            if (is_score_row && tok < a.N) {
                                if (cc < 2) s0 += xv; else s1 += xv;
                            }
                            if (full_tile || visible(tok)) mx = fmaxf(mx, xv);
                        }
                    }
                }
                if (is_score_row) {
                    tl->score_part[it & 1][j][0] = s0;
                    tl->score_part[it & 1][j][1] = s1;
                    tc::mbar_arrive(&tl->score_bar[it & 1]);
                }
                if (is_score_reducer) {
                    // the G score rows may sit in two warps: gather them through shared memory
                    if (tc::mbar_wait(&tl->score_bar[it & 1], (uint32_t)(it >> 1) & 1u, abort_flag)) {
                        for (int hh = 0; hh < 2; ++hh) {
                            const int64_t cidx = (int64_t)tile * 2 + hh;
                            if (cidx * 64 < a.N) {
                                float best = tl->score_part[it & 1][0][hh];
                                for (int jj = 1; jj < G; ++jj) best = fmaxf(best, tl->score_part[it & 1][jj][hh]);
                                a.chunk_scores[(size_t)g * a.n_chunks + cidx] = best;
                            }
                        }
                    } else {
                        raise_abort(tl);
                    }
                }
                const float m_new = fmaxf(m_run, mx * c);
                const bool resc = m_new > m_run + RESCALE_THRESHOLD;
                const float alpha = resc ? ex2(m_run - m_new) : 1.f;
                if (it > 0 && __any_sync(0xffffffffu, resc)) {
                    // O_m holds the previous tiles: wait for their P.V, then scale this warp's rows
                    ok = tc::mbar_wait(&tl->o_done[wg], (uint32_t)(it - 1) & 1u, abort_flag);
                    if (!(ok = __all_sync(0xffffffffu, ok))) break;
                    tc::fence_after_sync();
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t ov[32];
                        tc::tmem_ld32(lane_addr + o_col + cc * 32, ov);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tc::tmem_st32(lane_addr + o_col + cc * 32, ov);
                    }
                    tc::tmem_wait_st();
                }
                if (resc) {
                    l_run *= alpha;
                    m_run = m_new;
                }
                // ---- pass 2: P = 2^(s*c - m) in bf16 over the first 64 columns of S_m
                // (token k -> column k/2, even k in the lower half).  Chunk cc of S
                // lands in P columns [16cc, 16cc+16), all already read.
                const bool none_visible = (m_run == -INFINITY) || !row_valid;
                const float neg_m = none_visible ? 0.f : -m_run;
                float lsum = 0.f;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t v[32];
                    tc::tmem_ld32(lane_addr + s_col + cc * 32, v);
                    tc::tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int64_t tok = tok0 + cc * 32 + 2 * i;
                        float p0 = ex2(fmaf(__uint_as_float(v[2 * i]), c, neg_m));
                        float p1 = ex2(fmaf(__uint_as_float(v[2 * i + 1]), c, neg_m));
                        if (none_visible) { p0 = 0.f; p1 = 0.f; }
                        if (!full_tile) {
                            if (!visible(tok)) p0 = 0.f;
                            if (!visible(tok + 1)) p1 = 0.f;
                        }
                        lsum += p0 + p1;
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
                        pk[i] = *reinterpret_cast<uint32_t *>(&b2);
                    }
                    tc::tmem_st16(lane_addr + s_col + cc * 16, pk);
                }
                l_run += lsum;
                tc::tmem_wait_st();
                tc::fence_before_sync();
                tc::mbar_arrive(&tl->p_full[wg]);
            }
            // ---- epilogue: final O_m of this split
            if (ok) ok = tc::mbar_wait(&tl->o_done[wg], (uint32_t)(n_my - 1) & 1u, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                raise_abort(tl);
            } else {
                tc::fence_after_sync();
                const int h = g * G + j;
                const size_t row = (size_t)t * a.Hq + h;
                const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t ov[32];
                    tc::tmem_ld32(lane_addr + o_col + cc * 32, ov);
                    tc::tmem_wait_ld();
                    if (row_valid) {
                        if (a.splits == 1) {
                            uint32_t pk[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(ov[2 * i]) * inv,
                                                                          __uint_as_float(ov[2 * i + 1]) * inv);
                                pk[i] = *reinterpret_cast<uint32_t *>(&b2);
                            }
                            uint4 *dst = reinterpret_cast<uint4 *>(a.out + row * 128 + cc * 32);
#pragma unroll
                            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                        } else {
                            float4 *dst = reinterpret_cast<float4 *>(a.ws_o + ((size_t)split * a.T * a.Hq + row) * 128 + cc * 32);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                dst[i] = make_float4(__uint_as_float(ov[4 * i]), __uint_as_float(ov[4 * i + 1]),
                                                     __uint_as_float(ov[4 * i + 2]), __uint_as_float(ov[4 * i + 3]));
                        }
                    }
                }
                if (row_valid) {
                    if (a.splits == 1) {
                        if (a.lse != nullptr) a.lse[row] = (m_run + log2f(l_run)) * TS_LN2;
                    } else {
                        reinterpret_cast<float2 *>(a.ws_ml)[(size_t)split * a.T * a.Hq + row] = make_float2(m_run, l_run);
                    }
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tbase, 512);
    }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
size_t tc_smem_bytes() { return TC_SMEM_BYTES; }

TcPlan tc_plan(int T, int Hq, int Hkv, int d, int64_t N, int num_sms) {
    TcPlan p{};
    const int G = Hq / Hkv;
    p.ok = d == 128 && T >= 64 && T <= 128 && G <= 32;
    if (!p.ok) return p;
    p.tpb = 128 / G;
    p.n_mtiles = (T + p.tpb - 1) / p.tpb;
    p.n_mpairs = (p.n_mtiles + 1) / 2;
    p.n_tiles = (int)((N + T + KV_TILE - 1) / KV_TILE);
    const int base = Hkv * p.n_mpairs;
    int splits = num_sms / base;
    if (splits < 1) splits = 1;
    if (splits > p.n_tiles) splits = p.n_tiles;
    p.tiles_per_split = (p.n_tiles + splits - 1) / splits;
    p.splits = (p.n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    return p;
}

cudaError_t launch_tree_attn_tc(const AttnArgs &a, const TcPlan &p, const CUtensorMap &tq, const CUtensorMap &tk,
                                const CUtensorMap &tv, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(tree_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)TC_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(p.splits, p.n_mpairs, a.Hkv);
    tree_attn_tc_kernel<<<grid, TC_THREADS, TC_SMEM_BYTES, st>>>(tq, tk, tv, a, p.n_mtiles);
    return cudaGetLastError();
}

cudaError_t read_device_error(int *value, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
    if (e != cudaSuccess || !clear) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace ts
