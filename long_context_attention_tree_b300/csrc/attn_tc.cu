// Split-KV tree-masked GQA attention on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators, TMA), for the TokenSwift verify pass: a batch
// of T >= 64 speculative rows (draft tree + n-gram chains) against the full
// bf16 KV cache (the drafts are checked by the target model over its whole KV
// cache, "How it works" on the TokenSwift tool listing).
//
// Rows of one KV head g are the T x G pairs (t, j), t-major; an M-tile is
// tpb = floor(128/G) whole batch rows times the G query heads of the group,
// so every K/V byte staged in shared memory serves all G heads.  A CTA owns
// one or two M-tiles of one KV head (a pair stream or a single stream) and a
// contiguous range of 64-token KV tiles.
//
// KV tiles are 64 tokens (one scoring chunk), so TMEM holds two S buffers per
// M-tile: S(m, 0) S(m, 1) (64 columns each) and O(m) (128 columns); for a
// pair stream that is 4 x 64 + 2 x 128 = all 512 columns.  With S double
// buffered the MMAs of tile i+1's S run while the softmax of tile i works,
// so an M-tile's chain is no longer softmax -> P.V -> next S -> softmax: the
// issuer computes S(i+1) of both M-tiles, then P.V(i) of each as its P lands.
// The split counts are chosen on the host so that every CTA carries about
// the same tensor-core work; the partials are combined by the log-sum-exp
// merge kernel.
//
// Per KV tile and M-tile: S = Q K^T (8 MMAs, M=128 N=64 K=16, operands
// K-major in shared memory), softmax, O += P V (4 MMAs, M=128 N=128 K=16, P
// read from TMEM, V MN-major in shared memory).  Every MMA descriptor is
// precomputed, so the issuing thread only adds constants.
//
// Warp roles (384 threads, three warpgroups):
//   warp 0      TMA producer: Q once, then K and V tiles into 4-stage rings;
//   warp 1      owns TMEM (512 columns); one thread issues every tcgen05.mma;
//   warp 2      chunk-score reducer: takes the scoring rows' chunk sums from a
//               shared-memory ring and writes the max over the group's heads;
//   warp 3      idle;
//   warps 4-7   softmax warpgroup 0 (thread = row of M-tile 0);
//   warps 8-11  softmax warpgroup 1 (M-tile 1 of a pair stream).
// A softmax thread loads its row of S (64 fp32) into registers and writes
// P = 2^(s*c - m) as bf16 over the first 32 columns of that S buffer.  The
// running max is lazy: O and l are rescaled only when a row's max grows by
// more than 2^20 (P stays below 2^20, far inside bf16 and fp32 range), so the
// TMEM round trip of a rescale is rare.  The normaliser l sums the
// bf16-rounded weights that the P.V product uses.  The chunk importance of
// the scoring row is summed from the same S values and handed to warp 2, so
// the softmax warps never wait for the reduction.
// Every wait is bounded (see tc_ptx.cuh): a wait that gives up raises the
// CTA's abort flag and the sticky device status word, and the CTA winds down.
#include "internal.h"
#include "tc_ptx.cuh"
#include "ts_common.cuh"

namespace ts {

__device__ int g_device_error = 0;

namespace {

constexpr int TC_THREADS = 384;  // 168 registers per thread (3 warps per SM sub-partition)
constexpr int KV_TILE = TC_KV_TILE;           // 64 tokens: one scoring chunk
constexpr int Q_TILE_BYTES = 128 * 128 * 2;   // 128 rows x 128 dims, two 64-column swizzled halves
constexpr int Q_HALF_BYTES = Q_TILE_BYTES / 2;
constexpr int KV_TILE_BYTES = KV_TILE * 128 * 2;  // 64 tokens x 128 dims
constexpr int KV_HALF_BYTES = KV_TILE_BYTES / 2;
constexpr int NSTAGE = 4;                     // K and V ring depth
constexpr int SMEM_DATA_BYTES = 2 * Q_TILE_BYTES + 2 * NSTAGE * KV_TILE_BYTES;  // 192 KB
constexpr float RESCALE_THRESHOLD = 20.0f;    // log2 units
constexpr int SCORE_RING = 4;                 // chunk-score slots between the scoring rows and warp 2

struct __align__(8) TcSmemTail {
    uint64_t q_full;
    uint64_t k_full[NSTAGE], k_empty[NSTAGE];
    uint64_t v_full[NSTAGE], v_empty[NSTAGE];
    // [M-tile][S buffer]: completion n of a buffer is tile 2n + b, parity n & 1
    uint64_t s_full[2][2], p_full[2][2];
    uint64_t o_done[2];   // one commit per tile: the P.V of tile i completes phase i
    uint64_t o_final[2];  // one commit after the last P.V of the M-tile (epilogue)
    uint64_t mma_done;
    // Chunk scores: the G scoring rows put their chunk sum of a KV tile into a
    // ring slot (tile & 3); warp 2 takes the max over the group's heads.
    uint64_t score_full[SCORE_RING], score_empty[SCORE_RING];
    float score_sum[SCORE_RING][32];  // [slot][head j]
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t TC_SMEM_BYTES = 1024 /*alignment slack*/ + (size_t)SMEM_DATA_BYTES + sizeof(TcSmemTail);
static_assert(TC_SMEM_BYTES <= 232448, "shared memory above the 227 KB per-block limit");

// Per-launch constants derived from the host plan.
struct TcLaunch {
    int tpb, n_mtiles, n_pair, s_pair, s_single, tl_pair, tl_single, n_tiles, ctas_per_head;
    int direct;  // 1: every stream has one split, write the normalised output directly
};

__device__ __forceinline__ void raise_abort(TcSmemTail *tl) {
    *(volatile int *)&tl->abort_flag = 1;
    atomicExch(&g_device_error, (int)TS_ERR_TIMEOUT);
}

// Descriptors of swizzled tile halves, as 64-bit values to which a byte
// offset >> 4 is added directly (the 14-bit start field cannot overflow
// inside the 227 KB shared-memory window).
__device__ __forceinline__ uint64_t desc_k(uint32_t addr) { return tc::smem_desc_sw128(addr, 16, 1024); }
__device__ __forceinline__ uint64_t desc_mn(uint32_t addr) { return tc::smem_desc_sw128(addr, KV_HALF_BYTES, 1024); }
__device__ __forceinline__ uint64_t dplus(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

// S[128 x 64] = Q[128 x 128] K^T: 8 MMAs with K = 16 over the head dim.
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint64_t dq, uint64_t dk, uint32_t idesc) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t col = (uint32_t)((k & 3) * 32);
        tc::mma_ss(d_tmem, dplus(dq, (uint32_t)(k >> 2) * Q_HALF_BYTES + col),
                   dplus(dk, (uint32_t)(k >> 2) * KV_HALF_BYTES + col), idesc, k > 0);
    }
}
// O[128 x 128] += P[128 x 64 tokens] V[64 tokens x 128]: 4 MMAs with K = 16 tokens.
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint64_t dv, uint32_t idesc, bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        tc::mma_ts(o_tmem, p_tmem + kk * 8, dplus(dv, (uint32_t)kk * 2048), idesc, (accumulate || kk > 0) ? 1u : 0u);
}

// Softmax helpers on one 32-token chunk of a row of S held in registers.
// Hide tokens this row may not see: prefix tokens at or past the head's
// prefix length plen (<= N), batch tokens whose row is not an
// ancestor-or-self (mask bits), tokens past the batch.
// mrow is the row's mask (uint64 words), or null for a padding row, which
// sees no batch token; a 32-token chunk touches at most two of its words.
__device__ __forceinline__ void mask_chunk(uint32_t (&x)[32], int64_t tok0, int64_t plen, int64_t N, int T,
                                           const uint64_t *mrow) {
    const int64_t u0 = tok0 - N;  // batch index of the chunk's first token (may be negative)
    uint64_t wa = 0, wb = 0;
    int wbase = 0;
    if (mrow != nullptr && u0 + 32 > 0 && u0 < T) {
        const int ufirst = u0 > 0 ? (int)u0 : 0;
        const int ulast = u0 + 31 < T - 1 ? (int)(u0 + 31) : T - 1;
        wbase = ufirst >> 6;
        wa = mrow[wbase];
        if ((ulast >> 6) != wbase) wb = mrow[wbase + 1];
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int64_t tok = tok0 + i;
        bool vis = tok < plen;
        if (tok >= N && tok < N + T) {
            const int u = (int)(tok - N);
            vis = ((((u >> 6) == wbase ? wa : wb) >> (u & 63)) & 1ull) != 0;
        }
        if (!vis) x[i] = __float_as_uint(-INFINITY);
    }
}
__device__ __forceinline__ float max_chunk(const uint32_t (&x)[32]) {
    float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
        m0 = tc::fmax3(m0, __uint_as_float(x[i + 0]), __uint_as_float(x[i + 1]));
        m1 = tc::fmax3(m1, __uint_as_float(x[i + 2]), __uint_as_float(x[i + 3]));
        m2 = tc::fmax3(m2, __uint_as_float(x[i + 4]), __uint_as_float(x[i + 5]));
        m3 = tc::fmax3(m3, __uint_as_float(x[i + 6]), __uint_as_float(x[i + 7]));
    }
    return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}
// P = 2^(x*c - m) for 32 tokens -> 16 packed bf16x2 words (even token in the
// lower half); returns the fp32 sum of the 32 bf16-rounded values, so that the
// normaliser sums exactly the weights the P.V product uses (a row dominated
// by one key then reproduces that key's value without the weight's rounding).
__device__ __forceinline__ float exp_chunk(const uint32_t (&x)[32], float2 c2, float2 nm2, uint32_t (&pk)[16]) {
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float2 y0 = __ffma2_rn(make_float2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1])), c2, nm2);
        const float2 y1 =
            __ffma2_rn(make_float2(__uint_as_float(x[2 * i + 2]), __uint_as_float(x[2 * i + 3])), c2, nm2);
        pk[i] = tc::pack_bf16x2(tc::ex2(y0.x), tc::ex2(y0.y));
        pk[i + 1] = tc::pack_bf16x2(tc::ex2(y1.x), tc::ex2(y1.y));
        acc0 = __fadd2_rn(acc0, make_float2(__uint_as_float(pk[i] << 16), __uint_as_float(pk[i] & 0xffff0000u)));
        acc1 = __fadd2_rn(acc1,
                          make_float2(__uint_as_float(pk[i + 1] << 16), __uint_as_float(pk[i + 1] & 0xffff0000u)));
    }
    return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}
// Chunk sum of the scoring row.  A whole 64-token chunk (a[] and b[]) is a
// tree of packed adds (32 instructions); the chunk at the end of the prefix
// sums x[0..lim) (lim clamped to [0, 32]) with eight partial sums.
__device__ __forceinline__ float sum64(const uint32_t (&a)[32], const uint32_t (&b)[32]) {
    float2 p[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        p[i] = __fadd2_rn(make_float2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1])),
                          make_float2(__uint_as_float(b[2 * i]), __uint_as_float(b[2 * i + 1])));
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) p[i] = __fadd2_rn(p[i], p[i + w]);
    return p[0].x + p[0].y;
}
__device__ __forceinline__ float sum_chunk(const uint32_t (&x)[32], int lim) {
    float p[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 32; ++i) p[i & 7] += (i < lim) ? __uint_as_float(x[i]) : 0.f;
    return ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
}

// TMEM columns: S(m, b) at 64 (2m + b); O(m) at 256 + 128 m.
__device__ __forceinline__ uint32_t s_col(int m, int b) { return (uint32_t)(64 * (2 * m + b)); }
__device__ __forceinline__ uint32_t o_col(int m) { return (uint32_t)(256 + 128 * m); }

}  // namespace

__global__ void __launch_bounds__(TC_THREADS, 1)
tree_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnArgs a, const TcLaunch L) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    TcSmemTail *tl = reinterpret_cast<TcSmemTail *>(base + SMEM_DATA_BYTES);
    volatile int *abort_flag = &tl->abort_flag;

    // ---- which (KV head, stream, KV range) this CTA owns
    const int g = blockIdx.x / L.ctas_per_head;
    int rr = blockIdx.x % L.ctas_per_head;
    bool pair;
    int mt0, split, tiles_per;
    if (rr < L.n_pair * L.s_pair) {
        pair = true;
        mt0 = 2 * (rr / L.s_pair);
        split = rr % L.s_pair;
        tiles_per = L.tl_pair;
    } else {
        rr -= L.n_pair * L.s_pair;
        pair = false;
        mt0 = 2 * L.n_pair + rr / L.s_single;
        split = rr % L.s_single;
        tiles_per = L.tl_single;
    }
    const int nm = pair ? 2 : 1;
    const int tile_begin = split * tiles_per;
    const int n_my = max(0, min(L.n_tiles, tile_begin + tiles_per) - tile_begin);
    unsigned char *sQ = base;                            // [2][Q_TILE_BYTES]
    unsigned char *sK = sQ + (size_t)2 * Q_TILE_BYTES;   // [NSTAGE][KV_TILE_BYTES]
    unsigned char *sV = sK + (size_t)NSTAGE * KV_TILE_BYTES;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.G, tpb = L.tpb;
    const int rows_loaded = tpb * G;
    // M-tile slot (0/1) holding the row whose chunk scores this pass produces, or -1
    const int score_wm = (a.chunk_scores != nullptr && a.score_row / tpb >= mt0 && a.score_row / tpb < mt0 + nm)
                             ? a.score_row / tpb - mt0 : -1;

    if (threadIdx.x == 0) {
        tc::mbar_init(&tl->q_full, 1);
        for (int s = 0; s < NSTAGE; ++s) {
            tc::mbar_init(&tl->k_full[s], 1);
            tc::mbar_init(&tl->k_empty[s], 1);
            tc::mbar_init(&tl->v_full[s], 1);
            tc::mbar_init(&tl->v_empty[s], 1);
        }
        for (int m = 0; m < 2; ++m) {
            for (int b = 0; b < 2; ++b) {
                tc::mbar_init(&tl->s_full[m][b], 1);
                tc::mbar_init(&tl->p_full[m][b], 128);
            }
            tc::mbar_init(&tl->o_done[m], 1);
            tc::mbar_init(&tl->o_final[m], 1);
        }
        tc::mbar_init(&tl->mma_done, 1);
        for (int sl = 0; sl < SCORE_RING; ++sl) {
            tc::mbar_init(&tl->score_full[sl], (uint32_t)G);
            tc::mbar_init(&tl->score_empty[sl], 1);
        }
        tl->abort_flag = 0;
        tc::fence_mbar_init();
    }
    // Q rows the TMA box does not cover (rows_loaded..127 of each M-tile) are
    // zeroed so that every S row is finite.
    if (rows_loaded < 128) {
        const int per_half = (128 - rows_loaded) * 8;  // 16-byte units
        for (int e = threadIdx.x; e < nm * 2 * per_half; e += TC_THREADS) {
            const int mh = e / per_half, u = e % per_half;
            uint4 *dst = reinterpret_cast<uint4 *>(sQ + (size_t)mh * Q_HALF_BYTES + (size_t)rows_loaded * 128) + u;
            *dst = make_uint4(0u, 0u, 0u, 0u);
        }
        tc::fence_proxy_async();
    }
    if (warp == 1) {
        tc::tmem_alloc(&tl->tmem_base, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = tl->tmem_base;

    if (warp < 4) {
      if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && n_my > 0) {
            tc::prefetch_tmap(&tm_q);
            tc::prefetch_tmap(&tm_k);
            tc::prefetch_tmap(&tm_v);
            const uint32_t qbytes = (uint32_t)(2 * 128 * rows_loaded);  // two 64-column halves
            tc::mbar_arrive_expect_tx(&tl->q_full, qbytes * nm);
            for (int m = 0; m < nm; ++m)
                for (int h = 0; h < 2; ++h)
                    tc::tma_load_3d(sQ + m * Q_TILE_BYTES + h * Q_HALF_BYTES, &tm_q, &tl->q_full, h * 64, g * G,
                                    (mt0 + m) * tpb);
            int nk = 0, nv = 0;  // K and V tiles issued
            int st = 0;
            uint32_t ph = 0;
            for (int it = 0; it < n_my; ++it) {
                const int tok0 = (tile_begin + it) * KV_TILE;
                if (it >= NSTAGE && !tc::mbar_wait(&tl->k_empty[st], ph ^ 1u, abort_flag)) { raise_abort(tl); break; }
                tc::mbar_arrive_expect_tx(&tl->k_full[st], KV_TILE_BYTES);
                for (int h = 0; h < 2; ++h)
                    tc::tma_load_3d(sK + st * KV_TILE_BYTES + h * KV_HALF_BYTES, &tm_k, &tl->k_full[st], h * 64, tok0, g);
                nk = it + 1;
                if (it >= NSTAGE && !tc::mbar_wait(&tl->v_empty[st], ph ^ 1u, abort_flag)) { raise_abort(tl); break; }
                tc::mbar_arrive_expect_tx(&tl->v_full[st], KV_TILE_BYTES);
                for (int h = 0; h < 2; ++h)
                    tc::tma_load_3d(sV + st * KV_TILE_BYTES + h * KV_HALF_BYTES, &tm_v, &tl->v_full[st], h * 64, tok0, g);
                nv = it + 1;
                if (++st == NSTAGE) { st = 0; ph ^= 1u; }
            }
            // never leave with a copy in flight into this CTA's shared memory
            tc::mbar_wait(&tl->q_full, 0, nullptr);
            for (int j = max(0, nk - NSTAGE); j < nk; ++j)
                tc::mbar_wait(&tl->k_full[j % NSTAGE], (uint32_t)(j / NSTAGE) & 1u, nullptr);
            for (int j = max(0, nv - NSTAGE); j < nv; ++j)
                tc::mbar_wait(&tl->v_full[j % NSTAGE], (uint32_t)(j / NSTAGE) & 1u, nullptr);
        }
      } else if (warp == 2) {
        // ------------------------------------------------------------ chunk-score reducer
        // Off the softmax's critical path: per KV tile (one chunk), the max over
        // the group's heads of the scoring rows' chunk sums.
        if (lane == 0 && score_wm >= 0) {
            for (int it = 0; it < n_my; ++it) {
                const int sl = it & (SCORE_RING - 1);
                if (!tc::mbar_wait(&tl->score_full[sl], (uint32_t)(it / SCORE_RING) & 1u, abort_flag)) {
                    raise_abort(tl);
                    break;
                }
                float b0 = -INFINITY;
                for (int j = 0; j < G; ++j) b0 = fmaxf(b0, tl->score_sum[sl][j]);
                tc::mbar_arrive(&tl->score_empty[sl]);
                const int tile = tile_begin + it;
                if ((int64_t)tile * KV_TILE < a.N) a.chunk_scores[(size_t)g * a.n_chunks + tile] = b0;
            }
        }
      } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // S(i+1) of every M-tile is issued before P.V(i): the S buffers alternate,
        // so S(i+1) overwrites the buffer of tile i-1, whose P.V was issued (and,
        // the pipe being in order, executed) before.
        if (lane == 0 && n_my > 0) {
            const uint32_t id_s = tc::idesc_bf16_f32(128, KV_TILE, false);
            const uint32_t id_o = tc::idesc_bf16_f32(128, 128, true);
            const uint64_t dq[2] = {desc_k(tc::smem_u32(sQ)), desc_k(tc::smem_u32(sQ + Q_TILE_BYTES))};
            const uint64_t dk0 = desc_k(tc::smem_u32(sK)), dv0 = desc_mn(tc::smem_u32(sV));
            bool ok = tc::mbar_wait(&tl->q_full, 0, abort_flag);
            if (ok) ok = tc::mbar_wait(&tl->k_full[0], 0, abort_flag);
            if (ok) {
                tc::fence_after_sync();
                for (int m = 0; m < nm; ++m) {
                    issue_s(tbase + s_col(m, 0), dq[m], dk0, id_s);
                    tc::mma_commit(&tl->s_full[m][0]);
                }
                tc::mma_commit(&tl->k_empty[0]);
            }
            for (int it = 0; ok && it < n_my; ++it) {
                if (it + 1 < n_my) {
                    const int kst = (it + 1) % NSTAGE;
                    if (!(ok = tc::mbar_wait(&tl->k_full[kst], (uint32_t)((it + 1) / NSTAGE) & 1u, abort_flag))) break;
                    tc::fence_after_sync();
                    const uint64_t dk = dplus(dk0, (uint32_t)kst * KV_TILE_BYTES);
                    const int b = (it + 1) & 1;
                    for (int m = 0; m < nm; ++m) {
                        issue_s(tbase + s_col(m, b), dq[m], dk, id_s);
                        tc::mma_commit(&tl->s_full[m][b]);
                    }
                    tc::mma_commit(&tl->k_empty[kst]);
                }
                const int vst = it % NSTAGE;
                if (!(ok = tc::mbar_wait(&tl->v_full[vst], (uint32_t)(it / NSTAGE) & 1u, abort_flag))) break;
                const uint64_t dv = dplus(dv0, (uint32_t)vst * KV_TILE_BYTES);
                const int b = it & 1;
                for (int m = 0; m < nm && ok; ++m) {
                    if (!(ok = tc::mbar_wait(&tl->p_full[m][b], (uint32_t)(it >> 1) & 1u, abort_flag))) break;
                    tc::fence_after_sync();
                    issue_pv(tbase + o_col(m), tbase + s_col(m, b), dv, id_o, it > 0);
                    tc::mma_commit(&tl->o_done[m]);
                }
                if (ok) tc::mma_commit(&tl->v_empty[vst]);
            }
            if (ok)
                for (int m = 0; m < nm; ++m) tc::mma_commit(&tl->o_final[m]);
            if (!ok) raise_abort(tl);
            // drain: every issued MMA completes before TMEM is released
            tc::mma_commit(&tl->mma_done);
            tc::mbar_wait(&tl->mma_done, 0, nullptr);
        }
      }
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        const int wm = (warp - 4) >> 2;  // M-tile slot 0 or 1
        const int quad = warp & 3;       // TMEM lane quadrant this warp may access
        const int r = quad * 32 + lane;  // row inside the M-tile
        const uint32_t lane_addr = tbase + ((uint32_t)(quad * 32) << 16);
        if (wm < nm && n_my > 0) {
            const int mt = mt0 + wm;
            const int t = mt * tpb + r / G;
            const int j = r % G;
            const bool row_valid = r < rows_loaded && t < a.T;
            const uint64_t *mrow = row_valid ? a.mask + (size_t)a.mw * t : nullptr;
            const bool is_score_row = score_wm == wm && row_valid && t == a.score_row;
            const bool score_warp = __any_sync(0xffffffffu, is_score_row);
            const int64_t plen = prefix_of(a, g);
            const uint32_t o_addr = lane_addr + o_col(wm);
            const float c = a.scale_log2;
            const float2 c2 = make_float2(c, c);
            float m_run = -INFINITY, l_run = 0.f;
            bool ok = true;
            for (int it = 0; it < n_my; ++it) {
                const int b = it & 1;
                const int tile = tile_begin + it;
                const int64_t tok0 = (int64_t)tile * KV_TILE;
                ok = tc::mbar_wait(&tl->s_full[wm][b], (uint32_t)(it >> 1) & 1u, abort_flag);
                if (!(ok = __all_sync(0xffffffffu, ok))) break;
                tc::fence_after_sync();
                const uint32_t s_addr = lane_addr + s_col(wm, b);
                uint32_t x0[32], x1[32];
                tc::tmem_ld32(s_addr + 0, x0);
                tc::tmem_ld32(s_addr + 32, x1);
                tc::tmem_wait_ld();

                // ---- fused chunk importance of the scoring row: chunk `tile`
                // (raw q.k summed over its tokens < N) into the ring for warp 2
                if (score_warp) {
                    if (is_score_row) {
                        float s0;
                        if (tok0 + KV_TILE <= a.N) {
                            s0 = sum64(x0, x1);
                        } else {
                            const int64_t lim64 = a.N - tok0;
                            const int lim = lim64 < 0 ? 0 : (int)lim64;
                            s0 = sum_chunk(x0, lim) + sum_chunk(x1, lim - 32);
                        }
                        const int sl = it & (SCORE_RING - 1);
                        if (it < SCORE_RING ||
                            tc::mbar_wait(&tl->score_empty[sl], (uint32_t)(it / SCORE_RING - 1) & 1u, abort_flag)) {
                            tl->score_sum[sl][j] = s0;
                            tc::mbar_arrive(&tl->score_full[sl]);
                        } else {
                            raise_abort(tl);
                        }
                    }
                    __syncwarp();
                }

                // ---- tiles that reach past the head's prefix: hide what this row may not see
                if (tok0 + KV_TILE > plen) {
                    mask_chunk(x0, tok0 + 0, plen, a.N, a.T, mrow);
                    mask_chunk(x1, tok0 + 32, plen, a.N, a.T, mrow);
                }

                // ---- row max (raw units), lazy running-max update
                const float mx = fmaxf(max_chunk(x0), max_chunk(x1));
                const float m_new = fmaxf(m_run, mx * c);
                const bool resc = m_new > m_run + RESCALE_THRESHOLD;
                const float alpha = resc ? tc::ex2(m_run - m_new) : 1.f;
                if (resc) {
                    l_run *= alpha;
                    m_run = m_new;
                }

                // ---- rescale O by alpha before this tile's P.V: the previous
                // tile's P.V into O must have completed
                if (it > 0 && __any_sync(0xffffffffu, resc)) {
                    ok = tc::mbar_wait(&tl->o_done[wm], (uint32_t)(it - 1) & 1u, abort_flag);
                    if (!(ok = __all_sync(0xffffffffu, ok))) break;
                    tc::fence_after_sync();
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t ov[32];
                        tc::tmem_ld32(o_addr + cc * 32, ov);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tc::tmem_st32(o_addr + cc * 32, ov);
                    }
                }

                // ---- P = 2^(s*c - m) in bf16 over the first 32 columns of this S
                // buffer (token k -> column k/2, even k in the lower half)
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
                const float2 nm2 = make_float2(neg_m, neg_m);
                float lsum;
                {
                    uint32_t pk[16];
                    lsum = exp_chunk(x0, c2, nm2, pk);
                    tc::tmem_st16(s_addr + 0, pk);
                }
                {
                    uint32_t pk[16];
                    lsum += exp_chunk(x1, c2, nm2, pk);
                    tc::tmem_st16(s_addr + 16, pk);
                }
                l_run += lsum;
                tc::tmem_wait_st();
                tc::fence_before_sync();
                tc::mbar_arrive(&tl->p_full[wm][b]);
            }

            // ---- epilogue: O of this range.  S(i+1) is issued before P.V(i), so the
            // last softmax does not imply that the P.V before the last one has
            // completed: wait on the commit that follows every P.V of this M-tile.
            if (ok) ok = tc::mbar_wait(&tl->o_final[wm], 0u, abort_flag);
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
                    tc::tmem_ld32(o_addr + cc * 32, ov);
                    tc::tmem_wait_ld();
                    if (row_valid) {
                        if (L.direct) {
                            uint32_t pk[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                pk[i] = tc::pack_bf16x2(__uint_as_float(ov[2 * i]) * inv,
                                                        __uint_as_float(ov[2 * i + 1]) * inv);
                            uint4 *dst = reinterpret_cast<uint4 *>(a.out + row * 128 + cc * 32);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                        } else {
                            float4 *dst =
                                reinterpret_cast<float4 *>(a.ws_o + ((size_t)split * a.T * a.Hq + row) * 128 + cc * 32);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                dst[i] = make_float4(__uint_as_float(ov[4 * i]), __uint_as_float(ov[4 * i + 1]),
                                                     __uint_as_float(ov[4 * i + 2]), __uint_as_float(ov[4 * i + 3]));
                        }
                    }
                    __syncwarp();
                }
                if (row_valid) {
                    if (L.direct) {
                        if (a.lse != nullptr) a.lse[row] = (m_run + log2f(l_run)) * TS_LN2;
                    } else {
                        reinterpret_cast<float2 *>(a.ws_ml)[(size_t)split * a.T * a.Hq + row] =
                            make_float2(m_run, l_run);
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

static int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

TcPlan tc_plan(int T, int Hq, int Hkv, int d, int64_t N, int num_sms) {
    TcPlan p{};
    const int G = Hq / Hkv;
    p.ok = d == 128 && T >= 64 && T <= TS_MAX_T && G >= 1 && G <= 32;
    if (!p.ok) return p;
    p.tpb = 128 / G;
    p.n_mtiles = ceil_div(T, p.tpb);
    p.n_pair = p.n_mtiles / 2;
    p.n_single = p.n_mtiles % 2;
    p.n_tiles = ceil_div(N + T, KV_TILE);
    const int budget = num_sms / Hkv > 1 ? num_sms / Hkv : 1;  // CTAs per KV head that fit in one wave
    int sp = 0, ss = 0;
    if (p.n_pair == 0) {
        ss = budget / p.n_single;
    } else if (p.n_single == 0) {
        sp = budget / p.n_pair;
    } else {
        // A pair stream does twice the MMA work per KV tile of a single stream:
        // choose the split counts that minimise the largest CTA's work.
        int best_cost = 0;
        for (int cand = 1; cand <= p.n_tiles; ++cand) {
            const int rest = budget - p.n_pair * cand;
            if (rest < p.n_single) break;
            const int cs = rest / p.n_single < p.n_tiles ? rest / p.n_single : p.n_tiles;
            const int cost = 2 * ceil_div(p.n_tiles, cand) > ceil_div(p.n_tiles, cs) ? 2 * ceil_div(p.n_tiles, cand)
                                                                                     : ceil_div(p.n_tiles, cs);
            if (best_cost == 0 || cost < best_cost) {
                best_cost = cost;
                sp = cand;
                ss = cs;
            }
        }
    }
    if (p.n_pair > 0) {
        sp = sp < 1 ? 1 : (sp > p.n_tiles ? p.n_tiles : sp);
        p.tl_pair = ceil_div(p.n_tiles, sp);
        p.s_pair = ceil_div(p.n_tiles, p.tl_pair);
    }
    if (p.n_single > 0) {
        ss = ss < 1 ? 1 : (ss > p.n_tiles ? p.n_tiles : ss);
        p.tl_single = ceil_div(p.n_tiles, ss);
        p.s_single = ceil_div(p.n_tiles, p.tl_single);
    }
    p.ctas_per_head = p.n_pair * p.s_pair + p.n_single * p.s_single;
    p.splits = p.s_pair > p.s_single ? p.s_pair : p.s_single;
    return p;
}

cudaError_t launch_tree_attn_tc(const AttnArgs &a, const TcPlan &p, const CUtensorMap &tq, const CUtensorMap &tk,
                                const CUtensorMap &tv, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(tree_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)TC_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    TcLaunch L{};
    L.tpb = p.tpb;
    L.n_mtiles = p.n_mtiles;
    L.n_pair = p.n_pair;
    L.s_pair = p.s_pair;
    L.s_single = p.s_single;
    L.tl_pair = p.tl_pair;
    L.tl_single = p.tl_single;
    L.n_tiles = p.n_tiles;
    L.ctas_per_head = p.ctas_per_head;
    L.direct = p.splits == 1 ? 1 : 0;
    dim3 grid(p.ctas_per_head * a.Hkv);
    tree_attn_tc_kernel<<<grid, TC_THREADS, TC_SMEM_BYTES, st>>>(tq, tk, tv, a, L);
    return cudaGetLastError();
}

// Self-test of the bounded-wait failure path: one warp waits on an mbarrier
// that no thread arrives at (no copy or MMA is in flight), gives up after
// budget_ns, records TS_ERR_TIMEOUT in the sticky status word and returns --
// the same path a stalled pipeline takes in the kernels above.
__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(uint64_t budget_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        abort_flag = 0;
        tc::fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !tc::mbar_wait_for(&bar, 0, &abort_flag, budget_ns))
        atomicExch(&g_device_error, (int)TS_ERR_TIMEOUT);
}

cudaError_t launch_bounded_wait_selftest(uint64_t budget_ns, cudaStream_t st) {
    if (injected_launch_failure()) return cudaErrorInvalidValue;
    bounded_wait_selftest_kernel<<<1, 32, 0, st>>>(budget_ns);
    return cudaGetLastError();
}

cudaError_t read_device_error(int *value, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(int));
    if (e != cudaSuccess || !clear) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace ts
