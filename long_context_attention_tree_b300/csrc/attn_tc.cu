// Split-KV tree-masked GQA attention on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators, TMA), for the TokenSwift verify pass: a batch
// of T >= 64 speculative rows (draft tree + n-gram chains) against the full
// bf16 KV cache (the drafts are checked by the target model over its whole KV
// cache, "How it works" on the TokenSwift tool listing).
//
// Rows of one KV head g are the T x G pairs (t, j), t-major; an M-tile is
// tpb = floor(128/G) whole batch rows times the G query heads of the group,
// so every K/V byte staged in shared memory serves all G heads.  A CTA owns
// one or two M-tiles of one KV head and a contiguous range of 128-token KV
// tiles:
//   pair stream   two M-tiles sharing every K/V load; the MMAs of one tile
//                 run while the softmax of the other works (ping-pong).
//                 TMEM: S_0 S_1 O_0 O_1 (128 columns each), P_m over S_m.
//   single stream one M-tile; S is double-buffered so the MMA of the next
//                 KV tile runs while the softmax works.  TMEM: S_a S_b O.
// The split counts are chosen on the host so that every CTA carries about
// the same tensor-core work; the partials are combined by the log-sum-exp
// merge kernel.
//
// Per KV tile and M-tile: S = Q K^T (8 MMAs, M=128 N=128 K=16, operands
// K-major in shared memory), softmax, O += P V (8 MMAs, P read from TMEM,
// V MN-major in shared memory).  Every MMA descriptor is precomputed, so the
// issuing thread only adds constants between MMAs.
//
// Warp roles (608 threads, 19 warps):
//   warp 0       TMA producer: Q once, then K and V tiles into 2-stage rings;
//   warp 1       owns TMEM (512 columns); one thread issues every tcgen05.mma;
//   warp 2       chunk-score reducer: takes the scoring rows' chunk sums from a
//                shared-memory ring and writes the max over the group's heads;
//   warps 3-10   softmax of M-tile slot 0, warps 11-18 of slot 1 (pair stream).
// Two threads own each row of S: of the eight warps of a slot, the first four
// take tokens 0-63 of every KV tile and the next four tokens 64-127 (warp w
// reaches TMEM lanes 32 (w % 4) .. +31, so warps w and w + 4 share a lane
// quadrant).  A softmax thread loads its 64 values of S into registers; the
// two threads of a row swap their maxima through one tagged 64-bit shared-
// memory word each and write P = 2^(s*c - m) as bf16 over the first 64
// columns of S (tokens 0-63 in columns 0-31).  The second half's P lands on
// columns 32-63, which hold the first half's S values for tokens 32-63: it is
// written only after the swap, which the first half enters after its loads.
// The running max is lazy: O and l are rescaled only when a row's max grows by
// more than 2^20 (P stays below 2^20, far inside bf16 and fp32 range), so the
// TMEM round trip of a rescale is rare; each thread rescales its 64 columns of
// O.  The output's normaliser sums the bf16-rounded weights that the P.V
// product uses; when the call asks for the log-sum-exp, a second sum of the
// unrounded weights gives it (and the split merge's weights).  The chunk
// importance of the scoring row is summed from the same S values (one 64-token
// chunk per thread) and handed to warp 2, so the softmax warps never wait for
// the reduction.
// Every wait is bounded (see tc_ptx.cuh): a wait that gives up raises the
// CTA's abort flag and the sticky device status word, and the CTA winds down.
#include "internal.h"
#include "tc_ptx.cuh"
#include "ts_common.cuh"

namespace ts {

__device__ int g_device_error = 0;

namespace {

constexpr int TC_THREADS = 608;  // 19 warps, at most 104 registers per thread
constexpr int KV_TILE = TC_KV_TILE;         // 128 tokens
constexpr int TILE_BYTES = 128 * 128 * 2;   // 128 rows x 128 dims, two 64-column swizzled halves
constexpr int HALF_BYTES = TILE_BYTES / 2;
constexpr int NSTAGE = 2;                   // K and V ring depth (pair: 2 Q + 2 K + 2 V = 192 KB)
static_assert(NSTAGE == 2, "the MMA issuer derives ring stages from the tile's parity");
constexpr int SMEM_DATA_BYTES = 6 * TILE_BYTES;
constexpr float RESCALE_THRESHOLD = 20.0f;  // log2 units
constexpr int SCORE_RING = 4;               // chunk-score slots between the scoring rows and warp 2

struct __align__(8) TcSmemTail {
    uint64_t q_full;
    uint64_t k_full[NSTAGE], k_empty[NSTAGE];
    uint64_t v_full[NSTAGE], v_empty[NSTAGE];
    // [slot]: the M-tile (pair stream, phase = tile) or the S buffer tile & 1
    // (single stream, phase = tile >> 1).  A single stream's warps may run a
    // tile ahead of one another, so its barriers are per buffer: a parity
    // wait must never be two phases behind.
    uint64_t s_full[2], p_half[2], p_full[2], o_done[2];  // p_half: P of tokens 0-63 written
    uint64_t mma_done;
    // Chunk scores: the G scoring rows put their two chunk sums of a KV tile
    // into a ring slot (tile & 3); warp 2 takes the max over the group's heads.
    uint64_t score_full[SCORE_RING], score_empty[SCORE_RING];
    float score_sum[SCORE_RING][2][32];          // [slot][chunk half][head j]
    // Row-max (and final normaliser) swap between the two threads of a row:
    // [tile parity][M-tile slot][token half][row] = (tile + 1) << 32 | value bits.
    uint64_t xch[2][2][2][128];
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

// Descriptors of 128-row swizzled tile halves, as 64-bit values to which a
// byte offset >> 4 is added directly (the 14-bit start field cannot overflow
// inside the 227 KB shared-memory window).
__device__ __forceinline__ uint64_t desc_k(uint32_t addr) { return tc::smem_desc_sw128(addr, 16, 1024); }
__device__ __forceinline__ uint64_t desc_mn(uint32_t addr) { return tc::smem_desc_sw128(addr, HALF_BYTES, 1024); }
__device__ __forceinline__ uint64_t dplus(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

// S[128 x 128] = Q[128 x 128] K^T: 8 MMAs with K = 16 over the head dim.
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint64_t dq, uint64_t dk, uint32_t idesc) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t off = (uint32_t)((k >> 2) * HALF_BYTES + (k & 3) * 32);
        tc::mma_ss(d_tmem, dplus(dq, off), dplus(dk, off), idesc, k > 0);
    }
}
// O[128 x 128] += P[128 x 64 tokens] V[64 tokens x 128] for one half of the
// tile (tokens 64h..64h+63): 4 MMAs with K = 16 tokens.
__device__ __forceinline__ void issue_pv_half(uint32_t o_tmem, uint32_t p_tmem, uint64_t dv, uint32_t idesc, int h,
                                              bool accumulate) {
#pragma unroll
    for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
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
// lower half).  Adds the fp32 sum of the 32 bf16-rounded values to lr, so that
// the output's normaliser sums exactly the weights the P.V product uses (a row
// dominated by one key then reproduces that key's value without the weight's
// rounding), and (EXACT) the sum of the unrounded weights to le, for the
// log-sum-exp.
template <bool EXACT>
__device__ __forceinline__ void exp_chunk(const uint32_t (&x)[32], float2 c2, float2 nm2, uint32_t (&pk)[16],
                                          float &lr, float &le) {
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f), ex = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float2 y0 = __ffma2_rn(make_float2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1])), c2, nm2);
        const float2 y1 =
            __ffma2_rn(make_float2(__uint_as_float(x[2 * i + 2]), __uint_as_float(x[2 * i + 3])), c2, nm2);
        const float2 e0 = make_float2(tc::ex2(y0.x), tc::ex2(y0.y));
        const float2 e1 = make_float2(tc::ex2(y1.x), tc::ex2(y1.y));
        pk[i] = tc::pack_bf16x2(e0.x, e0.y);
        pk[i + 1] = tc::pack_bf16x2(e1.x, e1.y);
        acc0 = __fadd2_rn(acc0, make_float2(__uint_as_float(pk[i] << 16), __uint_as_float(pk[i] & 0xffff0000u)));
        acc1 = __fadd2_rn(acc1,
                          make_float2(__uint_as_float(pk[i + 1] << 16), __uint_as_float(pk[i + 1] & 0xffff0000u)));
        if constexpr (EXACT) ex = __fadd2_rn(ex, __fadd2_rn(e0, e1));
    }
    lr += (acc0.x + acc0.y) + (acc1.x + acc1.y);
    if constexpr (EXACT) le += ex.x + ex.y;
}
// Chunk sums of the scoring row.  A whole 64-token chunk (a[] and b[]) is
// summed with packed adds into four running pairs (few live registers); the
// chunk at the end of the prefix sums x[0..lim) (lim clamped to [0, 32]) with
// eight partial sums.
__device__ __forceinline__ float sum64(const uint32_t (&a)[32], const uint32_t (&b)[32]) {
    float2 p[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        p[i & 3] = __fadd2_rn(p[i & 3], make_float2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1])));
        p[(i + 2) & 3] = __fadd2_rn(p[(i + 2) & 3], make_float2(__uint_as_float(b[2 * i]), __uint_as_float(b[2 * i + 1])));
    }
    const float2 q = __fadd2_rn(__fadd2_rn(p[0], p[1]), __fadd2_rn(p[2], p[3]));
    return q.x + q.y;
}
__device__ __forceinline__ float sum_chunk(const uint32_t (&x)[32], int lim) {
    float p[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 32; ++i) p[i & 7] += (i < lim) ? __uint_as_float(x[i]) : 0.f;
    return ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
}

// A compile-time ring stage (the issuer's tile step is instantiated per parity).
template <int V>
struct StageC {
    static constexpr int value = V;
};

// Publish this thread's value for tile `tag - 1` and wait (bounded) for the
// partner thread's word with the same tag; false if the wait gave up.
__device__ __forceinline__ bool swap_with_partner(uint64_t *mine, const uint64_t *theirs, uint32_t tag, float val,
                                                  float &other, volatile int *abort) {
    *reinterpret_cast<volatile uint64_t *>(mine) = ((uint64_t)tag << 32) | __float_as_uint(val);
    const volatile uint64_t *p = reinterpret_cast<const volatile uint64_t *>(theirs);
    uint64_t v = *p;
    if ((uint32_t)(v >> 32) != tag) {
        const uint64_t t0 = tc::globaltimer();
        for (uint32_t i = 1;; ++i) {
            v = *p;
            if ((uint32_t)(v >> 32) == tag) break;
            if ((i & 63u) == 0 && (*abort || tc::globaltimer() - t0 > tc::WAIT_BUDGET_NS)) return false;
        }
    }
    other = __uint_as_float((uint32_t)v);
    return true;
}

}  // namespace

// EXACT_LSE: the call wants the log-sum-exp, which takes the second sum.
template <bool EXACT_LSE>
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
    unsigned char *sQ = base;                          // [nm][TILE_BYTES]
    unsigned char *sK = sQ + (size_t)nm * TILE_BYTES;  // [NSTAGE][TILE_BYTES]
    unsigned char *sV = sK + (size_t)NSTAGE * TILE_BYTES;

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
            tc::mbar_init(&tl->s_full[m], 1);
            // one arrival per softmax warp, by lane 0 after the warp's lanes have
            // finished their TMEM stores (__syncwarp orders them before it)
            tc::mbar_init(&tl->p_half[m], 8);  // P of tokens 0-63 written, O rescaled by both halves
            tc::mbar_init(&tl->p_full[m], 4);  // P of tokens 64-127 written
            tc::mbar_init(&tl->o_done[m], 1);
        }
        tc::mbar_init(&tl->mma_done, 1);
        for (int sl = 0; sl < SCORE_RING; ++sl) {
            tc::mbar_init(&tl->score_full[sl], (uint32_t)(2 * G));
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
            uint4 *dst = reinterpret_cast<uint4 *>(sQ + (size_t)mh * HALF_BYTES + (size_t)rows_loaded * 128) + u;
            *dst = make_uint4(0u, 0u, 0u, 0u);
        }
        tc::fence_proxy_async();
    }
    // swap words start untagged (shared memory holds an earlier CTA's values)
    for (int e = threadIdx.x; e < (int)(sizeof(tl->xch) / sizeof(uint64_t)); e += TC_THREADS)
        (&tl->xch[0][0][0][0])[e] = 0ull;
    if (warp == 1) {
        tc::tmem_alloc(&tl->tmem_base, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = tl->tmem_base;
    // a programmatic dependent: the set-up above overlaps the previous kernel's
    // tail; every global access of this kernel comes after the wait
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp < 3) {
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
                    tc::tma_load_3d(sQ + m * TILE_BYTES + h * HALF_BYTES, &tm_q, &tl->q_full, h * 64, g * G,
                                    (mt0 + m) * tpb);
            int nk = 0, nv = 0;  // K and V tiles issued
            int st = 0;
            uint32_t ph = 0;
            for (int it = 0; it < n_my; ++it) {
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
        // Off the softmax's critical path: per KV tile, the max over the group's
        // heads of the scoring rows' two chunk sums.
        if (lane == 0 && score_wm >= 0) {
            for (int it = 0; it < n_my; ++it) {
                const int sl = it & (SCORE_RING - 1);
                if (!tc::mbar_wait(&tl->score_full[sl], (uint32_t)(it / SCORE_RING) & 1u, abort_flag)) {
                    raise_abort(tl);
                    break;
                }
                float b0 = -INFINITY, b1 = -INFINITY;
                for (int j = 0; j < G; ++j) {
                    b0 = fmaxf(b0, tl->score_sum[sl][0][j]);
                    b1 = fmaxf(b1, tl->score_sum[sl][1][j]);
                }
                tc::mbar_arrive(&tl->score_empty[sl]);
                const int tile = tile_begin + it;
                const int64_t tok0 = (int64_t)tile * KV_TILE;
                if (tok0 < a.N) a.chunk_scores[(size_t)g * a.n_chunks + 2 * tile] = b0;
                if (tok0 + 64 < a.N) a.chunk_scores[(size_t)g * a.n_chunks + 2 * tile + 1] = b1;
            }
        }
      } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_my > 0) {
            const uint32_t id_s = tc::idesc_bf16_f32(128, 128, false);
            const uint32_t id_o = tc::idesc_bf16_f32(128, 128, true);
            const uint64_t dq0 = desc_k(tc::smem_u32(sQ)), dq1 = desc_k(tc::smem_u32(sQ + TILE_BYTES));
            const uint64_t dk0 = desc_k(tc::smem_u32(sK)), dv0 = desc_mn(tc::smem_u32(sV));
            // S of tile 0 (K stage 0, phase 0)
            bool ok = tc::mbar_wait(&tl->q_full, 0, abort_flag);
            if (ok) ok = tc::mbar_wait(&tl->k_full[0], 0, abort_flag);
            if (ok) {
                tc::fence_after_sync();
                issue_s(tbase + 0, dq0, dk0, id_s);
                tc::mma_commit(&tl->s_full[0]);
                if (pair) {
                    issue_s(tbase + 128, dq1, dk0, id_s);
                    tc::mma_commit(&tl->s_full[1]);
                }
                tc::mma_commit(&tl->k_empty[0]);
            }
            // One tile: V of tile it sits in ring stage it % 2 and K of tile it+1 in
            // stage (it + 1) % 2, so the stages (and every descriptor and barrier
            // address derived from them) are compile-time constants of the
            // tile's parity P; the two parities alternate.
            auto tile_step = [&](auto Pc, int it) -> bool {
                constexpr int VS = decltype(Pc)::value;  // V stage of tile it
                constexpr int KS = VS ^ 1;               // K stage of tile it + 1
                const uint32_t vph = (uint32_t)(it >> 1) & 1u;
                const uint32_t kph = (uint32_t)((it + 1) >> 1) & 1u;
                const bool more = it + 1 < n_my;
                const uint64_t dv = dplus(dv0, (uint32_t)VS * TILE_BYTES);
                const uint64_t dk = dplus(dk0, (uint32_t)KS * TILE_BYTES);
                if (pair) {
                    // PV_0(it), S_0(it+1), PV_1(it), S_1(it+1): while one M-tile's
                    // softmax works, the tensor pipe runs the other tile's MMAs.
                    const uint32_t par = (uint32_t)it & 1u;
                    if (!tc::mbar_wait(&tl->v_full[VS], vph, abort_flag)) return false;
                    // each half of P goes to the tensor pipe as soon as it is written
                    if (!tc::mbar_wait(&tl->p_half[0], par, abort_flag)) return false;
                    tc::fence_after_sync();
                    issue_pv_half(tbase + 256, tbase + 0, dv, id_o, 0, it > 0);
                    if (!tc::mbar_wait(&tl->p_full[0], par, abort_flag)) return false;
                    tc::fence_after_sync();
                    issue_pv_half(tbase + 256, tbase + 0, dv, id_o, 1, true);
                    tc::mma_commit(&tl->o_done[0]);
                    if (more) {
                        if (!tc::mbar_wait(&tl->k_full[KS], kph, abort_flag)) return false;
                        tc::fence_after_sync();
                        issue_s(tbase + 0, dq0, dk, id_s);
                        tc::mma_commit(&tl->s_full[0]);
                    }
                    if (!tc::mbar_wait(&tl->p_half[1], par, abort_flag)) return false;
                    tc::fence_after_sync();
                    issue_pv_half(tbase + 384, tbase + 128, dv, id_o, 0, it > 0);
                    if (!tc::mbar_wait(&tl->p_full[1], par, abort_flag)) return false;
                    tc::fence_after_sync();
                    issue_pv_half(tbase + 384, tbase + 128, dv, id_o, 1, true);
                    tc::mma_commit(&tl->o_done[1]);
                    tc::mma_commit(&tl->v_empty[VS]);
                    if (more) {
                        issue_s(tbase + 128, dq1, dk, id_s);
                        tc::mma_commit(&tl->s_full[1]);
                        tc::mma_commit(&tl->k_empty[KS]);
                    }
                } else {
                    // S(it+1) into the other S buffer (buffer KS), then PV(it) from
                    // buffer VS.
                    if (more) {
                        if (!tc::mbar_wait(&tl->k_full[KS], kph, abort_flag)) return false;
                        tc::fence_after_sync();
                        issue_s(tbase + 128 * KS, dq0, dk, id_s);
                        tc::mma_commit(&tl->s_full[KS]);
                        tc::mma_commit(&tl->k_empty[KS]);
                    }
                    if (!tc::mbar_wait(&tl->v_full[VS], vph, abort_flag)) return false;
                    // P of tokens 0-63 (and both halves' O rescale), then P of tokens 64-127:
                    // the two halves are written by different threads
                    if (!tc::mbar_wait(&tl->p_half[VS], vph, abort_flag)) return false;
                    tc::fence_after_sync();
                    issue_pv_half(tbase + 256, tbase + 128 * VS, dv, id_o, 0, it > 0);
                    if (!tc::mbar_wait(&tl->p_full[VS], vph, abort_flag)) return false;
                    tc::fence_after_sync();
                    issue_pv_half(tbase + 256, tbase + 128 * VS, dv, id_o, 1, true);
                    tc::mma_commit(&tl->o_done[VS]);
                    tc::mma_commit(&tl->v_empty[VS]);
                }
                return true;
            };
            for (int it = 0; ok && it < n_my; ++it)
                ok = (it & 1) ? tile_step(StageC<1>{}, it) : tile_step(StageC<0>{}, it);
            if (!ok) raise_abort(tl);
            // drain: every issued MMA completes before TMEM is released
            tc::mma_commit(&tl->mma_done);
            tc::mbar_wait(&tl->mma_done, 0, nullptr);
        }
      }
    } else {
        // ------------------------------------------------------------ softmax warps
        const int sw = warp - 3;
        const int wm = sw >> 3;          // M-tile slot 0 or 1
        const int hh = (sw >> 2) & 1;    // token half of every KV tile: 64 hh .. 64 hh + 63
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
            // this thread's 64 columns of O
            const uint32_t o_addr = lane_addr + (pair ? 256u + 128u * (uint32_t)wm : 256u) + 64u * (uint32_t)hh;
            const float c = a.scale_log2;
            const float2 c2 = make_float2(c, c);
            // l_run: sum of the bf16-rounded weights (the output's normaliser);
            // e_run: sum of the unrounded weights (the log-sum-exp)
            float m_run = -INFINITY, l_run = 0.f, e_run = 0.f;
            bool ok = true;
            for (int it = 0; it < n_my; ++it) {
                const int slot = pair ? wm : (it & 1);
                const uint32_t spar = pair ? ((uint32_t)it & 1u) : ((uint32_t)(it >> 1) & 1u);
                const int64_t tok0 = (int64_t)(tile_begin + it) * KV_TILE + 64 * hh;  // this thread's first token
                ok = tc::mbar_wait(&tl->s_full[slot], spar, abort_flag);
                if (!(ok = __all_sync(0xffffffffu, ok))) break;
                tc::fence_after_sync();
                const uint32_t s_addr = lane_addr + 128u * (uint32_t)slot + 64u * (uint32_t)hh;
                uint32_t x0[32], x1[32];
                tc::tmem_ld32(s_addr + 0, x0);
                tc::tmem_ld32(s_addr + 32, x1);
                tc::tmem_wait_ld();
                // the scoring row's chunk sum (chunk 2 tile + hh, its tokens < N) from
                // raw S; the masking below only hides tokens the sum leaves out anyway
                float cs = 0.f;
                if (is_score_row) {
                    const int64_t lim = a.N - tok0;
                    cs = lim >= 64 ? sum64(x0, x1)
                                   : (lim <= 0 ? 0.f : sum_chunk(x0, (int)lim) + sum_chunk(x1, (int)lim - 32));
                }
                if (tok0 + 64 > plen) {
                    mask_chunk(x0, tok0 + 0, plen, a.N, a.T, mrow);
                    mask_chunk(x1, tok0 + 32, plen, a.N, a.T, mrow);
                }
                float mx = fmaxf(max_chunk(x0), max_chunk(x1));
                // ---- the row max over both halves, lazy running-max update
                {
                    float other;
                    ok = swap_with_partner(&tl->xch[it & 1][wm][hh][r], &tl->xch[it & 1][wm][hh ^ 1][r],
                                           (uint32_t)it + 1u, mx, other, abort_flag);
                    if (!(ok = __all_sync(0xffffffffu, ok))) break;
                    mx = fmaxf(mx, other);
                }
                const float m_new = fmaxf(m_run, mx * c);
                const bool resc = m_new > m_run + RESCALE_THRESHOLD;
                const float alpha = resc ? tc::ex2(m_run - m_new) : 1.f;
                if (resc) {
                    l_run *= alpha;
                    e_run *= alpha;
                    m_run = m_new;
                }
                const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
                const float2 nm2 = make_float2(neg_m, neg_m);

                // A warp whose rows need no rescale lets the tile's first P.V start now
                // (for tokens 64-127: the P of tokens 0-63 is the other half's).
                const bool warp_resc = it > 0 && __any_sync(0xffffffffu, resc);
                if (hh == 1 && !warp_resc) {
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&tl->p_half[slot]);
                }

                // ---- P = 2^(s*c - m) in bf16: token 64 hh + k -> column 32 hh + k/2
                const uint32_t p_addr = lane_addr + 128u * (uint32_t)slot + 32u * (uint32_t)hh;
                {
                    uint32_t pk[16];
                    exp_chunk<EXACT_LSE>(x0, c2, nm2, pk, l_run, e_run);
                    tc::tmem_st16(p_addr + 0, pk);
                }
                {
                    uint32_t pk[16];
                    exp_chunk<EXACT_LSE>(x1, c2, nm2, pk, l_run, e_run);
                    tc::tmem_st16(p_addr + 16, pk);
                }

                // ---- rescale this thread's 64 columns of O by alpha before this tile's
                // first P.V (which waits for both halves' arrivals on p_half)
                if (warp_resc) {
                    if (!pair) {
                        // a single stream computes S ahead: wait for the previous P.V into O
                        ok = tc::mbar_wait(&tl->o_done[(it - 1) & 1], (uint32_t)((it - 1) >> 1) & 1u, abort_flag);
                        if (!(ok = __all_sync(0xffffffffu, ok))) break;
                    }
                    // (a pair stream's S_m(it) was issued after P_m(it-1).V, so O_m is final here)
                    tc::fence_after_sync();
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint32_t ov[32];
                        tc::tmem_ld32(o_addr + cc * 32, ov);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tc::tmem_st32(o_addr + cc * 32, ov);
                    }
                }
                // every lane's P (and O) stores have completed; one lane hands the
                // warp's rows over
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if (hh == 0 || warp_resc) tc::mbar_arrive(&tl->p_half[slot]);
                    if (hh == 1) tc::mbar_arrive(&tl->p_full[slot]);
                }

                // ---- fused chunk importance of the scoring row into the ring for
                // warp 2, after P is handed over
                if (score_warp) {
                    if (is_score_row) {
                        const int sl = it & (SCORE_RING - 1);
                        if (it < SCORE_RING ||
                            tc::mbar_wait(&tl->score_empty[sl], (uint32_t)(it / SCORE_RING - 1) & 1u, abort_flag)) {
                            tl->score_sum[sl][hh][j] = cs;
                            tc::mbar_arrive(&tl->score_full[sl]);
                        } else {
                            raise_abort(tl);
                        }
                    }
                    __syncwarp();
                }
            }

            // ---- epilogue: O of this range
            // (the split merge, a programmatic dependent, may start launching now)
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            // (completion of the last P.V implies every earlier one: MMAs complete in order)
            if (ok) {
                if (pair)
                    ok = tc::mbar_wait(&tl->o_done[wm], (uint32_t)(n_my - 1) & 1u, abort_flag);
                else
                    ok = tc::mbar_wait(&tl->o_done[(n_my - 1) & 1], (uint32_t)((n_my - 1) >> 1) & 1u, abort_flag);
            }
            ok = __all_sync(0xffffffffu, ok);
            float l_tot = 0.f, e_tot = 0.f;
            if (ok) {
                // the row's two sums over both halves (swapped as tiles n_my, n_my + 1)
                float other;
                ok = swap_with_partner(&tl->xch[n_my & 1][wm][hh][r], &tl->xch[n_my & 1][wm][hh ^ 1][r],
                                       (uint32_t)n_my + 1u, l_run, other, abort_flag);
                l_tot = l_run + other;
                e_tot = l_tot;
                if (EXACT_LSE && ok)
                    ok = swap_with_partner(&tl->xch[(n_my + 1) & 1][wm][hh][r],
                                           &tl->xch[(n_my + 1) & 1][wm][hh ^ 1][r], (uint32_t)n_my + 2u, e_run,
                                           other, abort_flag);
                if (EXACT_LSE) e_tot = e_run + other;
                ok = __all_sync(0xffffffffu, ok);
            }
            if (!ok) {
                raise_abort(tl);
            } else {
                tc::fence_after_sync();
                const int h = g * G + j;
                const size_t row = (size_t)t * a.Hq + h;
                const float inv = (l_tot > 0.f) ? 1.f / l_tot : 0.f;
                // a split partial is scaled so that its ratio to the unrounded sum
                // (the merge's normaliser) is this range's O / l_tot
                const float to_e = (l_tot > 0.f) ? e_tot / l_tot : 0.f;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t ov[32];
                    tc::tmem_ld32(o_addr + cc * 32, ov);
                    tc::tmem_wait_ld();
                    const int d0 = 64 * hh + 32 * cc;  // first head dim of this piece
                    if (row_valid) {
                        if (L.direct) {
                            uint32_t pk[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                pk[i] = tc::pack_bf16x2(__uint_as_float(ov[2 * i]) * inv,
                                                        __uint_as_float(ov[2 * i + 1]) * inv);
                            uint4 *dst = reinterpret_cast<uint4 *>(a.out + row * 128 + d0);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                        } else {
                            float4 *dst =
                                reinterpret_cast<float4 *>(a.ws_o + ((size_t)split * a.T * a.Hq + row) * 128 + d0);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                dst[i] = make_float4(__uint_as_float(ov[4 * i]) * to_e, __uint_as_float(ov[4 * i + 1]) * to_e,
                                                     __uint_as_float(ov[4 * i + 2]) * to_e,
                                                     __uint_as_float(ov[4 * i + 3]) * to_e);
                        }
                    }
                    __syncwarp();
                }
                if (row_valid && hh == 0) {
                    if (L.direct) {
                        if (a.lse != nullptr) a.lse[row] = (m_run + log2f(e_tot)) * TS_LN2;
                    } else {
                        reinterpret_cast<float2 *>(a.ws_ml)[(size_t)split * a.T * a.Hq + row] =
                            make_float2(m_run, e_tot);
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
    const bool exact = a.lse != nullptr;
    cudaError_t e = exact ? cudaFuncSetAttribute(tree_attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)TC_SMEM_BYTES)
                          : cudaFuncSetAttribute(tree_attn_tc_kernel<false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM_BYTES);
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
    // launched as a programmatic dependent of whatever precedes it on the
    // stream (the kernel waits for that grid before touching global memory)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ctas_per_head * a.Hkv);
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = TC_SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return exact ? cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel<true>, tq, tk, tv, a, L)
                 : cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel<false>, tq, tk, tv, a, L);
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
