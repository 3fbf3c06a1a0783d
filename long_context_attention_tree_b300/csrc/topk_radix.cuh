// Top-k chunk selection by radix select, shared by the selection kernel and
// the drafting kernel that selects, gathers and attends in one pass.
//
// Every chunk c < n has a 32-bit order key: the score's bits mapped so that
// unsigned order is numeric order (-0 = +0); the first n_sink and the last
// n_recent chunks take the largest key.  The chosen set is the k largest keys,
// equal keys going to the lower chunk index (TokenSwift ICML 2025 summary,
// "Approach": the partial cache keeps the chunks whose keys score highest
// against the current query).  The k-th largest key tau is found in at most
// four passes of 8-bit digits: a 256-bin shared-memory histogram of the keys
// that match the digits found so far, then one warp's suffix scan.  The
// passes stop early when the digit's bin holds exactly the keys still to be
// taken; every key above tau is chosen, and of the keys equal to tau the
// lowest-indexed ones that complete k.  Each thread owns a contiguous index range, so one block scan
// of (keys above tau, keys equal to tau) gives every chosen index its
// position in ascending order.
#pragma once

#include <stdint.h>

namespace ts {

__device__ __forceinline__ uint32_t chunk_order_key(float x) {
    x = x + 0.0f;  // -0 -> +0 (round-to-nearest), so equal values get equal keys
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sums of the pair (a, b) over the CTA (NT threads) in
// thread order, returned as (a_before, b_before).  warp_tot: 2 * NT / 32 ints
// of shared memory.  Two CTA barriers.
template <int NT>
__device__ __forceinline__ int2 block_exclusive_scan2(int a, int b, int *warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = a, y = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int xa = __shfl_up_sync(0xffffffffu, x, o);
        const int yb = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) {
            x += xa;
            y += yb;
        }
    }
    if (lane == 31) {
        warp_tot[2 * warp] = x;
        warp_tot[2 * warp + 1] = y;
    }
    __syncthreads();
    int ba = 0, bb = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        if (w < warp) {
            ba += warp_tot[2 * w];
            bb += warp_tot[2 * w + 1];
        }
    }
    __syncthreads();  // warp_tot may be reused
    return make_int2(ba + x - a, bb + y - b);
}

// Histogram bin b sits at word b + b / 8: a lane reads eight consecutive
// bins, and with the padding the 32 lanes' reads of one bin position fall in
// 32 different banks.
constexpr int TOPK_HIST_WORDS = 256 + 32;
__device__ __forceinline__ int topk_bin(uint32_t b) { return (int)(b + (b >> 3)); }

// Shared memory the selection needs besides the keys: three histograms (the
// one a pass counts into was zeroed during the pass before, two barriers
// after warp 0 last read it), the scan's warp totals, and the digit that
// warp 0 finds with the counts around it.
struct TopkSmem {
    uint32_t hist[3][TOPK_HIST_WORDS];
    int warp_tot[64];
    uint32_t digit;
    int above, cnt;
};

// The k chosen chunk indices of scores sc[0..n), in ascending order: every
// thread of the CTA (NT threads) must call this; emit(pos, c) is called once
// for each chosen index c with its position pos in [0, k).  keys: n words of
// shared memory.  Returns true in the thread whose range holds index n - 1 if
// that chunk was chosen (false everywhere else).  Requires 1 <= k <= n.
template <int NT, typename Emit>
__device__ bool radix_topk_ascending(const float *sc, int n, int k, int n_sink, int n_recent, uint32_t *keys,
                                     TopkSmem &sm, Emit emit) {
    static_assert(NT >= 256 && NT % 32 == 0 && NT / 32 <= 32, "one histogram bin per thread, at most 32 warps");
    const int tid = threadIdx.x, lane = tid & 31;
    // eight independent score loads in flight per thread: a loop that stores
    // each key before loading the next would pay one L2 round trip per key
    constexpr int LB = 8;
    for (int c0 = tid; c0 < n; c0 += NT * LB) {
        float v[LB];
#pragma unroll
        for (int j = 0; j < LB; ++j) {
            const int c = c0 + j * NT;
            v[j] = c < n ? sc[c] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < LB; ++j) {
            const int c = c0 + j * NT;
            if (c < n) keys[c] = (c < n_sink || c >= n - n_recent) ? 0xffffffffu : chunk_order_key(v[j]);
        }
    }
    for (int i = tid; i < TOPK_HIST_WORDS; i += NT) sm.hist[0][i] = 0;
    __syncthreads();
    // after a pass, `prefix` holds tau's digits so far and `rem` how many of
    // the keys that match them are still to be taken
    uint32_t prefix = 0, pmask = 0;
    int rem = k;
    int need = -1;  // set when the digits found so far settle the whole choice
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        uint32_t *hist = sm.hist[pass % 3];
        // keys read in batches ahead of the atomics (which could alias them)
        for (int c0 = tid; c0 < n; c0 += NT * LB) {
            uint32_t u[LB];
#pragma unroll
            for (int j = 0; j < LB; ++j) {
                const int c = c0 + j * NT;
                u[j] = c < n ? keys[c] : 0u;
            }
#pragma unroll
            for (int j = 0; j < LB; ++j)
                if ((u[j] & pmask) == prefix && c0 + j * NT < n) atomicAdd(&hist[topk_bin((u[j] >> shift) & 255u)], 1u);
        }
        // the next pass's histogram (last read by warp 0 two passes ago)
        for (int i = tid; i < TOPK_HIST_WORDS; i += NT) sm.hist[(pass + 1) % 3][i] = 0;
        __syncthreads();
        // warp 0 finds the digit where the count from the top first reaches
        // rem: lane l holds digits 255 - 8l .. 248 - 8l (descending)
        if (tid < 32) {
            uint32_t h[8];
            int run = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                h[i] = hist[topk_bin(255u - 8u * lane - (uint32_t)i)];
                run += (int)h[i];
            }
            int incl = run;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int excl = incl - run;  // count of the digits above this lane's
            if (excl < rem && incl >= rem) {
                int a = excl;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (a + (int)h[i] >= rem) {
                        sm.digit = 255u - 8u * lane - (uint32_t)i;
                        sm.above = a;
                        sm.cnt = (int)h[i];
                        break;
                    }
                    a += (int)h[i];
                }
            }
        }
        __syncthreads();
        const uint32_t digit = sm.digit;
        const int above = sm.above, cnt = sm.cnt;
        __syncthreads();  // digit, above and cnt are rewritten by the next pass
        prefix |= digit << shift;
        pmask |= 255u << shift;
        rem -= above;
        if (cnt == rem) {
            // every key that matches the digits so far is chosen: the choice
            // is every key >= prefix (its lower digits zero)
            need = n;
            break;
        }
    }
    const uint32_t tau = prefix;
    if (need < 0) need = rem;  // keys equal to tau to take, the lowest-indexed ones

    // the chosen indices in ascending order: thread t owns [t * per, t * per + per)
    const int per = (n + NT - 1) / NT;
    const int c0 = tid * per, c1 = min(c0 + per, n);
    int n_gt = 0, n_eq = 0;
    for (int c = c0; c < c1; ++c) {
        const uint32_t u = keys[c];
        n_gt += u > tau ? 1 : 0;
        n_eq += u == tau ? 1 : 0;
    }
    // chosen before this range: every key above tau, and the first `need`
    // keys equal to it
    const int2 before = block_exclusive_scan2<NT>(n_gt, n_eq, sm.warp_tot);
    bool last_taken = false;
    int e = before.y, o = before.x + min(before.y, need);
    for (int c = c0; c < c1; ++c) {
        const uint32_t u = keys[c];
        const bool take = u > tau || (u == tau && e++ < need);
        if (take) emit(o++, c);
        if (c == n - 1) last_taken = take;
    }
    return last_taken;
}

}  // namespace ts
