// Top-k chunk selection by radix select, shared by the selection kernel and
// the drafting kernel that selects, gathers and attends in one pass.
//
// Every chunk c < n has a 32-bit order key: the score's bits mapped so that
// unsigned order is numeric order (-0 = +0); the first n_sink and the last
// n_recent chunks take the largest key.  The chosen set is the k largest keys,
// equal keys going to the lower chunk index (TokenSwift ICML 2025 summary,
// "Approach": the partial cache keeps the chunks whose keys score highest
// against the current query).  The k-th largest key tau is found in four
// passes of 8-bit digits (a 256-bin shared-memory histogram of the keys that
// match the digits found so far, then one warp's suffix scan); every key above
// tau is chosen, and of the keys equal to tau the lowest-indexed ones that
// complete k.  Each thread owns a contiguous index range, so two block scans
// give every chosen index its position in ascending order.
#pragma once

#include <stdint.h>

namespace ts {

__device__ __forceinline__ uint32_t chunk_order_key(float x) {
    x = x + 0.0f;  // -0 -> +0 (round-to-nearest), so equal values get equal keys
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum of v over the CTA (NT threads) in thread order; *total
// gets the sum.  warp_tot: NT/32 ints of shared memory.  Two CTA barriers.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    int base = 0, sum = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const int t = warp_tot[w];
        base += (w < warp) ? t : 0;
        sum += t;
    }
    __syncthreads();  // warp_tot may be reused
    *total = sum;
    return base + x - v;
}

// Shared memory the selection needs besides the keys.
struct TopkSmem {
    uint32_t hist[256];
    int warp_tot[32];
    uint32_t digit;
    int above;
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
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int c = tid; c < n; c += NT) keys[c] = (c < n_sink || c >= n - n_recent) ? 0xffffffffu : chunk_order_key(sc[c]);
    __syncthreads();
    // after a pass, `prefix` holds tau's digits so far and `rem` how many of
    // the keys that match them are still to be taken
    uint32_t prefix = 0, pmask = 0;
    int rem = k;
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
        if (tid < 256) sm.hist[tid] = 0;
        __syncthreads();
        for (int c = tid; c < n; c += NT) {
            const uint32_t u = keys[c];
            if ((u & pmask) == prefix) atomicAdd(&sm.hist[(u >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l holds digits 255 - 8l .. 248 - 8l (descending); the digit
            // where the count from the top first reaches rem
            uint32_t h[8];
            int run = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                h[i] = sm.hist[255 - 8 * lane - i];
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
                int above = excl;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (above + (int)h[i] >= rem) {
                        sm.digit = 255u - 8u * lane - (uint32_t)i;
                        sm.above = above;
                        break;
                    }
                    above += (int)h[i];
                }
            }
        }
        __syncthreads();
        prefix |= sm.digit << shift;
        pmask |= 255u << shift;
        rem -= sm.above;
        __syncthreads();  // digit / above are rewritten by the next pass
    }
    const uint32_t tau = prefix;
    const int need = rem;  // keys equal to tau to take, the lowest-indexed ones

    // the chosen indices in ascending order: thread t owns [t * per, t * per + per)
    const int per = (n + NT - 1) / NT;
    const int c0 = tid * per, c1 = min(c0 + per, n);
    int n_eq = 0;
    for (int c = c0; c < c1; ++c) n_eq += keys[c] == tau ? 1 : 0;
    int tot;
    const int eq_before = block_exclusive_scan<NT>(n_eq, sm.warp_tot, &tot);
    int n_take = 0;
    {
        int e = eq_before;
        for (int c = c0; c < c1; ++c) {
            const uint32_t u = keys[c];
            if (u > tau) ++n_take;
            else if (u == tau) n_take += (e++ < need) ? 1 : 0;
        }
    }
    const int out0 = block_exclusive_scan<NT>(n_take, sm.warp_tot, &tot);
    bool last_taken = false;
    int e = eq_before, o = out0;
    for (int c = c0; c < c1; ++c) {
        const uint32_t u = keys[c];
        const bool take = u > tau || (u == tau && e++ < need);
        if (take) emit(o++, c);
        if (c == n - 1) last_taken = take;
    }
    return last_taken;
}

}  // namespace ts
