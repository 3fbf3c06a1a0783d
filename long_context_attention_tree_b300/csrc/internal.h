// Internal launch interface between the C ABI (ts_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ts.h"

namespace ts {

constexpr int TS_MAX_T = 1024;  // largest speculative batch (rows) any call takes

// Counts every kernel launch the library enqueues (diagnostic).
void note_launches(int n);

// Records `msg` as this host thread's last error message and returns `st`.
ts_status report_error(ts_status st, const char *msg);

// Host-side fault injection for tests (ts_selftest_fail_launches): true when
// the launch about to be made should report cudaErrorInvalidValue instead of
// launching.  Every launch_* function asks before it launches.
bool injected_launch_failure();

struct AttnArgs {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k;
    const __nv_bfloat16 *v;
    int64_t ld_kv;
    int64_t N;
    int T, Hq, Hkv, G, d;
    float scale_log2;  // softmax scale * log2(e)
    const uint64_t *mask;       // uint64 [T][mw]
    int mw;                     // mask words per row: max(2, ceil(T / 64))
    const int32_t *prefix_len;  // nullable: KV head g sees prefix rows [0, min(prefix_len[g], N))
    __nv_bfloat16 *out;
    float *lse;
    float *chunk_scores;  // nullable
    int score_row;
    int n_chunks;         // ceil(N / 64)
    float *ws_o;          // [splits][T][Hq][d] unnormalised partial outputs
    float *ws_ml;         // [splits][T][Hq] (m, l) pairs, log2 domain
    // plan
    int splits, tiles_per_split, n_tiles, tpb;
};

struct MergeArgs {
    const float *ws_o;
    const float *ws_ml;
    __nv_bfloat16 *out;
    float *lse;
    int T, Hq;
    int splits;      // partials of rows t < t_split
    int t_split;     // first batch row whose partial count is splits_hi
    int splits_hi;   // partials of rows t >= t_split
};

struct SimtPlan {
    int rb, tpb, n_rb, n_tiles, splits, tiles_per_split;
};

SimtPlan simt_plan(int T, int Hq, int Hkv, int d, int64_t N, int num_sms);
cudaError_t launch_tree_attn_simt(const AttnArgs &a, const SimtPlan &p, cudaStream_t st);
cudaError_t launch_lse_merge(const MergeArgs &m, int d, cudaStream_t st);

// CUDA-core path for small batches (T * G <= 24, head dim 128): one 128-token
// KV range per CTA, splits = ceil((N + T) / 128)
bool small_ok(int T, int Hq, int Hkv, int d);
int small_splits(int T, int64_t N);
// The gather variant: the prefix rows [0, N) of the attention (N = 64 k_sel)
// come from the chosen 64-token chunks of a full cache and are written into
// k_dst / v_dst (the compact cache the attention's k / v point at) as they
// are read; rows of a short last chunk at or past the full cache's N are
// neither read, seen nor written.
struct SmallGather {
    const int32_t *sel = nullptr;  // [Hkv][k_sel], ascending chunk indices
    int k_sel = 0;
    int n_chunks = 0;              // chunks of the full cache, ceil(N / 64)
    const __nv_bfloat16 *k = nullptr, *v = nullptr;  // full cache [Hkv][ld][d]
    int64_t ld = 0, N = 0;
    __nv_bfloat16 *k_dst = nullptr, *v_dst = nullptr;
    // selection in the same pass (scores != nullptr): every CTA selects the
    // k_sel chunks of its KV head from scores [Hkv][n_chunks] itself; the
    // CTAs of the first range write sel_out [Hkv][k_sel] and part_len_out
    const float *scores = nullptr;
    int n_sink = 0, n_recent = 0;
    int32_t *sel_out = nullptr, *part_len_out = nullptr;
};
cudaError_t launch_tree_attn_small(const AttnArgs &a, const SmallGather *gs, int splits, cudaStream_t st);

// tensor-core (tcgen05) path, head_dim 128, 64 <= T <= 128.
constexpr int TC_KV_TILE = 128;  // KV tokens per pipeline step (two 64-token scoring chunks)
// Per KV head the M-tiles are grouped into n_pair two-tile streams (ping-pong
// between the two tiles) and n_single one-tile streams (double-buffered S);
// each stream's KV tiles are split into s_pair / s_single contiguous ranges.
struct TcPlan {
    bool ok;
    int tpb;                  // whole batch rows per M-tile (floor(128 / G))
    int n_mtiles;             // ceil(T / tpb)
    int n_pair, n_single;     // streams per KV head
    int s_pair, s_single;     // KV splits per stream kind
    int tl_pair, tl_single;   // KV tiles per split
    int n_tiles;              // ceil((N + T) / TC_KV_TILE)
    int ctas_per_head;        // n_pair * s_pair + n_single * s_single
    int splits;               // max(s_pair, s_single): workspace slices
};
TcPlan tc_plan(int T, int Hq, int Hkv, int d, int64_t N, int num_sms);
size_t tc_smem_bytes();
cudaError_t launch_tree_attn_tc(const AttnArgs &a, const TcPlan &p, const CUtensorMap &tq, const CUtensorMap &tk,
                                const CUtensorMap &tv, cudaStream_t st);
// sticky device-side error word (TS_ERR_TIMEOUT when a bounded wait gave up)
cudaError_t read_device_error(int *value, bool clear);
// one warp whose bounded wait on an mbarrier nobody arrives at gives up
cudaError_t launch_bounded_wait_selftest(uint64_t budget_ns, cudaStream_t st);

// Visible prefix length of KV head g (ragged partial caches clamp to [0, N]).
__device__ __forceinline__ int64_t prefix_of(const AttnArgs &a, int g) {
    if (a.prefix_len == nullptr) return a.N;
    const int64_t p = a.prefix_len[g];
    return p < 0 ? 0 : (p > a.N ? a.N : p);
}

// chunk scoring / selection / gather
// scores[g * ld_scores + c] for the chunks c in [c_begin, ceil(N / 64))
cudaError_t launch_score_chunks(const __nv_bfloat16 *q_row, const __nv_bfloat16 *k, int64_t ld_kv, int64_t N,
                                int Hq, int Hkv, int d, float *scores, int64_t ld_scores, int c_begin,
                                cudaStream_t st);
// scores_new[g][c] = scores_old[g][c] for c < c_keep (row strides nc_new / nc_old)
cudaError_t launch_copy_scores(const float *scores_old, int nc_old, float *scores_new, int nc_new, int c_keep,
                               int Hkv, cudaStream_t st);
// top-k chunk selection (a programmatic dependent of the kernel before it)
cudaError_t launch_select(const float *scores, int Hkv, int64_t N, int n_chunks, int k_sel, int n_sink, int n_recent,
                          int32_t *sel, int32_t *part_len, cudaStream_t st);
// gather of the selected chunks (a programmatic dependent of the selection)
cudaError_t launch_gather(const int32_t *sel, int Hkv, int64_t N, int n_chunks, int k_sel,
                          const __nv_bfloat16 *k, const __nv_bfloat16 *v, int64_t ld_kv, int d,
                          __nv_bfloat16 *k_part, __nv_bfloat16 *v_part, int64_t ld_part, cudaStream_t st);

// vocab stage
struct VocabArgs {
    const float *logits;
    int T, V;
    const int32_t *history;
    int W;
    float theta, temperature;
    double log_min_p;
    const int32_t *draft;
    const int32_t *parent;
    int32_t anchor;
    int32_t *target, *kept, *result, *path;
    int sample;                      // 1: target = min-p sample (Gumbel-max), 0: greedy
    int path_window;                 // 1: each row's window ends with the drafts on its path
    unsigned long long seed, offset; // Philox4x64-10 key word 0 and counter word 2
};
cudaError_t launch_vocab(const VocabArgs &a, cudaStream_t st);

// n-gram table: int4 keys [C], int32 counts [C], int32 first positions [C]
// (C a power of two >= 64)
cudaError_t launch_ngram_reset(void *table, uint32_t C, cudaStream_t st);
cudaError_t launch_ngram_update(void *table, uint32_t C, const int32_t *seq, int64_t n_old, int64_t n_new,
                                int32_t *status, cudaStream_t st);
cudaError_t launch_ngram_topk(const void *table, uint32_t C, const int32_t *seq, int64_t n, const int32_t *anchor,
                              int k, int32_t *chains, int32_t *counts, int32_t *found, cudaStream_t st);

// commit of the accepted path into the full cache (T <= 128)
cudaError_t launch_commit_path(__nv_bfloat16 *k, __nv_bfloat16 *v, int64_t ld_kv, int64_t N, int T, int Hkv, int d,
                               int32_t *result, const int32_t *path, cudaStream_t st);

}  // namespace ts
