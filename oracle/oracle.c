/*
 * oracle.c -- plain, slow fp64 CPU oracle of the TokenSwift attention-side
 * hot path.  TEST INFRASTRUCTURE ONLY: the test-suite, the smoke check and
 * the benchmark's CPU-baseline leg call it; the product library never does.
 * It shares no code, header or table with the CUDA path.
 *
 * Sources (TokenSwift pages):
 *   - model card "TokenSwift-Qwen2.5-7B", "Example using TokenSwift command
 *     line": retrieval budget 4096, gamma 4, min_p 0.1, temperature 1.0,
 *     ngram_topk 20, penalty 1.2, penalty_length 1024;
 *   - tool listing, "How it works": drafts from a partial KV cache, a
 *     tree-based attention over candidates, verification with the full KV
 *     cache, exact match of draft and target tokens, one longest valid draft
 *     kept;
 *   - ICML 2025 summary, "Approach": the partial KV cache keeps the chunks whose
 *     importance, windowed contextual penalty; ablation table: tree
 *     [1,3,3,3], theta 1.2, W 1024.
 * Where the pages are silent the plainest reading is used; every reading is
 * listed in the design notes (scale 1/sqrt(d); head h uses KV head h/G;
 * chunk score = max over the group of q . sum(K_chunk); ties to the lower
 * index; penalty divides positive logits and multiplies the others once per
 * distinct id in the window; penalty, then temperature, then min-p; greedy
 * target; lowest row among the longest accepted paths).
 *
 * Everything is computed straight from the definitions, in fp64 unless the
 * decision itself is taken in the kernel's precision (selection on fp32
 * scores, penalty/min-p on fp32 logits).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE binary32 word. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---------------------------------------------------------------------- */
/* Visibility inside the speculative batch.  Row i sees row j (j in the     */
/* batch) iff j == i or j is an ancestor of i in the parent forest.  The    */
/* tree-based attention of "How it works"; chains are parent = previous.    */
/* vis is T*T bytes, row-major.  Returns 0, or 1 for an invalid parent.     */
/* ---------------------------------------------------------------------- */
int oracle_visible(const int32_t *parent, int T, uint8_t *vis)
{
    for (int i = 0; i < T; ++i)
        if (parent[i] < -1 || parent[i] >= i) return 1;
    memset(vis, 0, (size_t)T * (size_t)T);
    for (int i = 0; i < T; ++i)
        for (int j = i; j >= 0; j = parent[j]) vis[(size_t)i * T + j] = 1;
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Tree-masked attention for a list of output rows.                        */
/*   q: bf16 [T][Hq][d];  k, v: bf16 [Hkv][ld_kv][d]; prefix rows [0,N),   */
/*   the batch's own rows at [N, N+T).  Row id r = t*Hq + h.               */
/*   For row (t,h), KV head g = h / (Hq/Hkv).  Visible keys: every prefix  */
/*   token j < P_g, and batch token N+u when u is t itself or an ancestor  */
/*   of t.  P_g = N, or prefix_len[g] when prefix_len is given (a compact  */
/*   partial cache whose heads hold different numbers of valid rows).      */
/*   s_j = scale * (q . k_j)   (fp64 from the bf16 values)                  */
/*   o   = sum_j softmax(s)_j v_j,   lse = log sum_j exp(s_j)               */
/*   out: double [n_rows][d];  lse_out: double [n_rows] (nullable).         */
/* Returns 0, 1 on a bad parent array, 2 on bad sizes.                     */
/* ---------------------------------------------------------------------- */
int oracle_tree_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          int64_t ld_kv, int64_t N, int T, int Hq, int Hkv, int d,
                          double scale, const int32_t *parent, const int32_t *prefix_len,
                          const int32_t *row_ids, int n_rows,
                          double *out, double *lse_out)
{
    if (T < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || N < 0 || ld_kv < N + T)
        return 2;
    if (prefix_len)
        for (int g = 0; g < Hkv; ++g)
            if (prefix_len[g] < 0 || prefix_len[g] > N) return 2;
    uint8_t *vis = (uint8_t *)malloc((size_t)(T > 0 ? T : 1) * (size_t)(T > 0 ? T : 1));
    if (!vis) return 2;
    if (T > 0 && oracle_visible(parent, T, vis)) { free(vis); return 1; }
    for (int r = 0; r < n_rows; ++r)
        if (row_ids[r] < 0 || row_ids[r] >= T * Hq) { free(vis); return 2; }
    const int G = Hq / Hkv;
    const int64_t L = N + T;
    int err = 0;

#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        uint8_t *seen = (uint8_t *)malloc((size_t)(L > 0 ? L : 1));
        double *acc = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !seen || !acc) {
#pragma omp atomic write
            err = 2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n_rows; ++r) {
            if (!s || !seen || !acc) continue;
            const int t = row_ids[r] / Hq;
            const int h = row_ids[r] % Hq;
            const int g = h / G;
            const uint16_t *qr = q + ((size_t)t * Hq + h) * d;
            const uint16_t *kh = k + (size_t)g * ld_kv * d;
            const uint16_t *vh = v + (size_t)g * ld_kv * d;
            const int64_t P = prefix_len ? prefix_len[g] : N;
            double m = -INFINITY;
            for (int64_t j = 0; j < L; ++j) {
                seen[j] = (j < N) ? (j < P) : vis[(size_t)t * T + (j - N)];
                if (!seen[j]) continue;
                double dot = 0.0;
                for (int c = 0; c < d; ++c)
                    dot += bf16_value(qr[c]) * bf16_value(kh[j * d + c]);
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int c = 0; c < d; ++c) acc[c] = 0.0;
            for (int64_t j = 0; j < L; ++j) {
                if (!seen[j]) continue;
                double p = exp(s[j] - m);
                l += p;
                for (int c = 0; c < d; ++c) acc[c] += p * bf16_value(vh[j * d + c]);
            }
            for (int c = 0; c < d; ++c) out[(size_t)r * d + c] = acc[c] / l;
            if (lse_out) lse_out[r] = m + log(l);
        }
        free(s);
        free(seen);
        free(acc);
    }
    free(vis);
    return err;
}

/* ---------------------------------------------------------------------- */
/* Chunk importance (ICML 2025 summary, "Approach": the partial cache is   */
/* chosen by how strongly the query attends to each part of the keys).     */
/*   score[g][c] = max_{h in group g} q_h . sum_{t in chunk c} k_t          */
/* over prefix tokens only; the last chunk may be partial.  Unscaled.      */
/*   q_row: bf16 [Hq][d];  scores: double [Hkv][ceil(N/chunk)].             */
/* ---------------------------------------------------------------------- */
int oracle_score_chunks(const uint16_t *q_row, const uint16_t *k, int64_t ld_kv, int64_t N,
                        int Hq, int Hkv, int d, int chunk, double *scores)
{
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || d > 512 || chunk <= 0 || N < 0 || ld_kv < N)
        return 2;
    const int G = Hq / Hkv;
    const int64_t nc = (N + chunk - 1) / chunk;
#pragma omp parallel for collapse(2) schedule(static)
    for (int g = 0; g < Hkv; ++g) {
        for (int64_t c = 0; c < nc; ++c) {
            double ksum[512];
            for (int e = 0; e < d; ++e) ksum[e] = 0.0;
            int64_t t_end = (c + 1) * chunk < N ? (c + 1) * chunk : N;
            for (int64_t t = c * chunk; t < t_end; ++t)
                for (int e = 0; e < d; ++e)
                    ksum[e] += bf16_value(k[((size_t)g * ld_kv + t) * d + e]);
            double best = -INFINITY;
            for (int j = 0; j < G; ++j) {
                const uint16_t *qh = q_row + (size_t)(g * G + j) * d;
                double dot = 0.0;
                for (int e = 0; e < d; ++e) dot += bf16_value(qh[e]) * ksum[e];
                if (dot > best) best = dot;
            }
            scores[(size_t)g * nc + c] = best;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Top-k chunk selection up to the retrieval budget.                       */
/* Per KV head: the k chunks with the largest fp32 score; equal scores go  */
/* to the lower chunk index; the chosen indices are returned ascending.    */
/* Scores compare as values (so -0 equals +0).                             */
/*   scores: float [Hkv][nc];  sel: int32 [Hkv][k] with k = min(k, nc).     */
/* ---------------------------------------------------------------------- */
static const float *g_sort_keys;
static int by_score_then_index(const void *a, const void *b)
{
    int ia = *(const int *)a, ib = *(const int *)b;
    float sa = g_sort_keys[ia], sb = g_sort_keys[ib];
    if (sa > sb) return -1;
    if (sa < sb) return 1;
    return (ia > ib) - (ia < ib);
}
static int ascending(const void *a, const void *b)
{
    int ia = *(const int *)a, ib = *(const int *)b;
    return (ia > ib) - (ia < ib);
}

/* Always-kept chunks (the SnapKV / TriForce lineage the summary's related   */
/* work names: attention sinks at the start, a recent window at the end):    */
/* with n_sink, n_recent > 0 the chunks [0, n_sink) and [nc - n_recent, nc)  */
/* are selected first, and the rest of the k by score among the others.      */
/* Requires n_sink + n_recent <= k.                                          */
static int g_nc_forced, g_n_sink, g_n_recent;
static int forced(int c) { return c < g_n_sink || c >= g_nc_forced - g_n_recent; }
static int forced_then_score_then_index(const void *a, const void *b)
{
    int ia = *(const int *)a, ib = *(const int *)b;
    int fa = forced(ia), fb = forced(ib);
    if (fa != fb) return fa ? -1 : 1;
    return by_score_then_index(a, b);
}

int oracle_select_kept(const float *scores, int Hkv, int nc, int k, int n_sink, int n_recent, int32_t *sel)
{
    if (Hkv <= 0 || nc < 0 || k < 0 || n_sink < 0 || n_recent < 0 || n_sink + n_recent > k) return 2;
    if (k > nc) k = nc;
    int *idx = (int *)malloc(sizeof(int) * (size_t)(nc > 0 ? nc : 1));
    if (!idx) return 2;
    g_nc_forced = nc; g_n_sink = n_sink; g_n_recent = n_recent;
    for (int g = 0; g < Hkv; ++g) {
        for (int c = 0; c < nc; ++c) {
            if (scores[(size_t)g * nc + c] != scores[(size_t)g * nc + c]) { free(idx); return 3; }
            idx[c] = c;
        }
        g_sort_keys = scores + (size_t)g * nc;
        qsort(idx, (size_t)nc, sizeof(int), forced_then_score_then_index);
        qsort(idx, (size_t)k, sizeof(int), ascending);
        for (int i = 0; i < k; ++i) sel[(size_t)g * k + i] = idx[i];
    }
    free(idx);
    return 0;
}

int oracle_select(const float *scores, int Hkv, int nc, int k, int32_t *sel)
{
    return oracle_select_kept(scores, Hkv, nc, k, 0, 0, sel);
}

/* Gather the selected chunks into a compact cache (byte copy).            */
/*   dst[g][i*chunk + t] = src[g][sel[g][i]*chunk + t] for i<k, t<chunk,    */
/* rows of d bf16 elements; tokens at or past N are not copied (a partial  */
/* last chunk leaves its trailing rows of dst untouched).                  */
/* part_len (nullable): int32 [Hkv], the number of tokens gathered for     */
/* head g -- the rows [0, part_len[g]) of dst hold real tokens when the    */
/* selection is ascending (only the last chunk of the prefix can be short, */
/* and it is the largest index, so it sits last).                          */
int oracle_gather(const int32_t *sel, int Hkv, int k, int chunk, int64_t N,
                  const uint16_t *src, int64_t ld_src, int d, uint16_t *dst, int64_t ld_dst,
                  int32_t *part_len)
{
    if ((int64_t)k * chunk > ld_dst) return 2;
    for (int g = 0; g < Hkv; ++g) {
        int32_t copied = 0;
        for (int i = 0; i < k; ++i) {
            int64_t c = sel[(size_t)g * k + i];
            for (int t = 0; t < chunk; ++t) {
                int64_t s = c * chunk + t;
                if (s >= N) break;
                memcpy(dst + ((size_t)g * ld_dst + (size_t)i * chunk + t) * d,
                       src + ((size_t)g * ld_src + s) * d, sizeof(uint16_t) * (size_t)d);
                ++copied;
            }
        }
        if (part_len) part_len[g] = copied;
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Windowed contextual penalty, temperature, min-p and greedy target.      */
/*   S = distinct ids among the last W generated tokens (history[0..W)).   */
/*   For v in S: l > 0 ? l / theta : l * theta   (fp32 result, IEEE RN: the */
/*   fp64 quotient/product rounded once to fp32 equals the fp32 operation). */
/*   Then l / temperature (same rounding argument).                        */
/*   m = max, target = lowest id attaining m.                              */
/*   kept = #{v : (double)l_v >= fl64(m + log_min_p)}  -- min-p in logit    */
/*   space, p_v >= min_p * p_max; log_min_p is computed once by the caller. */
/*   pen_out (nullable): the final fp32 logits.                             */
/* Returns 0, or 4 for a history id outside [0, V).                        */
/* ---------------------------------------------------------------------- */
/* Path-aware window (path_parent and path_draft given): the logits of row i */
/* follow the drafts on its path root..i (depth d_i tokens), so its window is */
/* the last W tokens of history ++ (draft of the root, ..., draft[i]):        */
/* history[min(d_i, W) .. W) and the last min(d_i, W) drafts of the path     */
/* (a draft outside [0, V), such as an unused n-gram row's -1, is no token   */
/* and adds nothing).                                                        */
/* Returns 0, 4 for a history id outside [0, V), 1 for a bad parent array.   */
int oracle_penalty_minp_path(const float *logits, int T, int V, const int32_t *history, int W,
                             const int32_t *path_parent, const int32_t *path_draft,
                             float theta, float temperature, double log_min_p,
                             int32_t *target, int32_t *kept, float *pen_out)
{
    uint8_t *inwin = (uint8_t *)calloc((size_t)(V > 0 ? V : 1), 1);
    if (!inwin) return 2;
    for (int w = 0; w < W; ++w) {
        if (history[w] < 0 || history[w] >= V) { free(inwin); return 4; }
        inwin[history[w]] = 1;
    }
    if (path_parent) {
        for (int i = 0; i < T; ++i)
            if (path_parent[i] < -1 || path_parent[i] >= i) { free(inwin); return 1; }
    }
    int err = 0;
#pragma omp parallel for schedule(static)
    for (int i = 0; i < T; ++i) {
        float *row = (float *)malloc(sizeof(float) * (size_t)(V > 0 ? V : 1));
        uint8_t *mine = NULL;  /* this row's window, when it differs by path */
        if (path_parent) {
            mine = (uint8_t *)calloc((size_t)(V > 0 ? V : 1), 1);
            int depth = 0;
            for (int j = i; j >= 0; j = path_parent[j]) ++depth;
            int take = depth < W ? depth : W;   /* path drafts in the window */
            for (int w = take; w < W; ++w) mine[history[w]] = 1;
            int pos = depth;                     /* 1-based position of j on the path */
            for (int j = i; j >= 0; j = path_parent[j], --pos)
                if (pos > depth - take && path_draft[j] >= 0 && path_draft[j] < V) mine[path_draft[j]] = 1;
        }
        const uint8_t *win = mine ? mine : inwin;
        if (!row || (path_parent && !mine)) {
#pragma omp atomic write
            err = 2;
            free(row);
            free(mine);
            continue;
        }
        float m = -INFINITY;
        int arg = -1;
        for (int vv = 0; vv < V; ++vv) {
            float l = logits[(size_t)i * V + vv];
            if (win[vv]) {
                if (l > 0.0f) l = (float)((double)l / (double)theta);
                else          l = (float)((double)l * (double)theta);
            }
            l = (float)((double)l / (double)temperature);
            row[vv] = l;
            if (arg < 0 || l > m) { m = l; arg = vv; }
        }
        double thr = (double)m + log_min_p;
        int cnt = 0;
        for (int vv = 0; vv < V; ++vv)
            if ((double)row[vv] >= thr) ++cnt;
        target[i] = arg;
        kept[i] = cnt;
        if (pen_out) memcpy(pen_out + (size_t)i * V, row, sizeof(float) * (size_t)V);
        free(row);
        free(mine);
    }
    free(inwin);
    return err;
}

int oracle_penalty_minp(const float *logits, int T, int V, const int32_t *history, int W,
                        float theta, float temperature, double log_min_p,
                        int32_t *target, int32_t *kept, float *pen_out)
{
    return oracle_penalty_minp_path(logits, T, V, history, W, NULL, NULL, theta, temperature, log_min_p, target,
                                    kept, pen_out);
}

/* ---------------------------------------------------------------------- */
/* Exact-match acceptance along every tree / n-gram path ("How it works":  */
/* a draft counts only when it equals the target token; a longest        */
/* drafts is kept -- here the lowest row among them).                      */
/*   expected(i) = parent[i] >= 0 ? target[parent[i]] : anchor              */
/*   acc(i) = draft[i] == expected(i) && (parent[i] < 0 || acc(parent[i]))  */
/*   depth(root) = 1, depth(i) = depth(parent[i]) + 1                       */
/*   L = max depth over accepted rows (0 if none); best = lowest such row;  */
/*   bonus = L > 0 ? target[best] : anchor; path = root..best.              */
/*   result = {L, best, bonus, status}; path int32[T], unused entries -1.   */
/* ---------------------------------------------------------------------- */
/* The pages keep a random longest accepted draft ("How it works").       */
/* With choose != 0 the kept row is drawn uniformly from the m accepted rows  */
/* of depth L, listed in ascending row order S[0..m): index                   */
/*   j = floor(x * m / 2^64)   (the high word of the 128-bit product)         */
/* with x = word 0 of Philox4x64-10 (below) at counter (0, 0, offset, 1) under */
/* key (seed, 0) -- the last counter word keeps this draw apart from the       */
/* token draws of oracle_sample, which use 0 there.  choose == 0 keeps S[0].   */
void oracle_philox4x64(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]);

int oracle_accept_ex(const int32_t *draft, const int32_t *parent, const int32_t *target, int T,
                     int32_t anchor, int choose, uint64_t seed, uint64_t offset,
                     int32_t *result, int32_t *path)
{
    for (int i = 0; i < T; ++i) path[i] = -1;
    for (int i = 0; i < T; ++i)
        if (parent[i] < -1 || parent[i] >= i) {
            result[0] = 0; result[1] = -1; result[2] = anchor; result[3] = 5;
            return 1;
        }
    int *acc = (int *)calloc((size_t)(T > 0 ? T : 1), sizeof(int));
    int *depth = (int *)calloc((size_t)(T > 0 ? T : 1), sizeof(int));
    int L = 0, best = -1;
    for (int i = 0; i < T; ++i) {
        int p = parent[i];
        int32_t expected = p >= 0 ? target[p] : anchor;
        acc[i] = (draft[i] == expected) && (p < 0 || acc[p]);
        depth[i] = p >= 0 ? depth[p] + 1 : 1;
        if (acc[i] && depth[i] > L) { L = depth[i]; best = i; }
    }
    if (choose && L > 0) {
        uint64_t m = 0;
        for (int i = 0; i < T; ++i) m += (acc[i] && depth[i] == L);
        const uint64_t ctr[4] = {0, 0, offset, 1}, key[2] = {seed, 0};
        uint64_t x[4];
        oracle_philox4x64(ctr, key, x);
        const uint64_t j = (uint64_t)(((unsigned __int128)x[0] * m) >> 64);
        uint64_t seen = 0;
        for (int i = 0; i < T; ++i)
            if (acc[i] && depth[i] == L) {
                if (seen == j) { best = i; break; }
                ++seen;
            }
    }
    result[0] = L;
    result[1] = best;
    result[2] = L > 0 ? target[best] : anchor;
    result[3] = 0;
    for (int j = best, pos = L - 1; j >= 0; j = parent[j], --pos) path[pos] = j;
    free(acc);
    free(depth);
    return 0;
}

int oracle_accept(const int32_t *draft, const int32_t *parent, const int32_t *target, int T,
                  int32_t anchor, int32_t *result, int32_t *path)
{
    return oracle_accept_ex(draft, parent, target, T, anchor, 0, 0, 0, result, path);
}

/* ---------------------------------------------------------------------- */
/* Commit of the accepted path (the kept draft becomes the continuation of */
/* the sequence, "How it works" on the TokenSwift tool listing).            */
/*   L = result[0]; for i < L and every KV head g:                          */
/*     cache'[g][N + i] = cache[g][N + path[i]]                              */
/*   (all sources read before any row is written).  0 <= L <= T and a path  */
/*   strictly increasing inside [0, T) are required; otherwise nothing moves */
/*   and *status = 5 (data error).  cache is one of K or V, bf16 bits.      */
int oracle_commit(uint16_t *cache, int64_t ld, int64_t N, int T, int Hkv, int d,
                  const int32_t *result, const int32_t *path, int32_t *status)
{
    const int L = result[0];
    *status = 0;
    int ok = L >= 0 && L <= T;
    for (int i = 0; ok && i < L; ++i)
        if (path[i] < 0 || path[i] >= T || (i > 0 && path[i - 1] >= path[i])) ok = 0;
    if (!ok) {
        *status = 5;
        return 0;
    }
    if (L == 0) return 0;
    uint16_t *tmp = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)L * d);
    if (!tmp) return 1;
    for (int g = 0; g < Hkv; ++g) {
        uint16_t *base = cache + ((size_t)g * ld + (size_t)N) * d;
        for (int i = 0; i < L; ++i)
            memcpy(tmp + (size_t)i * d, base + (size_t)path[i] * d, sizeof(uint16_t) * (size_t)d);
        memcpy(base, tmp, sizeof(uint16_t) * (size_t)L * d);
    }
    free(tmp);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Min-p sampling at a temperature (model card flags --min_p 0.1           */
/* --temperature 1.0: the method samples its target tokens).               */
/*                                                                          */
/* Random numbers: Philox4x64-10, the counter-based generator of Salmon,   */
/* Moraes, Dror and Shaw ("Parallel random numbers: as easy as 1, 2, 3",    */
/* SC 2011): ten rounds of                                                  */
/*   (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2   (128-bit products)        */
/*   c = (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0)                           */
/* with the key advanced by the Weyl increments (W0, W1) before every round */
/* after the first.                                                         */
void oracle_philox4x64(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4])
{
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
    uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3], k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) { k0 += W0; k1 += W1; }
        const unsigned __int128 p0 = (unsigned __int128)M0 * c0, p1 = (unsigned __int128)M1 * c2;
        const uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
        const uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
        const uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Natural logarithm in fp32 for normal x > 0, every step an IEEE fp32      */
/* operation (no contraction): x = 2^e m, m in [sqrt(1/2), sqrt(2));         */
/* ln m = 2 atanh(s), s = (m - 1)/(m + 1), by the series                    */
/* 2s (1 + s^2/3 + s^4/5 + ... + s^10/11) (|s| <= 0.1716, truncation below  */
/* 1e-10 relative); ln x = e ln 2 + ln m.                                   */
float oracle_ln_f32(float x)
{
    uint32_t b;
    memcpy(&b, &x, 4);
    int e = (int)((b >> 23) & 0xff) - 127;
    const uint32_t mb = (b & 0x7fffffu) | 0x3f800000u;
    float m;
    memcpy(&m, &mb, 4);
    if (m > 0x1.6a09e6p+0f) { m = m * 0.5f; e += 1; }
    const float s = (m - 1.0f) / (m + 1.0f);
    const float z = s * s;
    float p = fmaf(z, 0x1.745d18p-4f, 0x1.c71c72p-4f);
    p = fmaf(z, p, 0x1.24924ap-3f);
    p = fmaf(z, p, 0x1.99999ap-3f);
    p = fmaf(z, p, 0x1.555556p-2f);
    p = fmaf(z, p, 1.0f);
    const float lm = (2.0f * s) * p;
    return fmaf((float)e, 0x1.62e430p-1f, lm);
}

/* Sampled target of every row from its final (penalised, tempered) fp32    */
/* logits l[0..V): the min-p kept set K = {v : (double)l_v >= m + ln min_p}  */
/* (m = max l), and the Gumbel-max draw                                      */
/*   target = argmax_{v in K} (l_v + G_v),  G_v = -ln(-ln U_v)               */
/* (lowest id on equal keys), which draws v with probability proportional to */
/* exp(l_v) over K.  U_v = (2 (x >> 41) + 1) 2^-24 (exact in fp32, inside    */
/* (0, 1)) with x = word (v mod 4) of Philox4x64-10 at counter               */
/* (v / 4, row, offset, 0) and key (seed, 0).                                */
int oracle_sample(const float *pen, int T, int V, double log_min_p, uint64_t seed, uint64_t offset,
                  int32_t *sampled)
{
#pragma omp parallel for schedule(static)
    for (int i = 0; i < T; ++i) {
        const float *row = pen + (size_t)i * V;
        float m = -INFINITY;
        for (int vv = 0; vv < V; ++vv)
            if (row[vv] > m) m = row[vv];
        const double thr = (double)m + log_min_p;
        float best = -INFINITY;
        int arg = -1;
        for (int vv = 0; vv < V; ++vv) {
            if (!((double)row[vv] >= thr)) continue;
            const uint64_t ctr[4] = {(uint64_t)(vv >> 2), (uint64_t)i, offset, 0};
            const uint64_t key[2] = {seed, 0};
            uint64_t out[4];
            oracle_philox4x64(ctr, key, out);
            const uint64_t x = out[vv & 3];
            const float u = (float)(2u * (uint32_t)(x >> 41) + 1u) * 0x1p-24f;
            const float g = -oracle_ln_f32(-oracle_ln_f32(u));
            const float k = row[vv] + g;
            if (arg < 0 || k > best) { best = k; arg = vv; }
        }
        sampled[i] = arg;
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* 4-gram table of the generated text and top-k retrieval ("How it works"  */
/* on the TokenSwift tool listing: the top-k candidate 4-grams form draft  */
/* tokens and the n-gram table is updated after every step; the summary's */
/* "Approach": n-gram retrieval from the generated text).                   */
/*   count(w) = #{p in [3, n) : seq[p-3..p] = w}  (the table after seq).     */
/*   For an anchor a (the next token, which every draft root must equal):   */
/*   the 4-grams w with w0 = a and count(w) > 0, by count descending, then   */
/*   (w1, w2, w3) ascending; the first k of them.  Returns how many were     */
/*   found (<= k) in *found; chains[i][0..4) = w, counts[i] = count(w).      */
typedef struct { int32_t w[3]; int32_t c; } ngram3_t;

static int by_tail(const void *x, const void *y)
{
    const int32_t *a = ((const ngram3_t *)x)->w, *b = ((const ngram3_t *)y)->w;
    for (int i = 0; i < 3; ++i)
        if (a[i] != b[i]) return a[i] < b[i] ? -1 : 1;
    return 0;
}
static int by_count_then_tail(const void *x, const void *y)
{
    const ngram3_t *a = (const ngram3_t *)x, *b = (const ngram3_t *)y;
    if (a->c != b->c) return a->c > b->c ? -1 : 1;
    return by_tail(x, y);
}

int oracle_ngram_topk(const int32_t *seq, int64_t n, int32_t anchor, int k, int32_t *chains, int32_t *counts,
                      int32_t *found)
{
    *found = 0;
    if (n < 4 || k <= 0) return 0;
    ngram3_t *g = (ngram3_t *)malloc(sizeof(ngram3_t) * (size_t)(n - 3));
    if (!g) return 1;
    int64_t m = 0;
    for (int64_t p = 3; p < n; ++p)
        if (seq[p - 3] == anchor) {
            g[m].w[0] = seq[p - 2]; g[m].w[1] = seq[p - 1]; g[m].w[2] = seq[p]; g[m].c = 1;
            ++m;
        }
    qsort(g, (size_t)m, sizeof(ngram3_t), by_tail);
    int64_t u = 0;  /* distinct tails with their counts */
    for (int64_t i = 0; i < m; ++i) {
        if (u > 0 && by_tail(&g[u - 1], &g[i]) == 0) ++g[u - 1].c;
        else g[u++] = g[i];
    }
    qsort(g, (size_t)u, sizeof(ngram3_t), by_count_then_tail);
    const int take = (int)(u < k ? u : k);
    for (int i = 0; i < take; ++i) {
        chains[4 * i] = anchor;
        for (int j = 0; j < 3; ++j) chains[4 * i + 1 + j] = g[i].w[j];
        counts[i] = g[i].c;
    }
    *found = take;
    free(g);
    return 0;
}
