/*
 * ts.h -- C ABI of the TokenSwift attention-side hot path on NVIDIA B300 (sm_103a).
 *
 * TokenSwift ("From Hours to Minutes: Lossless Acceleration of Ultra Long
 * Sequence Generation up to 100K Tokens", ICML 2025) drafts with the target
 * model over a partial KV cache, verifies a draft tree plus n-gram candidates
 * against the full KV cache, and keeps the longest draft that exactly matches
 * the target tokens.  This library implements the per-step work of that loop
 * that touches the KV cache and the vocabulary:
 *
 *   ts_tree_attn             tree-masked GQA attention over a bf16 KV cache
 *                            (verify pass over the full cache; draft pass over
 *                            the partial cache), split over the KV length with
 *                            a log-sum-exp merge, optional fused chunk scores;
 *   ts_tree_attn_unmerged/_merge  the same in two halves (attention, merge);
 *   ts_tree_attn_partial     the drafting pass over the compact partial cache
 *                            (per-KV-head count of gathered tokens);
 *   ts_score_chunks          query-key importance of every 64-token KV chunk;
 *   ts_rescore_tail          the same for the chunks a commit touched only;
 *   ts_select_gather         top-k chunks up to the retrieval budget, gathered
 *                            into a compact partial cache;
 *   ts_select_chunks         the selection alone;
 *   ts_gather_tree_attn      the gather fused with the drafting pass over the
 *                            gathered cache (the chosen K/V read once);
 *   ts_select_gather_tree_attn  the selection, the gather and the drafting
 *                            pass in one kernel;
 *   ts_penalty_minp_verify   windowed contextual penalty, temperature, min-p,
 *                            greedy target and exact-match acceptance.
 *   ts_penalty_minp_sample_verify  the same with min-p sampled targets;
 *   ts_commit_path           the accepted path's K/V rows become the
 *                            continuation of the full cache;
 *   ts_ngram_update/_topk    the n-gram table of the generated text and its
 *                            top-k 4-grams for the next anchor.
 *
 * Conventions shared by every call:
 *   - Pointers without a _host suffix are device memory owned by the caller.
 *     The library never allocates, frees or synchronizes: it validates its
 *     arguments on the host, enqueues kernels on `stream` and returns.
 *     Results are valid once the stream has reached that point.
 *   - bf16 tensors are raw IEEE bfloat16 (uint16 bit patterns).  Every device
 *     pointer must be 16-byte aligned.
 *   - Q/O layout [T][Hq][d]; K/V layout [Hkv][ld_kv][d] (row stride d, head
 *     stride ld_kv*d).  A cache holds N prefix tokens in rows [0, N) and the
 *     speculative batch's own T rows in [N, N+T), so ld_kv >= N + T.
 *   - Query head h reads KV head h / (Hq/Hkv)  (grouped-query attention).
 *   - Validation errors return before anything is enqueued.  Errors that can
 *     only be seen on the device (a history id outside the vocabulary, a bad
 *     parent index) are written to a status word, never trapped.
 *   - Not thread-safe per stream: concurrent calls on different streams are
 *     fine; ts_last_error() is per host thread.
 */
#ifndef TS_H_
#define TS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ts_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
    TS_OK = 0,
    TS_ERR_INVALID_ARG = 1,  /* bad pointer, size, stride or alignment */
    TS_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement */
    TS_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    TS_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up */
    TS_ERR_DATA = 5          /* bad data found on the device (status word) */
} ts_status;

/* Message describing the last non-OK status returned on this host thread. */
const char *ts_last_error(void);

/* Library version string. */
const char *ts_version(void);

/* Number of kernels this library has launched in this process so far
 * (all devices, all streams).  Diagnostic; monotonically increasing. */
uint64_t ts_launch_count(void);

/*
 * Ancestor-or-self mask of a speculative batch ("How it works": tree-based
 * attention over the candidate tokens; the n-gram candidates are chains).
 *   parent_host: int32[T], parent_host[i] = parent row of i, or -1 for a root;
 *                requires -1 <= parent_host[i] < i (topological order).
 *   mask_host:   uint64[T][mw], mw = ts_tree_mask_words(T) = max(2, ceil(T/64));
 *                bit u of row i (word u/64, bit u%64) is set iff u == i or u
 *                is an ancestor of i.
 *   T in [0, 1024] (a [1,9,9,9] tree is 820 rows).  Host memory only; no
 *   CUDA call.
 * Errors: TS_ERR_INVALID_ARG for a null pointer, T out of range or a parent
 * index out of order.
 */
int ts_tree_mask_words(int T);
ts_status ts_tree_mask_from_parents(const int32_t *parent_host, int T, uint64_t *mask_host);

/*
 * Device workspace (bytes) ts_tree_attn needs for these sizes on the current
 * device (the split count depends on the SM count).  0 means none.
 */
size_t ts_tree_attn_workspace_bytes(int T, int Hq, int Hkv, int d, int64_t N);

/*
 * Tree-masked grouped-query attention over a bf16 KV cache: the verify pass
 * (TokenSwift tool listing, "How it works": the drafted candidates go through
 * the target model, which attends over the whole KV cache) when k/v are the
 * full cache, and the self-drafting pass when they are the partial cache.
 *
 * For batch row t and query head h, with g = h / (Hq/Hkv):
 *   s_j  = scale * q[t][h] . k[g][j]   over j in [0, N) and j = N+u for every
 *          u with bit u of mask[t] set;
 *   out[t][h] = sum_j softmax(s)_j v[g][j]            (bf16, fp32 accumulate)
 *   lse[t][h] = log sum_j exp(s_j)                     (natural log, fp32)
 *
 *   q        bf16 [T][Hq][d]
 *   k, v     bf16 [Hkv][ld_kv][d], ld_kv >= N + T
 *   mask     device uint64 [T][ts_tree_mask_words(T)] from
 *            ts_tree_mask_from_parents; every row must see itself
 *   out      bf16 [T][Hq][d]
 *   lse      fp32 [T][Hq] or NULL
 *   chunk_scores  fp32 [Hkv][ceil(N/64)] or NULL: when given, the chunk
 *            importance of ts_score_chunks for query row `score_row` is
 *            produced by the same pass (for bf16 inputs whose products and
 *            chunk sums are exact in fp32 -- e.g. small integers -- the
 *            values are identical to ts_score_chunks; otherwise they agree
 *            up to fp32 summation order).
 *   workspace at least ts_tree_attn_workspace_bytes(T, Hq, Hkv, d, N) bytes,
 *            or NULL when that is 0.
 * Supported: d in {64, 128}; Hq % Hkv == 0; Hq/Hkv <= 32; 0 <= T <= 1024;
 * N >= 0; N + T >= 1 when T >= 1.  T >= 64 with d == 128 runs on the tensor
 * cores (tcgen05, TMEM accumulators); other shapes run on the CUDA cores
 * (batches of at most 24 (row, head) pairs per KV head with d == 128, such as
 * the 4-row drafting pass, on a kernel built for them).  T == 0 is a no-op.
 */
ts_status ts_tree_attn(const void *q, const void *k, const void *v, int64_t ld_kv,
                       int64_t N, int T, int Hq, int Hkv, int d, float scale,
                       const uint64_t *mask, void *out, float *lse,
                       float *chunk_scores, int score_row,
                       void *workspace, size_t ws_bytes, ts_stream_t stream);

/*
 * ts_tree_attn in two halves, for callers that run other work between the
 * attention kernel and the merge of its split partials (the chunk selection
 * needs only the chunk scores, so it can run beside the merge on another
 * stream; the merge then needs its own workspace).
 *   ts_tree_attn_unmerged: the same arguments and checks as ts_tree_attn; it
 *     enqueues the attention kernel only.  When the plan has one split the
 *     kernel writes out / lse itself; otherwise they are written by
 *     ts_tree_attn_merge, which must follow on the same stream (or after it)
 *     with the same T, Hq, Hkv, d, N, out, lse and workspace, before the
 *     workspace is reused.  chunk_scores are complete when this half is.
 *   ts_tree_attn_merge: the log-sum-exp merge of those partials (a no-op when
 *     the plan has one split).
 * Together they produce exactly what one ts_tree_attn call produces.
 */
ts_status ts_tree_attn_unmerged(const void *q, const void *k, const void *v, int64_t ld_kv,
                                int64_t N, int T, int Hq, int Hkv, int d, float scale,
                                const uint64_t *mask, void *out, float *lse,
                                float *chunk_scores, int score_row,
                                void *workspace, size_t ws_bytes, ts_stream_t stream);
ts_status ts_tree_attn_merge(int64_t N, int T, int Hq, int Hkv, int d, void *out, float *lse,
                             const void *workspace, size_t ws_bytes, ts_stream_t stream);

/*
 * The self-drafting pass over the compact partial cache that ts_select_gather
 * wrote (tool listing, "How it works": the target model drafts from a partial
 * KV cache).  Same as ts_tree_attn over k_part/v_part with N = B, except that
 * KV head g sees only the prefix rows [0, part_len[g]): when the last chunk of
 * the full cache is short (N not a multiple of 64) and head g selected it, its
 * partial cache holds fewer than B real tokens.
 *   k_part, v_part  bf16 [Hkv][ld_part][d]: rows [0, B) the gathered tokens
 *            (valid up to part_len[g]), rows [B, B+T) the draft batch's own K/V
 *   part_len device int32 [Hkv] as ts_select_gather wrote it (values outside
 *            [0, B] are clamped to it)
 * No chunk scores.  Other arguments, sizes and errors as for ts_tree_attn;
 * the workspace size is ts_tree_attn_workspace_bytes(T, Hq, Hkv, d, B).
 */
ts_status ts_tree_attn_partial(const void *q, const void *k_part, const void *v_part, int64_t ld_part,
                               int64_t B, int T, int Hq, int Hkv, int d, float scale,
                               const uint64_t *mask, const int32_t *part_len, void *out, float *lse,
                               void *workspace, size_t ws_bytes, ts_stream_t stream);

/*
 * 1 when ts_tree_attn runs these sizes on the tensor cores (tcgen05), 0 when
 * on the CUDA cores (or the sizes are unsupported).  Setting the environment
 * variable TS_FORCE_SIMT=1 before the call forces the CUDA-core kernel.
 */
int ts_tree_attn_uses_tensor_cores(int T, int Hq, int Hkv, int d, int64_t N);

/*
 * Sticky device-side status.  A kernel whose bounded wait gave up (a
 * pipeline stall of seconds, which correct inputs never cause) finishes
 * early, leaves its outputs undefined and records TS_ERR_TIMEOUT here.
 * Returns TS_OK or that status; `clear` != 0 resets it.  This call copies
 * from the device and therefore waits for the device: a diagnostic, not a
 * hot-path call.
 */
ts_status ts_device_error(int clear);

/*
 * Self-tests of the failure paths, for tests and health checks; neither
 * faults, traps or hangs the GPU.
 *
 * ts_selftest_bounded_wait launches one warp that waits on an mbarrier no
 * thread ever arrives at, with no copy or MMA in flight.  Its bounded wait
 * gives up after budget_ns of wall-clock time (0 < budget_ns <= 1e9), records
 * TS_ERR_TIMEOUT in the sticky status that ts_device_error reads, and the
 * kernel returns: the path a stalled attention pipeline takes, exercised on
 * purpose.  The context stays usable.
 *
 * ts_selftest_fail_launches(n) makes the next n kernel launches of this
 * library fail on the host without launching (the launch reports
 * cudaErrorInvalidValue, the call returns TS_ERR_CUDA); n = 0 turns it off.
 * Process-wide; not for concurrent use with real work.
 */
ts_status ts_selftest_bounded_wait(uint64_t budget_ns, ts_stream_t stream);
void ts_selftest_fail_launches(int n);

/*
 * Allocation-free ts_tree_attn.  The pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory -- code running
 * inside another runtime's execution callback (an inference-server plugin, a
 * host function queued in someone else's stream) or a C caller without an
 * allocator, where cudaMalloc is forbidden or would synchronize the device.
 * Same arguments, semantics and results as ts_tree_attn, without the
 * workspace: the split partials go to a file-scope device array of
 * TS_NOALLOC_SCRATCH_BYTES that every GPU loading this library holds until
 * the process exits.  It never calls cudaMalloc/cudaFree.
 *   - Sizes whose ts_tree_attn_workspace_bytes exceeds the array return
 *     TS_ERR_UNSUPPORTED.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture:
 *     a first call whose stream is capturing returns TS_ERR_UNSUPPORTED.
 *   - All calls share the array: calls whose kernels overlap on the GPU race
 *     on it; calls ordered on one stream are safe.  Its contents carry over
 *     between calls and nothing in it needs clearing.
 */
#define TS_NOALLOC_SCRATCH_BYTES (64u << 20)
ts_status ts_tree_attn_noalloc(const void *q, const void *k, const void *v, int64_t ld_kv,
                               int64_t N, int T, int Hq, int Hkv, int d, float scale,
                               const uint64_t *mask, void *out, float *lse,
                               float *chunk_scores, int score_row, ts_stream_t stream);

/*
 * Query-key importance of every KV chunk (ICML 2025 summary, "Approach": the
 * partial cache keeps the chunks whose keys score highest against the query):
 *   scores[g][c] = max over the query heads h of group g of
 *                  q_row[h] . sum_{t in chunk c, t < N} k[g][t]     (unscaled fp32)
 *   q_row   bf16 [Hq][d]   (the scoring query: one row of the verify batch)
 *   k       bf16 [Hkv][ld_kv][d], ld_kv >= N
 *   scores  fp32 [Hkv][ceil(N/chunk)]
 * Supported: chunk == 64, d in {64, 128}, Hq/Hkv <= 32, N >= 0.
 */
ts_status ts_score_chunks(const void *q_row, const void *k, int64_t ld_kv, int64_t N,
                          int Hq, int Hkv, int d, int chunk, float *scores, ts_stream_t stream);

/*
 * Incremental re-scoring after a commit (tool listing, "How it works": the KV
 * cache is updated after each step; ICML 2025 summary, ablation table: the
 * partial cache is refreshed every step).  The commit appends tokens
 * [N_old, N_new) to the full cache and leaves rows below N_old untouched, so
 * the chunks that were complete at N_old keep their scores; only the chunks
 * from floor(N_old/64) on are scored again.  Afterwards scores_new equals
 * ts_score_chunks(q_row, k, N_new) exactly.
 *   scores_old  fp32 [Hkv][ceil(N_old/64)]: the scores of the same q_row over
 *               the first N_old tokens (e.g. the verify pass's fused scores,
 *               q_row = its scoring row); may be NULL when N_old < 64
 *   scores_new  fp32 [Hkv][ceil(N_new/64)]; it may be scores_old itself only
 *               when both have the same number of chunks, and must not
 *               otherwise overlap it
 * Supported: chunk == 64, d in {64, 128}, Hq/Hkv <= 32, 0 <= N_old <= N_new.
 */
ts_status ts_rescore_tail(const float *scores_old, int64_t N_old, const void *q_row, const void *k, int64_t ld_kv,
                          int64_t N_new, int Hq, int Hkv, int d, int chunk, float *scores_new,
                          ts_stream_t stream);

/*
 * Top-k chunk selection and gather into the compact partial cache
 * (retrieval budget of the model card's command line, 4096 tokens; the
 * partial cache the drafting pass reads, "How it works").
 *   Per KV head g: the k = min(budget_tokens/chunk, ceil(N/chunk)) chunks
 *   with the largest scores[g][.]; equal scores (-0 equals +0) go to the
 *   lower chunk index; sel[g][0..k) lists them in ascending order.  Then
 *     k_part[g][i*chunk + t] = k[g][sel[g][i]*chunk + t]  (same for v)
 *   for i < k, t < chunk and sel[g][i]*chunk + t < N: the last chunk of the
 *   cache holds N - 64*floor(N/64) tokens when N is not a multiple of 64, and
 *   the rows past them are not written.  That chunk has the largest index, so
 *   when selected it is the last in the partial cache and the gathered tokens
 *   of head g are the rows [0, part_len[g]).
 *   The call takes N rather than the chunk count because the length of the
 *   last chunk matters.
 *   sink_chunks, recent_chunks: the first sink_chunks and the last
 *   recent_chunks chunks are always kept (attention sinks and the recent
 *   window of the SnapKV / TriForce line of work the ICML 2025 summary builds
 *   on); the rest of the k go by score.  0, 0 is pure top-k; their sum must
 *   not exceed budget_tokens / chunk.
 *   scores  fp32 [Hkv][ceil(N/chunk)], finite
 *   k, v    bf16 [Hkv][ld_kv][d], ld_kv >= N
 *   sel     int32 [Hkv][k]
 *   part_len int32 [Hkv] or NULL: tokens gathered for head g (k*chunk, less
 *           the missing rows of a short last chunk it selected); pass it to
 *           ts_tree_attn_partial
 *   k_part, v_part  bf16 [Hkv][ld_part][d], ld_part >= k*chunk
 * Supported: chunk == 64, d in {64, 128}, budget_tokens % chunk == 0,
 * ceil(N/chunk) <= 16384.
 */
ts_status ts_select_gather(const float *scores, int Hkv, int64_t N, int budget_tokens, int chunk,
                           int sink_chunks, int recent_chunks, const void *k, const void *v, int64_t ld_kv, int d,
                           int32_t *sel, int32_t *part_len, void *k_part, void *v_part, int64_t ld_part,
                           ts_stream_t stream);

/*
 * The selection of ts_select_gather without the gather: sel and part_len as
 * there, same arguments, sizes and errors (no cache is read or written).
 */
ts_status ts_select_chunks(const float *scores, int Hkv, int64_t N, int budget_tokens, int chunk,
                           int sink_chunks, int recent_chunks, int32_t *sel, int32_t *part_len,
                           ts_stream_t stream);

/*
 * The gather of ts_select_gather fused with the drafting pass over its result
 * (tool listing, "How it works": the partial KV cache is refreshed from the
 * full cache and the target model drafts over it).  In one pass over the
 * selected chunks it
 *   - writes k_part[g][i*64 + t] = k[g][sel[g][i]*64 + t] (and v) for i < k_sel,
 *     t < 64 and sel[g][i]*64 + t < N, exactly as ts_select_gather's gather
 *     (other rows of k_part / v_part are not written), and
 *   - computes ts_tree_attn_partial(q, k_part, v_part, ld_part, B = 64*k_sel,
 *     T, ..., part_len) over the gathered rows, where part_len[g] = B less the
 *     rows a selected short last chunk lacks; the batch's own K/V rows must
 *     already be in rows [B, B+T) of k_part / v_part.
 * The output equals ts_select_gather followed by ts_tree_attn_partial bit for
 * bit.
 *   q        bf16 [T][Hq][d]; k, v: the full cache, bf16 [Hkv][ld_kv][d],
 *            ld_kv >= N
 *   sel      device int32 [Hkv][k_sel] from ts_select_chunks (ascending
 *            chunk indices below ceil(N/64); values outside are clamped)
 *   k_part, v_part  bf16 [Hkv][ld_part][d], ld_part >= 64*k_sel + T
 *   mask, out, lse, scale: as ts_tree_attn
 *   workspace  ts_tree_attn_workspace_bytes(T, Hq, Hkv, d, 64*k_sel) bytes
 * Supported: d == 128 and T*Hq/Hkv <= 24 (the drafting pass's shapes),
 * 1 <= k_sel <= ceil(N/64).  Chunk size 64.
 */
ts_status ts_gather_tree_attn(const void *q, const void *k, const void *v, int64_t ld_kv, int64_t N,
                              const int32_t *sel, int k_sel, void *k_part, void *v_part, int64_t ld_part,
                              int T, int Hq, int Hkv, int d, float scale, const uint64_t *mask,
                              void *out, float *lse, void *workspace, size_t ws_bytes, ts_stream_t stream);

/*
 * ts_select_chunks and ts_gather_tree_attn in one pass: every CTA of the
 * drafting kernel selects its KV head's chunks from `scores` itself (the same
 * radix selection as ts_select_chunks), then gathers the chunks it attends
 * over.  sel and part_len are written as ts_select_chunks writes them; the
 * compact cache, out and lse are those of ts_gather_tree_attn with that sel.
 * Arguments, sizes and errors: those of ts_select_chunks (scores, N,
 * budget_tokens, chunk, sink_chunks, recent_chunks, sel, part_len) and of
 * ts_gather_tree_attn (the rest; k_sel = min(budget_tokens/chunk,
 * ceil(N/chunk)), at least 1).
 */
ts_status ts_select_gather_tree_attn(const float *scores, int64_t N, int budget_tokens, int chunk,
                                     int sink_chunks, int recent_chunks, int32_t *sel, int32_t *part_len,
                                     const void *q, const void *k, const void *v, int64_t ld_kv,
                                     void *k_part, void *v_part, int64_t ld_part, int T, int Hq, int Hkv, int d,
                                     float scale, const uint64_t *mask, void *out, float *lse,
                                     void *workspace, size_t ws_bytes, ts_stream_t stream);

/*
 * Vocabulary side of one verification step (model card flags --penalty,
 * --penalty_length, --min_p, --temperature; "How it works": exact-match
 * verification, one longest valid draft kept).
 *   For every batch row i of logits (fp32 [T][V]):
 *     a token id in history[0..W) (counted once) has l > 0 ? l/theta : l*theta;
 *     then l / temperature;  m = max;  target[i] = lowest id attaining m;
 *     kept[i] = #{v : l_v >= m + ln(min_p)}   (min-p: p_v >= min_p * p_max;
 *     the comparison is exact: ln(min_p) is taken in double on the host and
 *     m + ln(min_p) rounded up to fp32).
 *   Then acceptance along the parent forest: row i is accepted iff
 *     draft[i] == (parent[i] >= 0 ? target[parent[i]] : anchor) and its parent
 *     is accepted; L = the largest depth (roots have depth 1) of an accepted
 *     row, best = the lowest such row, bonus = L > 0 ? target[best] : anchor.
 *   result int32[4] = {L, best (-1 if L == 0), bonus, status}; status is
 *     TS_OK, TS_ERR_DATA if a history id is outside [0, V) or a parent
 *     index is out of order, or TS_ERR_TIMEOUT if a row's copy of its logits
 *     into shared memory never completed (a bounded wait gave up; that row's
 *     kept count reads -1).
 *   path   int32[T]: rows root..best in path[0..L), -1 after.
 *   draft, parent: int32 [T] device.  history: int32 [W] device (W >= 0).
 *   workspace: unused, pass NULL / 0.
 * Supported: 1 <= T <= 1024, 1 <= V <= 163840, theta > 0, temperature > 0,
 * 0 <= min_p <= 1.
 */
ts_status ts_penalty_minp_verify(const float *logits, int T, int V, const int32_t *history, int W,
                                 float theta, float min_p, float temperature,
                                 const int32_t *draft, const int32_t *parent, int32_t anchor,
                                 int32_t *target, int32_t *kept, int32_t *result, int32_t *path,
                                 void *workspace, size_t ws_bytes, ts_stream_t stream);

/*
 * The vocabulary step with options; ts_penalty_minp_verify is flags = 0 and
 * ts_penalty_minp_sample_verify is flags = TS_VOCAB_SAMPLE.
 *   TS_VOCAB_SAMPLE       min-p sampled targets and a uniformly drawn longest
 *                         path, from (seed, offset), as described below.
 *   TS_VOCAB_PATH_WINDOW  row i's logits follow the drafts on its path, so its
 *                         penalty window is the last W tokens of
 *                         history ++ (draft of the root, ..., draft[i]):
 *                         history[min(d_i, W)..W) plus the path's last
 *                         min(d_i, W) drafts, d_i = depth of row i (roots 1);
 *                         draft ids outside [0, V) (e.g. -1 of an unused
 *                         n-gram row) add nothing.
 */
#define TS_VOCAB_SAMPLE 1u
#define TS_VOCAB_PATH_WINDOW 2u
ts_status ts_vocab_verify(const float *logits, int T, int V, const int32_t *history, int W, float theta, float min_p,
                          float temperature, unsigned flags, uint64_t seed, uint64_t offset, const int32_t *draft,
                          const int32_t *parent, int32_t anchor, int32_t *target, int32_t *kept, int32_t *result,
                          int32_t *path, ts_stream_t stream);

/*
 * The same step with sampled targets (model card: --min_p 0.1 with
 * --temperature 1.0 samples; "How it works": drafts are checked against the
 * target tokens).  Identical to ts_penalty_minp_verify except that
 *   target[i] = argmax over the min-p kept ids v of (l_v + G_v),
 *   G_v = -ln(-ln U_v)   (Gumbel-max: v is drawn with probability
 *                         proportional to exp(l_v) over the kept ids),
 * lowest id on equal keys, where l are the final (penalised, tempered) fp32
 * logits, U_v = (2 (x >> 41) + 1) * 2^-24 and x is word (v % 4) of
 * Philox4x64-10 (Salmon et al., SC 2011) at counter (v / 4, i, offset, 0)
 * under key (seed, 0); ln is evaluated in fp32 as ln x = e ln 2 + 2 atanh(s),
 * s = (m - 1)/(m + 1), x = 2^e m, m in [sqrt(1/2), sqrt(2)), with the series
 * s (1 + s^2/3 + ... + s^10/11), every operation an IEEE fp32 one.
 * Acceptance then uses these sampled targets, and the kept row among the m
 * longest accepted rows S (ascending row order) is drawn uniformly ("How it
 * works": a random longest accepted draft is kept):
 * best = S[floor(x m / 2^64)], x = word 0 of Philox4x64-10 at counter
 * (0, 0, offset, 1) under key (seed, 0).  kept, result and path as for
 * ts_penalty_minp_verify.
 */
ts_status ts_penalty_minp_sample_verify(const float *logits, int T, int V, const int32_t *history, int W,
                                        float theta, float min_p, float temperature, uint64_t seed,
                                        uint64_t offset, const int32_t *draft, const int32_t *parent,
                                        int32_t anchor, int32_t *target, int32_t *kept, int32_t *result,
                                        int32_t *path, ts_stream_t stream);

/*
 * Commit of the accepted path into the full cache, the step after
 * verification ("How it works" on the TokenSwift tool listing: the longest
 * valid draft is kept and generation continues from it).  Reads L =
 * result[0] and path[0..L) as ts_penalty_minp_verify wrote them (device
 * memory: no host round trip) and moves the accepted batch rows to the front
 * of the batch region, for every KV head g:
 *     k[g][N + i] = k[g][N + path[i]]   (same for v),   i < L,
 * so rows [0, N + L) of the cache are the sequence afterwards; rows
 * N + L .. N + T - 1 keep stale values.  path must be strictly increasing
 * with values in [0, T) (root..best of a topologically ordered forest) and
 * 0 <= L <= T; otherwise nothing moves and result[3] is set to TS_ERR_DATA.
 *   k, v    bf16 [Hkv][ld_kv][d], ld_kv >= N + T (updated in place)
 *   result  int32[4] device (result[0] read, result[3] written on a data error)
 *   path    int32[T] device
 * Supported: 1 <= T <= 1024, d in {64, 128}.
 */
ts_status ts_commit_path(void *k, void *v, int64_t ld_kv, int64_t N, int T, int Hkv, int d, int32_t *result,
                         const int32_t *path, ts_stream_t stream);

/*
 * n-gram table of the generated text and top-k 4-gram retrieval (TokenSwift
 * tool listing, "How it works": the top-k candidate 4-grams become draft
 * tokens and the n-gram table is updated after every step; model card:
 * --ngram_topk 20 --gamma 4).
 *
 * The table counts every 4-gram w = seq[p-3..p] of the sequence added to it.
 * The candidates for an anchor a (the token every draft root must equal) are
 * the 4-grams with w0 = a, by count descending, then (w1, w2, w3) ascending.
 *
 * Layout (caller-owned device memory, ts_ngram_table_bytes(capacity) bytes,
 * 16-byte aligned): int32 keys [capacity][4] (all ones = empty slot), int32
 * counts [capacity], int32 first [capacity] (start position of the 4-gram's
 * first occurrence).  capacity is a power of two in [64, 2^30]; keep it at
 * least twice the number of distinct 4-grams (a sequence of n tokens has at
 * most n - 3).  Open addressing with linear probing from a hash of all four
 * tokens.
 *
 * ts_ngram_reset   empties the table.
 * ts_ngram_update  adds the windows that end at positions [max(3, n_old),
 *                  n_new) of seq (device int32 [n_new], ids >= 0,
 *                  n_new < 2^31): call it with the old and new lengths after
 *                  each commit.  A full table or a negative id sets *status
 *                  (device int32) to TS_ERR_DATA; otherwise *status is left
 *                  as it was.
 * ts_ngram_topk    the top k 4-grams of seq[0, n) that start with the anchor;
 *                  the table must hold exactly the windows of seq[0, n).  It
 *                  reads the anchor from device memory (e.g. the bonus token
 *                  result + 2 of ts_penalty_minp_verify: no host round trip),
 *                  scans seq for it and takes each distinct 4-gram once (at
 *                  its first occurrence) with its count from the table.  It
 *                  writes chains int32 [k][4] (w0..w3 of the i-th candidate;
 *                  -1 past the last one), counts int32 [k] (0 past the last
 *                  one) and found (device int32: how many, <= k).  chains can
 *                  point straight at the draft tokens of the verify batch's
 *                  chain rows.  1 <= k <= 1024.
 */
size_t ts_ngram_table_bytes(int64_t capacity);
ts_status ts_ngram_reset(void *table, int64_t capacity, ts_stream_t stream);
ts_status ts_ngram_update(void *table, int64_t capacity, const int32_t *seq, int64_t n_old, int64_t n_new,
                          int32_t *status, ts_stream_t stream);
ts_status ts_ngram_topk(const void *table, int64_t capacity, const int32_t *seq, int64_t n, const int32_t *anchor,
                        int k, int32_t *chains, int32_t *counts, int32_t *found, ts_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TS_H_ */
