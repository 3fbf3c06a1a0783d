// C ABI of the ts library: argument validation, planning and kernel launch.
// Every entry point validates on the host and returns before enqueuing
// anything when an argument is wrong; nothing here allocates, frees or
// synchronizes.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

#include "../../include/ts.h"
#include "internal.h"
#include "ts_common.cuh"

namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_inject_failures{0};  // launches still to fail (ts_selftest_fail_launches)

ts_status fail(ts_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

ts_status cuda_fail(cudaError_t e, const char *where) {
    return fail(TS_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void *p) { return ((uintptr_t)p & 3u) == 0; }

// SM count of the current device (148 on B300); cached per device.
int num_sms() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 148;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 148;
        }
        cache[dev] = n;
    }
    return cache[dev];
}

bool force_simt() {
    const char *e = getenv("TS_FORCE_SIMT");
    return e != nullptr && e[0] == '1';
}

// Which kernel runs and how the KV length is split; used both to size the
// workspace and to launch, so the two always agree.
struct AttnPlan {
    bool tc;     // tensor cores (T >= 64, head dim 128)
    bool small;  // CUDA cores, small batch (T * G <= 24, head dim 128)
    ts::TcPlan tcp;
    ts::SimtPlan sp;
    int splits;
};

AttnPlan plan_attention(int T, int Hq, int Hkv, int d, int64_t N) {
    AttnPlan p{};
    const int sms = num_sms();
    p.tcp = ts::tc_plan(T, Hq, Hkv, d, N, sms);
    p.tc = p.tcp.ok && !force_simt();
    p.small = !p.tc && ts::small_ok(T, Hq, Hkv, d);
    if (p.tc) {
        p.splits = p.tcp.splits;
    } else if (p.small) {
        p.splits = ts::small_splits(T, N);
    } else {
        p.sp = ts::simt_plan(T, Hq, Hkv, d, N, sms);
        p.splits = p.sp.splits;
    }
    return p;
}

size_t workspace_for(const AttnPlan &p, int T, int Hq, int d) {
    return p.splits > 1 ? (size_t)p.splits * T * Hq * ((size_t)d + 2) * sizeof(float) : 0;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

// 3-D bf16 tensor map with 128-byte swizzle: dims/strides innermost first.
bool encode_map(CUtensorMap *m, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
                uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

ts_status check_attn_shape(int T, int Hq, int Hkv, int d, int64_t N) {
    if (d != 64 && d != 128) return fail(TS_ERR_UNSUPPORTED, "head dim d=%d (supported: 64, 128)", d);
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
        return fail(TS_ERR_INVALID_ARG, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
    if (Hq / Hkv > 32) return fail(TS_ERR_UNSUPPORTED, "group size Hq/Hkv=%d > 32", Hq / Hkv);
    if (T < 0 || T > ts::TS_MAX_T) return fail(TS_ERR_UNSUPPORTED, "T=%d outside [0, %d]", T, ts::TS_MAX_T);
    if (N < 0) return fail(TS_ERR_INVALID_ARG, "N=%lld < 0", (long long)N);
    if (N > (int64_t)1 << 30) return fail(TS_ERR_UNSUPPORTED, "N=%lld too large", (long long)N);
    return TS_OK;
}

}  // namespace

namespace ts {
void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
bool injected_launch_failure() {
    int n = g_inject_failures.load(std::memory_order_relaxed);
    while (n > 0)
        if (g_inject_failures.compare_exchange_weak(n, n - 1, std::memory_order_relaxed)) return true;
    return false;
}
ts_status report_error(ts_status st, const char *msg) { return fail(st, "%s", msg ? msg : "error"); }
}  // namespace ts

extern "C" {

uint64_t ts_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *ts_last_error(void) { return g_last_error.c_str(); }

const char *ts_version(void) { return "ts 0.1 (sm_103a)"; }

int ts_tree_mask_words(int T) { return T < 0 ? 0 : ts::mask_words(T); }

ts_status ts_tree_mask_from_parents(const int32_t *parent_host, int T, uint64_t *mask_host) {
    if (T < 0 || T > ts::TS_MAX_T) return fail(TS_ERR_INVALID_ARG, "T=%d outside [0, %d]", T, ts::TS_MAX_T);
    if (T > 0 && (parent_host == nullptr || mask_host == nullptr))
        return fail(TS_ERR_INVALID_ARG, "null parent or mask pointer");
    for (int i = 0; i < T; ++i)
        if (parent_host[i] < -1 || parent_host[i] >= i)
            return fail(TS_ERR_INVALID_ARG, "parent[%d]=%d must satisfy -1 <= parent[i] < i", i, parent_host[i]);
    const int mw = ts::mask_words(T);
    for (int i = 0; i < T; ++i) {
        // a row's ancestors are its parent's ancestors plus the parent itself
        uint64_t *row = mask_host + (size_t)mw * i;
        const int p = parent_host[i];
        for (int w = 0; w < mw; ++w) row[w] = p >= 0 ? mask_host[(size_t)mw * p + w] : 0;
        row[i >> 6] |= 1ull << (i & 63);
    }
    return TS_OK;
}

size_t ts_tree_attn_workspace_bytes(int T, int Hq, int Hkv, int d, int64_t N) {
    if (check_attn_shape(T, Hq, Hkv, d, N) != TS_OK || T == 0) return 0;
    return workspace_for(plan_attention(T, Hq, Hkv, d, N), T, Hq, d);
}

ts_status ts_device_error(int clear) {
    int v = 0;
    cudaError_t e = ts::read_device_error(&v, clear != 0);
    if (e != cudaSuccess) return cuda_fail(e, "ts_device_error");
    if (v != 0) return fail((ts_status)v, "a kernel reported device status %d (bounded wait gave up)", v);
    return TS_OK;
}

ts_status ts_selftest_bounded_wait(uint64_t budget_ns, ts_stream_t stream) {
    if (budget_ns == 0 || budget_ns > 1000000000ull)
        return fail(TS_ERR_INVALID_ARG, "budget_ns=%llu outside (0, 1e9]", (unsigned long long)budget_ns);
    cudaError_t e = ts::launch_bounded_wait_selftest(budget_ns, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "bounded_wait_selftest launch");
    ts::note_launches(1);
    return TS_OK;
}

void ts_selftest_fail_launches(int n) { g_inject_failures.store(n > 0 ? n : 0, std::memory_order_relaxed); }

int ts_tree_attn_uses_tensor_cores(int T, int Hq, int Hkv, int d, int64_t N) {
    if (check_attn_shape(T, Hq, Hkv, d, N) != TS_OK || T == 0) return 0;
    return plan_attention(T, Hq, Hkv, d, N).tc ? 1 : 0;
}

}  // extern "C"

// Shared body of ts_tree_attn and ts_tree_attn_partial.
static ts_status tree_attn_impl(const void *q, const void *k, const void *v, int64_t ld_kv, int64_t N, int T,
                                int Hq, int Hkv, int d, float scale, const uint64_t *mask,
                                const int32_t *prefix_len, void *out, float *lse, float *chunk_scores,
                                int score_row, void *workspace, size_t ws_bytes, ts_stream_t stream,
                                const ts::SmallGather *gather = nullptr, bool merge = true) {
    ts_status st = check_attn_shape(T, Hq, Hkv, d, N);
    if (st != TS_OK) return st;
    if (T == 0) return TS_OK;
    if (!q || !k || !v || !mask || !out) return fail(TS_ERR_INVALID_ARG, "null q/k/v/mask/out");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return fail(TS_ERR_INVALID_ARG, "q/k/v/out must be 16-byte aligned");
    if (!aligned4(mask) || (lse && !aligned4(lse)) || (chunk_scores && !aligned4(chunk_scores)) ||
        (prefix_len && !aligned4(prefix_len)))
        return fail(TS_ERR_INVALID_ARG, "mask/lse/chunk_scores/prefix_len misaligned");
    if (ld_kv < N + T) return fail(TS_ERR_INVALID_ARG, "ld_kv=%lld < N+T=%lld", (long long)ld_kv, (long long)(N + T));
    if (!(scale > 0.f) || !isfinite(scale)) return fail(TS_ERR_INVALID_ARG, "scale must be finite and > 0");
    if (chunk_scores && (score_row < 0 || score_row >= T))
        return fail(TS_ERR_INVALID_ARG, "score_row=%d outside [0, T=%d)", score_row, T);

    const AttnPlan plan = plan_attention(T, Hq, Hkv, d, N);
    if (gather != nullptr && !plan.small)
        return fail(TS_ERR_UNSUPPORTED, "the gather-fused drafting pass takes d = 128 and T*Hq/Hkv <= 24");
    const size_t need = workspace_for(plan, T, Hq, d);
    if (need > 0 && (workspace == nullptr || ws_bytes < need))
        return fail(TS_ERR_INVALID_ARG, "workspace of %zu bytes needed, %zu given", need, ws_bytes);
    if (need > 0 && !aligned16(workspace)) return fail(TS_ERR_INVALID_ARG, "workspace must be 16-byte aligned");

    ts::AttnArgs a{};
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k = static_cast<const __nv_bfloat16 *>(k);
    a.v = static_cast<const __nv_bfloat16 *>(v);
    a.ld_kv = ld_kv;
    a.N = N;
    a.T = T;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.d = d;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.mask = mask;
    a.mw = ts::mask_words(T);
    a.prefix_len = prefix_len;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.lse = lse;
    a.chunk_scores = chunk_scores;
    a.score_row = score_row;
    a.n_chunks = (int)((N + 63) / 64);
    a.ws_o = static_cast<float *>(workspace);
    a.ws_ml = need > 0 ? a.ws_o + (size_t)plan.splits * T * Hq * d : nullptr;
    a.splits = plan.splits;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (plan.tc) {
        const ts::TcPlan &p = plan.tcp;
        a.n_tiles = p.n_tiles;
        a.tpb = p.tpb;
        CUtensorMap tq, tk, tv;
        const uint64_t row_bytes = (uint64_t)d * 2;
        if (!encode_map(&tq, q, d, Hq, T, row_bytes, row_bytes * Hq, 64, a.G, p.tpb) ||
            !encode_map(&tk, k, d, N + T, Hkv, row_bytes, row_bytes * ld_kv, 64, ts::TC_KV_TILE, 1) ||
            !encode_map(&tv, v, d, N + T, Hkv, row_bytes, row_bytes * ld_kv, 64, ts::TC_KV_TILE, 1))
            return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled failed (or the driver entry point is missing)");
        e = ts::launch_tree_attn_tc(a, p, tq, tk, tv, s);
        if (e != cudaSuccess) return cuda_fail(e, "tree_attn_tc launch");
    } else if (plan.small) {
        e = ts::launch_tree_attn_small(a, gather, plan.splits, s);
        if (e != cudaSuccess) return cuda_fail(e, "tree_attn_small launch");
    } else {
        const ts::SimtPlan &p = plan.sp;
        a.tiles_per_split = p.tiles_per_split;
        a.n_tiles = p.n_tiles;
        a.tpb = p.tpb;
        e = ts::launch_tree_attn_simt(a, p, s);
        if (e != cudaSuccess) return cuda_fail(e, "tree_attn_simt launch");
    }
    ts::note_launches(1);
    if (plan.splits > 1 && merge) {
        ts::MergeArgs m{a.ws_o, a.ws_ml, a.out, a.lse, T, Hq, plan.splits, T, plan.splits};
        if (plan.tc) {
            // rows of pair streams have s_pair partials, rows of the single stream s_single
            m.splits = plan.tcp.s_pair;
            m.t_split = 2 * plan.tcp.n_pair * plan.tcp.tpb;
            m.splits_hi = plan.tcp.s_single;
        }
        e = ts::launch_lse_merge(m, d, s);
        if (e != cudaSuccess) return cuda_fail(e, "lse_merge launch");
        ts::note_launches(1);
    }
    return TS_OK;
}

extern "C" {

ts_status ts_tree_attn(const void *q, const void *k, const void *v, int64_t ld_kv,
                       int64_t N, int T, int Hq, int Hkv, int d, float scale,
                       const uint64_t *mask, void *out, float *lse,
                       float *chunk_scores, int score_row,
                       void *workspace, size_t ws_bytes, ts_stream_t stream) {
    return tree_attn_impl(q, k, v, ld_kv, N, T, Hq, Hkv, d, scale, mask, nullptr, out, lse, chunk_scores, score_row,
                          workspace, ws_bytes, stream);
}

ts_status ts_tree_attn_unmerged(const void *q, const void *k, const void *v, int64_t ld_kv,
                                int64_t N, int T, int Hq, int Hkv, int d, float scale,
                                const uint64_t *mask, void *out, float *lse,
                                float *chunk_scores, int score_row,
                                void *workspace, size_t ws_bytes, ts_stream_t stream) {
    return tree_attn_impl(q, k, v, ld_kv, N, T, Hq, Hkv, d, scale, mask, nullptr, out, lse, chunk_scores, score_row,
                          workspace, ws_bytes, stream, nullptr, false);
}

ts_status ts_tree_attn_merge(int64_t N, int T, int Hq, int Hkv, int d, void *out, float *lse,
                             const void *workspace, size_t ws_bytes, ts_stream_t stream) {
    ts_status st = check_attn_shape(T, Hq, Hkv, d, N);
    if (st != TS_OK) return st;
    if (T == 0) return TS_OK;
    const AttnPlan plan = plan_attention(T, Hq, Hkv, d, N);
    if (plan.splits <= 1) return TS_OK;  // the attention kernel wrote the output itself
    if (!out || !aligned16(out) || (lse && !aligned4(lse)))
        return fail(TS_ERR_INVALID_ARG, "null or misaligned out/lse");
    const size_t need = workspace_for(plan, T, Hq, d);
    if (workspace == nullptr || ws_bytes < need || !aligned16(workspace))
        return fail(TS_ERR_INVALID_ARG, "workspace of %zu bytes (16-byte aligned) needed, %zu given", need, ws_bytes);
    const float *ws_o = static_cast<const float *>(workspace);
    ts::MergeArgs m{ws_o, ws_o + (size_t)plan.splits * T * Hq * d, static_cast<__nv_bfloat16 *>(out), lse, T, Hq,
                    plan.splits, T, plan.splits};
    if (plan.tc) {
        m.splits = plan.tcp.s_pair;
        m.t_split = 2 * plan.tcp.n_pair * plan.tcp.tpb;
        m.splits_hi = plan.tcp.s_single;
    }
    cudaError_t e = ts::launch_lse_merge(m, d, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "lse_merge launch");
    ts::note_launches(1);
    return TS_OK;
}

ts_status ts_tree_attn_partial(const void *q, const void *k_part, const void *v_part, int64_t ld_part,
                               int64_t B, int T, int Hq, int Hkv, int d, float scale,
                               const uint64_t *mask, const int32_t *part_len, void *out, float *lse,
                               void *workspace, size_t ws_bytes, ts_stream_t stream) {
    if (T > 0 && part_len == nullptr) return fail(TS_ERR_INVALID_ARG, "null part_len");
    return tree_attn_impl(q, k_part, v_part, ld_part, B, T, Hq, Hkv, d, scale, mask, part_len, out, lse, nullptr,
                          0, workspace, ws_bytes, stream);
}

ts_status ts_score_chunks(const void *q_row, const void *k, int64_t ld_kv, int64_t N,
                          int Hq, int Hkv, int d, int chunk, float *scores, ts_stream_t stream) {
    if (chunk != 64) return fail(TS_ERR_UNSUPPORTED, "chunk=%d (supported: 64)", chunk);
    ts_status st = check_attn_shape(1, Hq, Hkv, d, N);
    if (st != TS_OK) return st;
    if (N == 0) return TS_OK;
    if (!q_row || !k || !scores) return fail(TS_ERR_INVALID_ARG, "null q_row/k/scores");
    if (!aligned16(q_row) || !aligned16(k) || !aligned4(scores))
        return fail(TS_ERR_INVALID_ARG, "q_row/k must be 16-byte aligned, scores 4-byte aligned");
    if (ld_kv < N) return fail(TS_ERR_INVALID_ARG, "ld_kv < N");
    cudaError_t e = ts::launch_score_chunks(static_cast<const __nv_bfloat16 *>(q_row),
                                            static_cast<const __nv_bfloat16 *>(k), ld_kv, N, Hq, Hkv, d, scores,
                                            (N + 63) / 64, 0, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "score_chunks launch");
    ts::note_launches(1);
    return TS_OK;
}

ts_status ts_rescore_tail(const float *scores_old, int64_t N_old, const void *q_row, const void *k, int64_t ld_kv,
                          int64_t N_new, int Hq, int Hkv, int d, int chunk, float *scores_new,
                          ts_stream_t stream) {
    if (chunk != 64) return fail(TS_ERR_UNSUPPORTED, "chunk=%d (supported: 64)", chunk);
    ts_status st = check_attn_shape(1, Hq, Hkv, d, N_new);
    if (st != TS_OK) return st;
    if (N_old < 0 || N_old > N_new) return fail(TS_ERR_INVALID_ARG, "need 0 <= N_old <= N_new");
    if (N_new == 0) return TS_OK;
    if (!q_row || !k || !scores_new || (N_old > 0 && !scores_old))
        return fail(TS_ERR_INVALID_ARG, "null q_row/k/scores");
    if (!aligned16(q_row) || !aligned16(k) || !aligned4(scores_new) || (scores_old && !aligned4(scores_old)))
        return fail(TS_ERR_INVALID_ARG, "q_row/k must be 16-byte aligned, scores 4-byte aligned");
    if (ld_kv < N_new) return fail(TS_ERR_INVALID_ARG, "ld_kv < N_new");
    const int nc_old = (int)((N_old + 63) / 64), nc_new = (int)((N_new + 63) / 64);
    const int c_keep = (int)(N_old / 64);  // chunks that were complete before the new tokens
    const bool in_place = scores_old == scores_new;
    if (in_place && nc_old != nc_new)
        return fail(TS_ERR_INVALID_ARG, "in-place rescoring needs ceil(N_old/64) == ceil(N_new/64)");
    if (!in_place && N_old > 0) {
        const uintptr_t a0 = (uintptr_t)scores_old, a1 = a0 + sizeof(float) * (size_t)Hkv * nc_old;
        const uintptr_t b0 = (uintptr_t)scores_new, b1 = b0 + sizeof(float) * (size_t)Hkv * nc_new;
        if (a0 < b1 && b0 < a1) return fail(TS_ERR_INVALID_ARG, "scores_old and scores_new overlap");
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (!in_place && c_keep > 0) {
        e = ts::launch_copy_scores(scores_old, nc_old, scores_new, nc_new, c_keep, Hkv, s);
        if (e != cudaSuccess) return cuda_fail(e, "copy_scores launch");
        ts::note_launches(1);
    }
    if (c_keep < nc_new) {
        e = ts::launch_score_chunks(static_cast<const __nv_bfloat16 *>(q_row), static_cast<const __nv_bfloat16 *>(k),
                                    ld_kv, N_new, Hq, Hkv, d, scores_new, nc_new, c_keep, s);
        if (e != cudaSuccess) return cuda_fail(e, "score_chunks launch");
        ts::note_launches(1);
    }
    return TS_OK;
}

// Shared checks of the selection calls; on success *k_sel is the number of
// chunks kept per head (0: nothing to do).
static ts_status check_select(const float *scores, int Hkv, int64_t N, int budget_tokens, int chunk, int sink_chunks,
                              int recent_chunks, const int32_t *sel, const int32_t *part_len, int *k_sel) {
    *k_sel = 0;
    if (chunk != 64) return fail(TS_ERR_UNSUPPORTED, "chunk=%d (supported: 64)", chunk);
    if (Hkv <= 0) return fail(TS_ERR_INVALID_ARG, "Hkv=%d", Hkv);
    if (N < 0 || budget_tokens < 0) return fail(TS_ERR_INVALID_ARG, "negative N or budget");
    if (budget_tokens % chunk) return fail(TS_ERR_INVALID_ARG, "budget %d not a multiple of chunk", budget_tokens);
    if (sink_chunks < 0 || recent_chunks < 0 || (int64_t)sink_chunks + recent_chunks > budget_tokens / chunk)
        return fail(TS_ERR_INVALID_ARG, "need sink_chunks, recent_chunks >= 0 and their sum <= budget/chunk");
    const int64_t nc = (N + chunk - 1) / chunk;
    if (nc > 16384) return fail(TS_ERR_UNSUPPORTED, "%lld chunks > 16384", (long long)nc);
    const int ks = (int)((int64_t)(budget_tokens / chunk) < nc ? budget_tokens / chunk : nc);
    if (ks == 0) return TS_OK;
    if (!scores || !sel) return fail(TS_ERR_INVALID_ARG, "null scores/sel");
    if (!aligned4(scores) || !aligned4(sel) || (part_len && !aligned4(part_len)))
        return fail(TS_ERR_INVALID_ARG, "misaligned scores/sel/part_len");
    *k_sel = ks;
    return TS_OK;
}

ts_status ts_select_gather(const float *scores, int Hkv, int64_t N, int budget_tokens, int chunk,
                           int sink_chunks, int recent_chunks, const void *k, const void *v, int64_t ld_kv, int d,
                           int32_t *sel, int32_t *part_len, void *k_part, void *v_part, int64_t ld_part,
                           ts_stream_t stream) {
    if (d != 64 && d != 128) return fail(TS_ERR_UNSUPPORTED, "head dim d=%d (supported: 64, 128)", d);
    int k_sel = 0;
    ts_status st = check_select(scores, Hkv, N, budget_tokens, chunk, sink_chunks, recent_chunks, sel, part_len,
                                &k_sel);
    if (st != TS_OK || k_sel == 0) return st;
    if (!k || !v || !k_part || !v_part) return fail(TS_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_part) || !aligned16(v_part))
        return fail(TS_ERR_INVALID_ARG, "misaligned pointer");
    if (ld_kv < N) return fail(TS_ERR_INVALID_ARG, "ld_kv < N");
    if (ld_part < (int64_t)k_sel * chunk)
        return fail(TS_ERR_INVALID_ARG, "ld_part=%lld < k*chunk=%lld", (long long)ld_part, (long long)k_sel * chunk);
    const int nc = (int)((N + chunk - 1) / chunk);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = ts::launch_select(scores, Hkv, N, nc, k_sel, sink_chunks, recent_chunks, sel, part_len, s);
    if (e != cudaSuccess) return cuda_fail(e, "select launch");
    ts::note_launches(1);
    e = ts::launch_gather(sel, Hkv, N, nc, k_sel, static_cast<const __nv_bfloat16 *>(k),
                          static_cast<const __nv_bfloat16 *>(v), ld_kv, d, static_cast<__nv_bfloat16 *>(k_part),
                          static_cast<__nv_bfloat16 *>(v_part), ld_part, s);
    if (e != cudaSuccess) return cuda_fail(e, "gather launch");
    ts::note_launches(1);
    return TS_OK;
}

ts_status ts_select_chunks(const float *scores, int Hkv, int64_t N, int budget_tokens, int chunk, int sink_chunks,
                           int recent_chunks, int32_t *sel, int32_t *part_len, ts_stream_t stream) {
    int k_sel = 0;
    ts_status st = check_select(scores, Hkv, N, budget_tokens, chunk, sink_chunks, recent_chunks, sel, part_len,
                                &k_sel);
    if (st != TS_OK || k_sel == 0) return st;
    cudaError_t e = ts::launch_select(scores, Hkv, N, (int)((N + chunk - 1) / chunk), k_sel, sink_chunks,
                                      recent_chunks, sel, part_len, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "select launch");
    ts::note_launches(1);
    return TS_OK;
}

ts_status ts_gather_tree_attn(const void *q, const void *k, const void *v, int64_t ld_kv, int64_t N,
                              const int32_t *sel, int k_sel, void *k_part, void *v_part, int64_t ld_part, int T,
                              int Hq, int Hkv, int d, float scale, const uint64_t *mask, void *out, float *lse,
                              void *workspace, size_t ws_bytes, ts_stream_t stream) {
    if (T == 0) return check_attn_shape(T, Hq, Hkv, d, N);
    if (N < 1) return fail(TS_ERR_INVALID_ARG, "N=%lld: nothing to gather", (long long)N);
    const int64_t nc = (N + 63) / 64;
    if (k_sel < 1 || k_sel > nc) return fail(TS_ERR_INVALID_ARG, "k_sel=%d outside [1, ceil(N/64)=%lld]", k_sel,
                                             (long long)nc);
    if (!sel || !aligned4(sel)) return fail(TS_ERR_INVALID_ARG, "null or misaligned sel");
    if (!k || !v || !aligned16(k) || !aligned16(v)) return fail(TS_ERR_INVALID_ARG, "null or misaligned k/v");
    if (!k_part || !v_part) return fail(TS_ERR_INVALID_ARG, "null k_part/v_part");
    if (ld_kv < N) return fail(TS_ERR_INVALID_ARG, "ld_kv < N");
    const int64_t B = (int64_t)k_sel * 64;
    ts::SmallGather gs;
    gs.sel = sel;
    gs.k_sel = k_sel;
    gs.n_chunks = (int)nc;
    gs.k = static_cast<const __nv_bfloat16 *>(k);
    gs.v = static_cast<const __nv_bfloat16 *>(v);
    gs.ld = ld_kv;
    gs.N = N;
    gs.k_dst = static_cast<__nv_bfloat16 *>(k_part);
    gs.v_dst = static_cast<__nv_bfloat16 *>(v_part);
    // the attention over the compact cache (rows [0, B) as they are gathered,
    // rows [B, B + T) the batch's own), every head's prefix complete but for
    // rows a short last chunk lacks
    return tree_attn_impl(q, k_part, v_part, ld_part, B, T, Hq, Hkv, d, scale, mask, nullptr, out, lse, nullptr, 0,
                          workspace, ws_bytes, stream, &gs);
}

ts_status ts_select_gather_tree_attn(const float *scores, int64_t N, int budget_tokens, int chunk, int sink_chunks,
                                     int recent_chunks, int32_t *sel, int32_t *part_len, const void *q, const void *k,
                                     const void *v, int64_t ld_kv, void *k_part, void *v_part, int64_t ld_part, int T,
                                     int Hq, int Hkv, int d, float scale, const uint64_t *mask, void *out, float *lse,
                                     void *workspace, size_t ws_bytes, ts_stream_t stream) {
    int k_sel = 0;
    ts_status st = check_select(scores, Hkv, N, budget_tokens, chunk, sink_chunks, recent_chunks, sel, part_len,
                                &k_sel);
    if (st != TS_OK) return st;
    if (k_sel == 0) return fail(TS_ERR_INVALID_ARG, "N=%lld: nothing to select", (long long)N);
    if (T == 0) return check_attn_shape(T, Hq, Hkv, d, N);
    if (!k || !v || !aligned16(k) || !aligned16(v)) return fail(TS_ERR_INVALID_ARG, "null or misaligned k/v");
    if (!k_part || !v_part) return fail(TS_ERR_INVALID_ARG, "null k_part/v_part");
    if (ld_kv < N) return fail(TS_ERR_INVALID_ARG, "ld_kv < N");
    const int64_t nc = (N + 63) / 64;
    ts::SmallGather gs;
    gs.k_sel = k_sel;
    gs.n_chunks = (int)nc;
    gs.k = static_cast<const __nv_bfloat16 *>(k);
    gs.v = static_cast<const __nv_bfloat16 *>(v);
    gs.ld = ld_kv;
    gs.N = N;
    gs.k_dst = static_cast<__nv_bfloat16 *>(k_part);
    gs.v_dst = static_cast<__nv_bfloat16 *>(v_part);
    gs.scores = scores;
    gs.n_sink = sink_chunks;
    gs.n_recent = recent_chunks;
    gs.sel_out = sel;
    gs.part_len_out = part_len;
    return tree_attn_impl(q, k_part, v_part, ld_part, (int64_t)k_sel * 64, T, Hq, Hkv, d, scale, mask, nullptr, out,
                          lse, nullptr, 0, workspace, ws_bytes, stream, &gs);
}

static ts_status vocab_stage(const float *logits, int T, int V, const int32_t *history, int W, float theta,
                             float min_p, float temperature, unsigned flags, uint64_t seed, uint64_t offset,
                             const int32_t *draft, const int32_t *parent, int32_t anchor, int32_t *target,
                             int32_t *kept, int32_t *result, int32_t *path, ts_stream_t stream) {
    if (T < 1 || T > 1024) return fail(TS_ERR_UNSUPPORTED, "T=%d outside [1, 1024]", T);
    if (flags & ~(unsigned)(TS_VOCAB_SAMPLE | TS_VOCAB_PATH_WINDOW))
        return fail(TS_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    if (V < 1 || V > 163840) return fail(TS_ERR_UNSUPPORTED, "V=%d outside [1, 163840]", V);
    if (W < 0) return fail(TS_ERR_INVALID_ARG, "W=%d < 0", W);
    if (!(theta > 0.f) || !isfinite(theta)) return fail(TS_ERR_INVALID_ARG, "theta must be finite and > 0");
    if (!(temperature > 0.f) || !isfinite(temperature))
        return fail(TS_ERR_INVALID_ARG, "temperature must be finite and > 0");
    if (!(min_p >= 0.f && min_p <= 1.f)) return fail(TS_ERR_INVALID_ARG, "min_p outside [0, 1]");
    if (!logits || !draft || !parent || !target || !kept || !result || !path || (W > 0 && !history))
        return fail(TS_ERR_INVALID_ARG, "null pointer");
    if (!aligned4(logits) || !aligned4(draft) || !aligned4(parent) || !aligned4(target) || !aligned4(kept) ||
        !aligned4(result) || !aligned4(path) || (history && !aligned4(history)))
        return fail(TS_ERR_INVALID_ARG, "misaligned pointer");
    ts::VocabArgs a{};
    a.logits = logits;
    a.T = T;
    a.V = V;
    a.history = history;
    a.W = W;
    a.theta = theta;
    a.temperature = temperature;
    // ln(min_p) in double on the host; the kernel compares against m + ln(min_p)
    a.log_min_p = min_p > 0.f ? log((double)min_p) : -INFINITY;
    a.draft = draft;
    a.parent = parent;
    a.anchor = anchor;
    a.target = target;
    a.kept = kept;
    a.result = result;
    a.path = path;
    a.sample = (flags & TS_VOCAB_SAMPLE) ? 1 : 0;
    a.path_window = (flags & TS_VOCAB_PATH_WINDOW) ? 1 : 0;
    a.seed = seed;
    a.offset = offset;
    cudaError_t e = ts::launch_vocab(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "vocab launch");
    ts::note_launches(2);
    return TS_OK;
}

}  // extern "C"

ts_status ts_penalty_minp_verify(const float *logits, int T, int V, const int32_t *history, int W,
                                 float theta, float min_p, float temperature,
                                 const int32_t *draft, const int32_t *parent, int32_t anchor,
                                 int32_t *target, int32_t *kept, int32_t *result, int32_t *path,
                                 void *workspace, size_t ws_bytes, ts_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    return vocab_stage(logits, T, V, history, W, theta, min_p, temperature, 0u, 0, 0, draft, parent, anchor, target,
                       kept, result, path, stream);
}

ts_status ts_vocab_verify(const float *logits, int T, int V, const int32_t *history, int W, float theta, float min_p,
                          float temperature, unsigned flags, uint64_t seed, uint64_t offset, const int32_t *draft,
                          const int32_t *parent, int32_t anchor, int32_t *target, int32_t *kept, int32_t *result,
                          int32_t *path, ts_stream_t stream) {
    return vocab_stage(logits, T, V, history, W, theta, min_p, temperature, flags, seed, offset, draft, parent, anchor,
                       target, kept, result, path, stream);
}

ts_status ts_penalty_minp_sample_verify(const float *logits, int T, int V, const int32_t *history, int W,
                                        float theta, float min_p, float temperature, uint64_t seed,
                                        uint64_t offset, const int32_t *draft, const int32_t *parent,
                                        int32_t anchor, int32_t *target, int32_t *kept, int32_t *result,
                                        int32_t *path, ts_stream_t stream) {
    return vocab_stage(logits, T, V, history, W, theta, min_p, temperature, TS_VOCAB_SAMPLE, seed, offset, draft,
                       parent, anchor, target, kept, result, path, stream);
}

static ts_status check_ngram_table(const void *table, int64_t capacity) {
    if (capacity < 64 || capacity > ((int64_t)1 << 30) || (capacity & (capacity - 1)))
        return fail(TS_ERR_INVALID_ARG, "capacity=%lld must be a power of two in [64, 2^30]", (long long)capacity);
    if (!table) return fail(TS_ERR_INVALID_ARG, "null table");
    if (!aligned16(table)) return fail(TS_ERR_INVALID_ARG, "table must be 16-byte aligned");
    return TS_OK;
}

size_t ts_ngram_table_bytes(int64_t capacity) {
    if (capacity < 64 || capacity > ((int64_t)1 << 30) || (capacity & (capacity - 1))) return 0;
    return (size_t)capacity * 24;
}

ts_status ts_ngram_reset(void *table, int64_t capacity, ts_stream_t stream) {
    ts_status st = check_ngram_table(table, capacity);
    if (st != TS_OK) return st;
    cudaError_t e = ts::launch_ngram_reset(table, (uint32_t)capacity, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ngram_reset launch");
    ts::note_launches(1);
    return TS_OK;
}

ts_status ts_ngram_update(void *table, int64_t capacity, const int32_t *seq, int64_t n_old, int64_t n_new,
                          int32_t *status, ts_stream_t stream) {
    ts_status st = check_ngram_table(table, capacity);
    if (st != TS_OK) return st;
    if (n_old < 0 || n_new < n_old) return fail(TS_ERR_INVALID_ARG, "need 0 <= n_old <= n_new");
    if (n_new > INT32_MAX) return fail(TS_ERR_UNSUPPORTED, "n_new=%lld above 2^31 - 1", (long long)n_new);
    if (n_new <= 3 || n_new <= n_old) return TS_OK;  // no new window
    if (!seq || !status) return fail(TS_ERR_INVALID_ARG, "null seq/status");
    if (!aligned4(seq) || !aligned4(status)) return fail(TS_ERR_INVALID_ARG, "misaligned seq/status");
    cudaError_t e = ts::launch_ngram_update(table, (uint32_t)capacity, seq, n_old, n_new, status,
                                            reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ngram_update launch");
    ts::note_launches(1);
    return TS_OK;
}

ts_status ts_ngram_topk(const void *table, int64_t capacity, const int32_t *seq, int64_t n, const int32_t *anchor,
                        int k, int32_t *chains, int32_t *counts, int32_t *found, ts_stream_t stream) {
    ts_status st = check_ngram_table(table, capacity);
    if (st != TS_OK) return st;
    if (k < 1 || k > 1024) return fail(TS_ERR_UNSUPPORTED, "k=%d outside [1, 1024]", k);
    if (n < 0 || n > INT32_MAX) return fail(TS_ERR_INVALID_ARG, "n=%lld outside [0, 2^31 - 1]", (long long)n);
    if (!anchor || !chains || !counts || !found || (n > 0 && !seq))
        return fail(TS_ERR_INVALID_ARG, "null seq/anchor/chains/counts/found");
    if (!aligned4(anchor) || !aligned4(chains) || !aligned4(counts) || !aligned4(found) || (seq && !aligned4(seq)))
        return fail(TS_ERR_INVALID_ARG, "misaligned pointer");
    cudaError_t e = ts::launch_ngram_topk(table, (uint32_t)capacity, seq, n, anchor, k, chains, counts, found,
                                          reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ngram_topk launch");
    ts::note_launches(1);
    return TS_OK;
}

ts_status ts_commit_path(void *k, void *v, int64_t ld_kv, int64_t N, int T, int Hkv, int d, int32_t *result,
                         const int32_t *path, ts_stream_t stream) {
    if (T < 1 || T > ts::TS_MAX_T) return fail(TS_ERR_UNSUPPORTED, "T=%d outside [1, %d]", T, ts::TS_MAX_T);
    if (d != 64 && d != 128) return fail(TS_ERR_UNSUPPORTED, "head dim d=%d (supported: 64, 128)", d);
    if (Hkv <= 0) return fail(TS_ERR_INVALID_ARG, "Hkv=%d", Hkv);
    if (N < 0) return fail(TS_ERR_INVALID_ARG, "N=%lld < 0", (long long)N);
    if (!k || !v || !result || !path) return fail(TS_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(k) || !aligned16(v) || !aligned4(result) || !aligned4(path))
        return fail(TS_ERR_INVALID_ARG, "misaligned pointer");
    if (ld_kv < N + T) return fail(TS_ERR_INVALID_ARG, "ld_kv=%lld < N + T", (long long)ld_kv);
    cudaError_t e = ts::launch_commit_path(static_cast<__nv_bfloat16 *>(k), static_cast<__nv_bfloat16 *>(v), ld_kv, N,
                                           T, Hkv, d, result, path, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "commit_path launch");
    ts::note_launches(1);
    return TS_OK;
}
