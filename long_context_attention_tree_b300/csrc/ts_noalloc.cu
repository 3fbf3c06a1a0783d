// Allocation-free variant of ts_tree_attn.
//
// Some callers cannot hand this library a device workspace: code that runs
// inside another runtime's execution callback (an inference-server plugin, a
// host function in someone else's stream), or a C caller with no allocator
// handle, where calling cudaMalloc is forbidden or would synchronize the
// device in the middle of a stream-ordered pipeline.  For them the split-KV
// partials live in one file-scope device array instead of caller memory.
//
// The array is TS_NOALLOC_SCRATCH_BYTES (64 MiB).  Every GPU that loads this
// library holds it until the process exits.  All calls share it, so calls
// whose kernels overlap on the GPU (different streams, or different host
// threads on one device) race on it; calls ordered on one stream are safe.
// Its contents persist from call to call; nothing in it needs to start at
// zero, because every partial the merge reads is written by the same call.
#include <stdio.h>

#include <mutex>

#include "../../include/ts.h"
#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[TS_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;

// Device address of g_noalloc_scratch for each device, looked up once with
// that device current.  In host code the array's name is only a host-side
// stand-in, so the address must come from cudaGetSymbolAddress.  The lookup
// may load the module on the device, which must not happen inside a stream
// capture: a first call whose stream is capturing is refused.
void *scratch_for_current_device(cudaStream_t stream, ts_status *st, const char **why) {
    static std::mutex mu;
    static void *addr[MAX_DEVICES] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *st = TS_ERR_CUDA;
        *why = "ts_tree_attn_noalloc: cudaGetDevice failed";
        return nullptr;
    }
    if (dev < 0 || dev >= MAX_DEVICES) {
        *st = TS_ERR_UNSUPPORTED;
        *why = "ts_tree_attn_noalloc: device index outside the 64 devices this entry point tracks";
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (addr[dev] == nullptr) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
            cudaGetLastError();
            *st = TS_ERR_UNSUPPORTED;
            *why = "ts_tree_attn_noalloc: the first call on a device sets up its scratch address and must come "
                   "before any stream capture";
            return nullptr;
        }
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) {
            *st = TS_ERR_CUDA;
            *why = cudaGetErrorString(e);
            return nullptr;
        }
        if (p == nullptr) {
            *st = TS_ERR_CUDA;
            *why = "ts_tree_attn_noalloc: the scratch array has no device address";
            return nullptr;
        }
        addr[dev] = p;
    }
    *st = TS_OK;
    return addr[dev];
}

}  // namespace

extern "C" ts_status ts_tree_attn_noalloc(const void *q, const void *k, const void *v, int64_t ld_kv,
                                          int64_t N, int T, int Hq, int Hkv, int d, float scale,
                                          const uint64_t *mask, void *out, float *lse,
                                          float *chunk_scores, int score_row, ts_stream_t stream) {
    const size_t need = ts_tree_attn_workspace_bytes(T, Hq, Hkv, d, N);
    if (need > (size_t)TS_NOALLOC_SCRATCH_BYTES) {
        char msg[160];
        snprintf(msg, sizeof msg, "ts_tree_attn_noalloc: these sizes need %zu bytes of scratch, above the %u-byte maximum",
                 need, (unsigned)TS_NOALLOC_SCRATCH_BYTES);
        return ts::report_error(TS_ERR_UNSUPPORTED, msg);
    }
    void *scratch = nullptr;
    if (need > 0) {
        ts_status st = TS_OK;
        const char *why = nullptr;
        scratch = scratch_for_current_device(reinterpret_cast<cudaStream_t>(stream), &st, &why);
        if (scratch == nullptr) return ts::report_error(st, why);
    }
    return ts_tree_attn(q, k, v, ld_kv, N, T, Hq, Hkv, d, scale, mask, out, lse, chunk_scores, score_row,
                        scratch, need > 0 ? (size_t)TS_NOALLOC_SCRATCH_BYTES : 0, stream);
}
