// noalloc.cu - sink_attn_bwd_preprocess_noalloc: backward step 1 without a
// caller-provided workspace.
//
// Some callers are handed their input and output buffers and nothing else: a
// plugin running inside a host framework that owns all device memory and
// exposes no scratch allocator, or code on a latency-critical path where a
// cudaMalloc would synchronise the device (or fail because a caching
// allocator has already reserved the memory). They cannot provide the
// workspace that sink_attn_bwd_preprocess needs for its per-chunk dS_h
// partial sums. This entry point keeps that scratch in a fixed file-scope
// device array instead, so it allocates nothing.
//
// Limits and sharing:
//   - the array holds kNoallocScratchFloats floats (1 MiB); a problem needing
//     more partials (h_q * ceil(T / 256)) is rejected with
//     SINK_ERR_SCRATCH_LIMIT before anything is enqueued;
//   - every GPU that loads this library holds the array until the process
//     exits;
//   - all calls on a device share the one array: calls whose work overlaps on
//     the GPU (for example on two streams without ordering) race and give
//     wrong results. Each call writes every partial it later reads, so no
//     clearing is needed between calls;
//   - the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it; make
//     that first call before any stream capture.
#include <mutex>

#include "../../include/sink_attn.h"
#include "kernels.h"
#include "validate.h"

namespace {

constexpr size_t kNoallocScratchFloats = (size_t)1 << 18;  // 1 MiB of fp32 partials
constexpr int kMaxDevices = 64;

__device__ __align__(256) float g_preprocess_scratch[kNoallocScratchFloats];

std::mutex g_setup_mutex;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_preprocess_scratch on the current device (host code
// cannot use the symbol itself as a device pointer).
cudaError_t scratch_for_current_device(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_preprocess_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool ok_ptr(const void* p) {
    if (!p || ((uintptr_t)p & 15u)) return false;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

}  // namespace

extern "C" {

size_t sink_attn_noalloc_scratch_bytes(void) { return kNoallocScratchFloats * sizeof(float); }

sink_status_t sink_attn_bwd_preprocess_noalloc(const sink_attn_params_t* p, const float* sinks,
                                               const void* o, const float* lse, const void* dout,
                                               float* delta, float* dsinks,
                                               sink_stream_t stream) {
    using namespace sinkattn;
    // the same field checks (and status codes) as sink_attn_bwd_preprocess
    const sink_status_t st = validate_params(p);
    if (st != SINK_OK) return st;
    const size_t need = (size_t)p->h_q * (size_t)preprocess_chunks(p->total_tokens);
    if (need > kNoallocScratchFloats) return SINK_ERR_SCRATCH_LIMIT;
    if (!ok_ptr(sinks) || !ok_ptr(dsinks)) return SINK_ERR_INVALID_ARG;
    if (p->total_tokens > 0 && (!ok_ptr(o) || !ok_ptr(lse) || !ok_ptr(dout) || !ok_ptr(delta)))
        return SINK_ERR_INVALID_ARG;
    float* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return SINK_ERR_CUDA;
    Problem P{};
    P.nseq = p->batch;
    P.max_seqlen = p->max_seqlen;
    P.total = p->total_tokens;
    P.h_q = p->h_q;
    P.h_kv = p->h_kv;
    P.group = p->h_q / p->h_kv;
    P.head_dim = p->head_dim;
    P.wait_ns = kDefaultWaitNs;
    cudaError_t e = bwd_preprocess(P, p->dtype == SINK_BF16, sinks, o, nullptr, lse, dout, delta,
                                   dsinks, scratch, nullptr, (cudaStream_t)stream);
    return e == cudaSuccess ? SINK_OK : SINK_ERR_CUDA;
}

}  // extern "C"
