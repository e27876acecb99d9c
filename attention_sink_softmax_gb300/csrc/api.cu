// api.cu - the C ABI of libsinkattn (declared in include/sink_attn.h):
// argument validation, workspace layout and kernel dispatch.
//
// Workspace layout (each region 256-byte aligned):
//   [0, 256)            device flag word (uint32) + reserved
//   backward only:
//   delta               fp32 [h_q, T]        dO . O per row
//   partial             fp32 [h_q, chunks]   per-chunk partial sums for dS_h
//   tc                  tensor-core path scratch (tc_bwd_workspace_bytes)
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "../../include/sink_attn.h"
#include "../../include/sink_attn_testing.h"
#include "kernels.h"
#include "tc.h"
#include "validate.h"

using namespace sinkattn;

static_assert(kFlagTimeout == SINK_FLAG_TIMEOUT && kFlagSeqTooLong == SINK_FLAG_SEQ_TOO_LONG &&
                  kFlagBadSeqlens == SINK_FLAG_BAD_SEQLENS,
              "device flag bits as published in sink_attn.h");

static std::atomic<uint64_t> g_launches{0};
// limit of every bounded device wait, and the test hook that withholds loads
static std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
static std::atomic<int> g_withhold_load{0};
static std::atomic<int> g_deterministic{0};

namespace sinkattn {
void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace sinkattn

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kHeaderBytes = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Device (or managed) memory that kernels may dereference. A host pointer
// handed to a kernel would fault the device, so it is refused up front.
bool device_accessible(const void* x) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, x) != cudaSuccess) {
        cudaGetLastError();  // clear the non-sticky error
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}


}  // namespace

namespace sinkattn {
sink_status_t validate_params(const sink_attn_params_t* p) {
    if (!p) return SINK_ERR_INVALID_ARG;
    if (p->batch < 0 || p->max_seqlen < 0 || p->total_tokens < 0) return SINK_ERR_INVALID_ARG;
    if (p->h_q <= 0 || p->h_kv <= 0 || p->h_q % p->h_kv != 0) return SINK_ERR_INVALID_ARG;
    if (p->head_dim <= 0) return SINK_ERR_INVALID_ARG;
    if (p->dtype != SINK_BF16 && p->dtype != SINK_FP32) return SINK_ERR_INVALID_ARG;
    if (p->causal != 0 && p->causal != 1) return SINK_ERR_INVALID_ARG;
    if (p->window > 0 && !p->causal) return SINK_ERR_INVALID_ARG;
    if (!(p->softmax_scale == p->softmax_scale)) return SINK_ERR_INVALID_ARG;  // NaN
    // sizes must keep every element index and every grid dimension in range
    if ((int64_t)p->total_tokens * p->h_q * p->head_dim > ((int64_t)1 << 40)) return SINK_ERR_INVALID_ARG;
    if (p->batch > 65535 || p->h_q > 65535) return SINK_ERR_UNSUPPORTED;
    if (p->head_dim != 64 && p->head_dim != 128) return SINK_ERR_UNSUPPORTED;
    return SINK_OK;
}

}  // namespace sinkattn

namespace {

sink_status_t validate(const sink_attn_params_t* p) { return validate_params(p); }

// Padded layout: total_tokens must equal batch * max_seqlen.
sink_status_t validate_layout(const sink_attn_params_t* p, const int32_t* cu) {
    if (!cu && (int64_t)p->batch * p->max_seqlen != p->total_tokens) return SINK_ERR_INVALID_ARG;
    if (cu && (((uintptr_t)cu & 3u) || !device_accessible(cu))) return SINK_ERR_INVALID_ARG;
    return SINK_OK;
}

Problem make_problem(const sink_attn_params_t* p, const int32_t* cu) {
    Problem P;
    P.nseq = p->batch;
    P.max_seqlen = p->max_seqlen;
    P.total = p->total_tokens;
    P.h_q = p->h_q;
    P.h_kv = p->h_kv;
    P.group = p->h_q / p->h_kv;
    P.head_dim = p->head_dim;
    P.causal = p->causal;
    P.window = p->causal ? (p->window > 0 ? p->window : 0) : 0;
    P.scale = p->softmax_scale > 0.f ? p->softmax_scale : 1.0f / sqrtf((float)p->head_dim);
    P.scale_log2 = P.scale * kLog2e;
    P.cu = cu;
    P.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    P.withhold_load = g_withhold_load.load(std::memory_order_relaxed);
    P.deterministic = g_deterministic.load(std::memory_order_relaxed);
    return P;
}

bool empty(const sink_attn_params_t* p) {
    return p->batch == 0 || p->max_seqlen == 0 || p->total_tokens == 0;
}

struct BwdLayout {
    size_t delta, partial, tc, total;
};

BwdLayout bwd_layout(const sink_attn_params_t* p) {
    BwdLayout L;
    const size_t T = (size_t)p->total_tokens;
    L.delta = kHeaderBytes;
    L.partial = L.delta + align_up(sizeof(float) * (size_t)p->h_q * T);
    L.tc = L.partial + align_up(sizeof(float) * (size_t)p->h_q * preprocess_chunks(p->total_tokens));
    L.total = L.tc + align_up(tc_bwd_workspace_bytes(make_problem(p, nullptr), p->dtype == SINK_BF16));
    return L;
}

size_t fwd_bytes(const sink_attn_params_t* p) {
    return kHeaderBytes + align_up(tc_fwd_workspace_bytes(make_problem(p, nullptr), p->dtype == SINK_BF16));
}

sink_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? SINK_OK : SINK_ERR_CUDA; }

bool all_aligned(std::initializer_list<const void*> ptrs) {
    for (const void* x : ptrs)
        if (!x || !aligned16(x) || !device_accessible(x)) return false;
    return true;
}

}  // namespace

extern "C" {

size_t sink_attn_workspace_bytes(const sink_attn_params_t* params, int is_bwd) {
    if (validate(params) != SINK_OK) return 0;
    return is_bwd ? bwd_layout(params).total : fwd_bytes(params);
}

// o_lo: NULL, or bf16 [T, h_q, d] (bf16 params only)
static sink_status_t check_o_lo(const sink_attn_params_t* p, const void* o_lo) {
    if (!o_lo) return SINK_OK;
    if (p->dtype != SINK_BF16) return SINK_ERR_INVALID_ARG;
    if (!empty(p) && !all_aligned({o_lo})) return SINK_ERR_INVALID_ARG;
    return SINK_OK;
}

sink_status_t sink_attn_fwd_ex(const sink_attn_params_t* params, const void* q, const void* k,
                               const void* v, const float* sinks, const int32_t* cu_seqlens,
                               void* o, void* o_lo, float* lse, void* workspace,
                               size_t workspace_bytes, sink_stream_t stream) {
    sink_status_t st = validate(params);
    if (st != SINK_OK) return st;
    if ((st = validate_layout(params, cu_seqlens)) != SINK_OK) return st;
    if (!workspace || !aligned16(workspace) || !device_accessible(workspace)) return SINK_ERR_WORKSPACE;
    if (workspace_bytes < fwd_bytes(params)) return SINK_ERR_WORKSPACE;
    if (!empty(params) && !all_aligned({q, k, v, sinks, o, lse})) return SINK_ERR_INVALID_ARG;
    if ((st = check_o_lo(params, o_lo)) != SINK_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t* flags = (uint32_t*)workspace;
    const Problem P = make_problem(params, cu_seqlens);
    const bool bf16 = params->dtype == SINK_BF16;
    // the tensor-core path's first kernel (V's f16 copy) zeroes the flag word
    if (!empty(params) && tc_fwd_supported(P, bf16))
        return cuda_status(tc_fwd(P, q, k, v, sinks, o, o_lo, lse, flags,
                                  (char*)workspace + kHeaderBytes, s));
    cudaError_t e = cudaMemsetAsync(flags, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess || empty(params)) return cuda_status(e);
    return cuda_status(simt_fwd(P, bf16, q, k, v, sinks, o, o_lo, lse, flags, s));
}

sink_status_t sink_attn_fwd(const sink_attn_params_t* params, const void* q, const void* k,
                            const void* v, const float* sinks, const int32_t* cu_seqlens, void* o,
                            float* lse, void* workspace, size_t workspace_bytes,
                            sink_stream_t stream) {
    return sink_attn_fwd_ex(params, q, k, v, sinks, cu_seqlens, o, nullptr, lse, workspace,
                            workspace_bytes, stream);
}

sink_status_t sink_attn_bwd_preprocess_ex(const sink_attn_params_t* params, const float* sinks,
                                          const void* o, const void* o_lo, const float* lse,
                                          const void* dout, float* delta, float* dsinks,
                                          void* workspace, size_t workspace_bytes,
                                          sink_stream_t stream) {
    sink_status_t st = validate(params);
    if (st != SINK_OK) return st;
    if (!workspace || !aligned16(workspace) || !device_accessible(workspace)) return SINK_ERR_WORKSPACE;
    const BwdLayout L = bwd_layout(params);
    if (workspace_bytes < L.total) return SINK_ERR_WORKSPACE;
    if (!all_aligned({sinks, dsinks})) return SINK_ERR_INVALID_ARG;
    if (params->total_tokens > 0 && !all_aligned({o, lse, dout, delta})) return SINK_ERR_INVALID_ARG;
    if (o_lo && (params->dtype != SINK_BF16 ||
                 (params->total_tokens > 0 && !all_aligned({o_lo}))))
        return SINK_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const Problem P = make_problem(params, nullptr);
    // the workspace's flag word is cleared by the call's last kernel
    cudaError_t e = bwd_preprocess(P, params->dtype == SINK_BF16, sinks, o, o_lo, lse, dout, delta,
                                   dsinks, (float*)((char*)workspace + L.partial),
                                   (uint32_t*)workspace, s);
    return cuda_status(e);
}

sink_status_t sink_attn_bwd_preprocess(const sink_attn_params_t* params, const float* sinks,
                                       const void* o, const float* lse, const void* dout,
                                       float* delta, float* dsinks, void* workspace,
                                       size_t workspace_bytes, sink_stream_t stream) {
    return sink_attn_bwd_preprocess_ex(params, sinks, o, nullptr, lse, dout, delta, dsinks,
                                       workspace, workspace_bytes, stream);
}

sink_status_t sink_attn_bwd_prepare(const sink_attn_params_t* params, const void* q,
                                    const void* k, void* workspace, size_t workspace_bytes,
                                    sink_stream_t stream) {
    sink_status_t st = validate(params);
    if (st != SINK_OK) return st;
    // the pass covers all total_tokens rows and needs no sequence layout
    if (!workspace || !aligned16(workspace) || !device_accessible(workspace)) return SINK_ERR_WORKSPACE;
    const BwdLayout L = bwd_layout(params);
    if (workspace_bytes < L.total) return SINK_ERR_WORKSPACE;
    if (!empty(params) && !all_aligned({q, k})) return SINK_ERR_INVALID_ARG;
    if (empty(params)) return SINK_OK;
    const Problem P = make_problem(params, nullptr);
    const bool bf16 = params->dtype == SINK_BF16;
    if (!tc_bwd_supported(P, bf16)) return SINK_OK;  // only the 64-wide tensor-core path prepares
    return cuda_status(tc_bwd_prepare(P, q, k, (char*)workspace + L.tc, (cudaStream_t)stream));
}

sink_status_t sink_attn_bwd_main(const sink_attn_params_t* params, const void* q, const void* k,
                                 const void* v, const int32_t* cu_seqlens, const float* lse,
                                 const float* delta, const void* dout, void* dq, void* dk,
                                 void* dv, void* workspace, size_t workspace_bytes,
                                 sink_stream_t stream) {
    return sink_attn_bwd_main_ex(params, q, k, v, cu_seqlens, lse, delta, dout, dq, dk, dv,
                                 workspace, workspace_bytes, 0u, stream);
}

sink_status_t sink_attn_bwd_main_ex(const sink_attn_params_t* params, const void* q,
                                    const void* k, const void* v, const int32_t* cu_seqlens,
                                    const float* lse, const float* delta, const void* dout,
                                    void* dq, void* dk, void* dv, void* workspace,
                                    size_t workspace_bytes, unsigned options, sink_stream_t stream) {
    if (options & ~SINK_BWD_PREPARED) return SINK_ERR_INVALID_ARG;
    sink_status_t st = validate(params);
    if (st != SINK_OK) return st;
    if ((st = validate_layout(params, cu_seqlens)) != SINK_OK) return st;
    if (!workspace || !aligned16(workspace) || !device_accessible(workspace)) return SINK_ERR_WORKSPACE;
    const BwdLayout L = bwd_layout(params);
    if (workspace_bytes < L.total) return SINK_ERR_WORKSPACE;
    if (!empty(params) && !all_aligned({q, k, v, lse, delta, dout, dq, dk, dv}))
        return SINK_ERR_INVALID_ARG;
    if (empty(params)) return SINK_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const Problem P = make_problem(params, cu_seqlens);
    const bool bf16 = params->dtype == SINK_BF16;
    cudaError_t e;
    if (tc_bwd_supported(P, bf16))
        e = tc_bwd(P, q, k, v, lse, delta, dout, dq, dk, dv, (uint32_t*)workspace,
                   (char*)workspace + L.tc, (options & SINK_BWD_PREPARED) != 0, s);
    else if (tc_bwd128_supported(P, bf16))
        e = tc_bwd128(P, q, k, v, lse, delta, dout, dq, dk, dv, (uint32_t*)workspace, s);
    else
        e = simt_bwd_main(P, bf16, q, k, v, lse, delta, dout, dq, dk, dv, (uint32_t*)workspace, s);
    return cuda_status(e);
}

sink_status_t sink_attn_bwd_ex(const sink_attn_params_t* params, const void* q, const void* k,
                               const void* v, const float* sinks, const int32_t* cu_seqlens,
                               const void* o, const void* o_lo, const float* lse, const void* dout,
                               void* dq, void* dk, void* dv, float* dsinks, void* workspace,
                               size_t workspace_bytes, sink_stream_t stream) {
    sink_status_t st = validate(params);
    if (st != SINK_OK) return st;
    if ((st = validate_layout(params, cu_seqlens)) != SINK_OK) return st;
    if (!workspace || !aligned16(workspace) || !device_accessible(workspace)) return SINK_ERR_WORKSPACE;
    const BwdLayout L = bwd_layout(params);
    if (workspace_bytes < L.total) return SINK_ERR_WORKSPACE;
    if (!all_aligned({sinks, dsinks})) return SINK_ERR_INVALID_ARG;
    if (!empty(params) && !all_aligned({q, k, v, o, lse, dout, dq, dk, dv}))
        return SINK_ERR_INVALID_ARG;
    if ((st = check_o_lo(params, o_lo)) != SINK_OK) return st;
    float* delta = (float*)((char*)workspace + L.delta);
    st = sink_attn_bwd_preprocess_ex(params, sinks, o, o_lo, lse, dout, delta, dsinks, workspace,
                                     workspace_bytes, stream);
    if (st != SINK_OK) return st;
    return sink_attn_bwd_main(params, q, k, v, cu_seqlens, lse, delta, dout, dq, dk, dv, workspace,
                              workspace_bytes, stream);
}

sink_status_t sink_attn_bwd(const sink_attn_params_t* params, const void* q, const void* k,
                            const void* v, const float* sinks, const int32_t* cu_seqlens,
                            const void* o, const float* lse, const void* dout, void* dq, void* dk,
                            void* dv, float* dsinks, void* workspace, size_t workspace_bytes,
                            sink_stream_t stream) {
    return sink_attn_bwd_ex(params, q, k, v, sinks, cu_seqlens, o, nullptr, lse, dout, dq, dk, dv,
                            dsinks, workspace, workspace_bytes, stream);
}

sink_status_t sink_attn_fetch_device_error(void* workspace, size_t workspace_bytes,
                                           sink_stream_t stream, uint32_t* flags_out) {
    if (!workspace || workspace_bytes < sizeof(uint32_t)) return SINK_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t flags = 0;
    if (cudaMemcpyAsync(&flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SINK_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SINK_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return SINK_ERR_CUDA;
    if (flags_out) *flags_out = flags;
    if (flags & kFlagTimeout) return SINK_ERR_TIMEOUT;
    if (flags) return SINK_ERR_DEVICE;
    return SINK_OK;
}

namespace {
// Decode: [header][partials], the split count fixed by the params so that the
// workspace size needs no device query.
DecodeArgs decode_args(const sink_attn_params_t* p) {
    DecodeArgs a;
    a.batch = p->batch;
    a.h_q = p->h_q;
    a.h_kv = p->h_kv;
    a.group = p->h_q / p->h_kv;
    a.total = p->total_tokens;
    a.max_len = p->max_seqlen;
    a.window = p->window > 0 ? p->window : 0;
    a.nsplit = decode_splits(p->batch, p->h_kv, p->max_seqlen);
    const float scale = p->softmax_scale > 0.f ? p->softmax_scale : 1.0f / sqrtf((float)p->head_dim);
    a.scale_log2 = scale * kLog2e;
    a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    return a;
}

// [header][per (query, key/value head) chunk counters][partials]; the header
// and the counters are zeroed together by one memset per call.
size_t decode_counter_bytes(const sink_attn_params_t* p) {
    return align_up(sizeof(int32_t) * (size_t)p->batch * p->h_kv);
}
size_t decode_bytes(const sink_attn_params_t* p) {
    return kHeaderBytes + decode_counter_bytes(p) +
           align_up(sizeof(float) * decode_partial_floats(p->batch, p->h_q));
}

sink_status_t validate_decode(const sink_attn_params_t* p) {
    sink_status_t st = validate(p);
    if (st != SINK_OK) return st;
    if (!p->causal) return SINK_ERR_INVALID_ARG;  // the query is the last token of its context
    if (p->h_q / p->h_kv > 64) return SINK_ERR_UNSUPPORTED;  // query heads per key/value head
    if (p->head_dim != 64) return SINK_ERR_UNSUPPORTED;      // the decode kernels are 64-wide
    return SINK_OK;
}
}  // namespace

size_t sink_attn_decode_workspace_bytes(const sink_attn_params_t* params) {
    if (validate_decode(params) != SINK_OK) return 0;
    return decode_bytes(params);
}

sink_status_t sink_attn_decode(const sink_attn_params_t* params, const void* q, const void* k_cache,
                               const void* v_cache, const float* sinks, const int32_t* kv_start,
                               const int32_t* kv_len, void* o, float* lse, void* workspace,
                               size_t workspace_bytes, sink_stream_t stream) {
    sink_status_t st = validate_decode(params);
    if (st != SINK_OK) return st;
    if (!workspace || !aligned16(workspace) || !device_accessible(workspace)) return SINK_ERR_WORKSPACE;
    if (workspace_bytes < decode_bytes(params)) return SINK_ERR_WORKSPACE;
    if (params->batch == 0) return SINK_OK;
    if (!all_aligned({q, o, (const void*)sinks, (const void*)lse})) return SINK_ERR_INVALID_ARG;
    if (params->total_tokens > 0 && !all_aligned({k_cache, v_cache})) return SINK_ERR_INVALID_ARG;
    for (const int32_t* x : {kv_start, kv_len})
        if (!x || ((uintptr_t)x & 3u) || !device_accessible(x)) return SINK_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t* flags = (uint32_t*)workspace;
    const size_t counters = decode_counter_bytes(params);
    cudaError_t e = cudaMemsetAsync(flags, 0, kHeaderBytes + counters, s);
    if (e != cudaSuccess) return SINK_ERR_CUDA;
    e = decode(decode_args(params), params->dtype == SINK_BF16, q, k_cache, v_cache, sinks, kv_start,
               kv_len, o, lse, (float*)((char*)workspace + kHeaderBytes + counters),
               (int32_t*)((char*)workspace + kHeaderBytes), flags, s);
    return cuda_status(e);
}

const char* sink_attn_status_str(sink_status_t status) {
    switch (status) {
        case SINK_OK: return "ok";
        case SINK_ERR_INVALID_ARG: return "invalid argument";
        case SINK_ERR_UNSUPPORTED: return "unsupported configuration";
        case SINK_ERR_CUDA: return "CUDA error";
        case SINK_ERR_WORKSPACE: return "workspace missing or too small";
        case SINK_ERR_TIMEOUT: return "a bounded device wait gave up";
        case SINK_ERR_DEVICE: return "device flagged an input condition";
        case SINK_ERR_SCRATCH_LIMIT: return "problem exceeds the fixed scratch of the no-allocation entry point";
    }
    return "unknown status";
}

uint64_t sink_attn_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

uint64_t sink_attn_set_wait_limit_ns(uint64_t limit_ns) {
    return g_wait_ns.exchange(limit_ns ? limit_ns : kDefaultWaitNs, std::memory_order_relaxed);
}

int sink_attn_set_deterministic(int on) {
    return g_deterministic.exchange(on ? 1 : 0, std::memory_order_relaxed);
}

void sink_attn_testing_withhold_load(int on) {
    g_withhold_load.store(on ? 1 : 0, std::memory_order_relaxed);
}

int sink_attn_version(void) { return 200; }

}  // extern "C"
