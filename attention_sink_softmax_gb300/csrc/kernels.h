// kernels.h - internal launchers of libsinkattn (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace sinkattn {

// Counts every kernel launch the library enqueues (sink_attn_kernel_launches).
void count_launches(unsigned n);

// Launch `kernel` so that it may start while the previous kernel in `st` (one
// this library launched in the same call) is finishing; the kernel calls
// pdl_wait() before it reads that kernel's outputs (common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_after(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// f16 copy of `elems` bf16 values (a multiple of 8; 16-byte aligned buffers),
// exact within f16's range (convert.cu).
// clear_flags (nullable): a device flag word zeroed by the kernel before the
// next kernel (launched with launch_after) may start.
cudaError_t convert_bf16_to_f16(const void* src, void* dst, size_t elems, cudaStream_t st,
                                uint32_t* clear_flags = nullptr);
// f16 copies of q (q_elems) and k (k_elems) and acc_floats zeros, in one pass
// (the 64-wide tensor-core backward's preparation; convert.cu).
cudaError_t bwd_prepare(const void* q, void* q16, size_t q_elems, const void* k, void* k16,
                        size_t k_elems, float* acc, size_t acc_floats, cudaStream_t st);

// CUDA-core path (any dtype the ABI accepts, head_dim 64).
// o_lo (nullable, bf16 only): receives bf16(O - bf16(O)) per element.
cudaError_t simt_fwd(const Problem& P, bool bf16, const void* q, const void* k, const void* v,
                     const float* sinks, void* o, void* o_lo, float* lse, uint32_t* flags,
                     cudaStream_t st);
cudaError_t simt_bwd_main(const Problem& P, bool bf16, const void* q, const void* k, const void* v,
                          const float* lse, const float* delta, const void* dout, void* dq,
                          void* dk, void* dv, uint32_t* flags, cudaStream_t st);

// Backward step 1 (memory-bound): delta [h_q, T] and dsinks [h_q] via
// per-chunk partials [h_q, preprocess_chunks(T)] reduced in a fixed order.
int preprocess_chunks(int total);
// o_lo (nullable, bf16 only): the low-order part of O written by the forward;
// when given, delta = dout . (o + o_lo).
// clear_flags (nullable): a device flag word zeroed before the call returns
// control to the stream's next kernel (the backward's own flags).
cudaError_t bwd_preprocess(const Problem& P, bool bf16, const float* sinks, const void* o,
                           const void* o_lo, const float* lse, const void* dout, float* delta,
                           float* dsinks, float* partial, uint32_t* clear_flags, cudaStream_t st);

// Decode (decode.cu): split kernel (+ merge kernel on the CUDA-core path).
// `part` holds decode_partial_floats(batch, h_q) floats; `counters` holds
// batch x h_kv int32 that are zero on entry and zero again on exit.
int decode_splits(int batch, int h_kv, int max_len);
size_t decode_partial_floats(int batch, int h_q);
cudaError_t decode(const DecodeArgs& a, bool bf16, const void* q, const void* k, const void* v,
                   const float* sinks, const int32_t* kv_start, const int32_t* kv_len, void* o,
                   float* lse, float* part, int32_t* counters, uint32_t* flags, cudaStream_t st);

}  // namespace sinkattn
