// tc.h - tensor-core (tcgen05 / TMEM / TMA) path of libsinkattn for sm_103a.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cuda.h>

#include "common.cuh"

namespace sinkattn {

bool tc_fwd_supported(const Problem& P, bool bf16);
size_t tc_fwd_workspace_bytes(const Problem& P, bool bf16);
cudaError_t tc_fwd(const Problem& P, const void* q, const void* k, const void* v,
                   const float* sinks, void* o, void* o_lo, float* lse, uint32_t* flags,
                   void* workspace, cudaStream_t st);

bool tc_bwd_supported(const Problem& P, bool bf16);
size_t tc_bwd_workspace_bytes(const Problem& P, bool bf16);
// The backward's inputs-only pass (f16 copies of Q and K, the fp32 dQ
// accumulator zeroed) into its workspace; tc_bwd skips it when `prepared`.
cudaError_t tc_bwd_prepare(const Problem& P, const void* q, const void* k, void* workspace,
                           cudaStream_t st);
cudaError_t tc_bwd(const Problem& P, const void* q, const void* k, const void* v,
                   const float* lse, const float* delta, const void* dout, void* dq, void* dk,
                   void* dv, uint32_t* flags, void* workspace, bool prepared, cudaStream_t st);

// The row-owning dQ kernel of the split 64-wide backward (tc_bwd_dq.cu): K as
// its f16 copy, V in bf16, Q's f16 copy; writes dq once, in bf16.
cudaError_t tc_bwd_dq64(const Problem& P, const CUtensorMap& mk16, const CUtensorMap& mv,
                        const void* q16, const void* dout, const float* lse, const float* delta,
                        void* dq, uint32_t* flags, cudaStream_t st);

// 128-wide heads: a dQ kernel and a dK/dV kernel (tc_bwd128.cu); no workspace.
bool tc_bwd128_supported(const Problem& P, bool bf16);
cudaError_t tc_bwd128(const Problem& P, const void* q, const void* k, const void* v,
                      const float* lse, const float* delta, const void* dout, void* dq, void* dk,
                      void* dv, uint32_t* flags, cudaStream_t st);

}  // namespace sinkattn
