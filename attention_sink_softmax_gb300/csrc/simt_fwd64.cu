// simt_fwd64.cu - the CUDA-core forward (simt_fwd.cuh) at head_dim 64, and
// its dispatch over head_dim and dtype.
#include "simt_fwd.cuh"

namespace sinkattn {

cudaError_t simt_fwd(const Problem& P, bool bf16, const void* q, const void* k, const void* v,
                     const float* sinks, void* o, void* o_lo, float* lse, uint32_t* flags,
                     cudaStream_t st) {
    if (P.nseq == 0 || P.max_seqlen == 0) return cudaSuccess;
    if (P.head_dim == 128)
        return bf16 ? launch_simt_fwd<__nv_bfloat16, 128>(P, q, k, v, sinks, o, o_lo, lse, flags, st)
                    : launch_simt_fwd<float, 128>(P, q, k, v, sinks, o, nullptr, lse, flags, st);
    return bf16 ? launch_simt_fwd<__nv_bfloat16, 64>(P, q, k, v, sinks, o, o_lo, lse, flags, st)
                : launch_simt_fwd<float, 64>(P, q, k, v, sinks, o, nullptr, lse, flags, st);
}

}  // namespace sinkattn
