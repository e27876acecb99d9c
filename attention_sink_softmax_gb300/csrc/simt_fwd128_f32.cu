// simt_fwd128_f32.cu - the CUDA-core forward (simt_fwd.cuh) at head_dim 128 for
// f32 inputs (one instance per file: they are the slowest to compile).
#include "simt_fwd.cuh"

namespace sinkattn {

template cudaError_t launch_simt_fwd<float, 128>(const Problem&, const void*, const void*,
                                               const void*, const float*, void*, void*, float*,
                                               uint32_t*, cudaStream_t);

}  // namespace sinkattn
