// tc_stub.cu - placeholder until the tensor-core backward lands: reports it
// as unavailable so the backward takes the CUDA-core kernels.
#include "tc.h"

namespace sinkattn {

bool tc_bwd_supported(const Problem&, bool) { return false; }
size_t tc_bwd_workspace_bytes(const Problem&, bool) { return 0; }
cudaError_t tc_bwd(const Problem&, const void*, const void*, const void*, const float*,
                   const float*, const void*, void*, void*, void*, uint32_t*, void*,
                   cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace sinkattn
