// convert.cu - f16 copies of bf16 operands for the tensor-core kernels.
//
// The forward's P V product and the backward's S^T = K Q^T, dK += dS^T Q and
// dQ = dS K run with f16 operands (P and dS need f16's 11 bits when logits are
// large; one product's A and B share a format). Their bf16 inputs V, Q and K
// are copied to f16 once per call into the caller's workspace by this
// memory-bound kernel, instead of converting every shared-memory tile inside
// the products' kernels (where each tile is loaded by many CTAs). bf16 -> f16
// keeps the value exactly for magnitudes within f16's range (up to 65504;
// below 2^-17 the f16 subnormal spacing of 2^-24 rounds it).
#include <algorithm>

#include "kernels.h"
#include "tc_ptx.cuh"

namespace sinkattn {
namespace {

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    return tc::pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// n16: number of 16-byte groups (8 elements each)
__global__ void __launch_bounds__(256) bf16_to_f16_kernel(const uint4* __restrict__ src,
                                                          uint4* __restrict__ dst, size_t n16) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16; i += stride) {
        const uint4 x = __ldg(src + i);
        dst[i] = make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z),
                            bf16x2_to_f16x2(x.w));
    }
}

}  // namespace

cudaError_t convert_bf16_to_f16(const void* src, void* dst, size_t elems, cudaStream_t st) {
    const size_t n16 = elems / 8;  // callers pass whole rows of 64 or 128 elements
    if (n16 == 0) return cudaSuccess;
    const int blocks = (int)std::min<size_t>((n16 + 255) / 256, (size_t)152 * 16);
    bf16_to_f16_kernel<<<blocks, 256, 0, st>>>(static_cast<const uint4*>(src),
                                                static_cast<uint4*>(dst), n16);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace sinkattn
