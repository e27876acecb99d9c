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

#include "kernels.h"
#include "tc_ptx.cuh"

namespace sinkattn {
namespace {

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    return tc::pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// n16: number of 16-byte groups (8 elements each). Each block converts
// kConvItems consecutive groups and exits (see bwd_prepare_kernel): with the
// backward's preparation running on a lower-priority stream at the same time,
// this kernel's pending blocks keep the SMs and the memory bandwidth.
constexpr int kConvPerThread = 8;
constexpr int kConvItems = 256 * kConvPerThread;

__global__ void __launch_bounds__(256) bf16_to_f16_kernel(const uint4* __restrict__ src,
                                                          uint4* __restrict__ dst, size_t n16,
                                                          uint32_t* clear_flags) {
    if (clear_flags && blockIdx.x == 0 && threadIdx.x == 0) {
        // the forward's device flag word: zeroed and made visible before the
        // forward (launched after this grid) may start and set a flag
        *clear_flags = 0u;
        __threadfence();
    }
    __syncthreads();
    pdl_trigger();  // the forward that reads dst may take the SMs this grid frees
    const size_t base = (size_t)blockIdx.x * kConvItems + threadIdx.x;
#pragma unroll
    for (int j = 0; j < kConvPerThread; ++j) {
        const size_t i = base + (size_t)j * 256;
        if (i >= n16) break;
        const uint4 x = __ldg(src + i);
        dst[i] = make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z),
                            bf16x2_to_f16x2(x.w));
    }
}

// The backward's preparation in one pass: f16 copies of Q and K, and the fp32
// dQ accumulator zeroed. Work items are 16-byte groups: [0, nq) of Q, then
// [nq, nq + nk) of K, then the accumulator's groups (4 floats each). Each
// block takes kPrepItems consecutive items and exits (no grid-stride loop):
// run on a low-priority stream beside the forward, short blocks hand their SM
// back to the forward's CTAs as soon as those are ready to run.
constexpr int kPrepPerThread = 8;
constexpr int kPrepItems = 256 * kPrepPerThread;

__global__ void __launch_bounds__(256) bwd_prepare_kernel(const uint4* __restrict__ q,
                                                          uint4* __restrict__ q16, size_t nq,
                                                          const uint4* __restrict__ k,
                                                          uint4* __restrict__ k16, size_t nk,
                                                          uint4* __restrict__ acc, size_t nacc) {
    const size_t total = nq + nk + nacc;
    const size_t base = (size_t)blockIdx.x * kPrepItems + threadIdx.x;
#pragma unroll
    for (int j = 0; j < kPrepPerThread; ++j) {
        const size_t i = base + (size_t)j * 256;
        if (i >= total) break;
        if (i < nq) {
            const uint4 x = __ldg(q + i);
            q16[i] = make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z),
                                bf16x2_to_f16x2(x.w));
        } else if (i < nq + nk) {
            const uint4 x = __ldg(k + (i - nq));
            k16[i - nq] = make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y),
                                     bf16x2_to_f16x2(x.z), bf16x2_to_f16x2(x.w));
        } else {
            acc[i - nq - nk] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

}  // namespace

cudaError_t bwd_prepare(const void* q, void* q16, size_t q_elems, const void* k, void* k16,
                        size_t k_elems, float* acc, size_t acc_floats, cudaStream_t st) {
    const size_t nq = q_elems / 8, nk = k_elems / 8, na = acc_floats / 4;
    const size_t total = nq + nk + na;
    if (total == 0) return cudaSuccess;
    const size_t blocks = (total + kPrepItems - 1) / kPrepItems;
    if (blocks > 0x7fffffffu) return cudaErrorInvalidValue;
    bwd_prepare_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint4*>(q), static_cast<uint4*>(q16), nq,
                                               static_cast<const uint4*>(k), static_cast<uint4*>(k16), nk,
                                               reinterpret_cast<uint4*>(acc), na);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t convert_bf16_to_f16(const void* src, void* dst, size_t elems, cudaStream_t st,
                                uint32_t* clear_flags) {
    const size_t n16 = elems / 8;  // callers pass whole rows of 64 or 128 elements
    if (n16 == 0) return cudaSuccess;
    const size_t blocks = (n16 + kConvItems - 1) / kConvItems;
    if (blocks > 0x7fffffffu) return cudaErrorInvalidValue;
    bf16_to_f16_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint4*>(src),
                                                          static_cast<uint4*>(dst), n16, clear_flags);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace sinkattn
