// preprocess.cu - backward step 1 of sink attention (page
// "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、超稳定！", section "反向传播的实现",
// simplified equation): D_i = dO_i . O_i per row, and the sink gradient
// dS_h = -sum_i exp(S_h - LSE_i) D_i, reduced in a fixed order so that it is
// bitwise reproducible. Memory-bound; shared by every path (bf16 and fp32,
// head_dim 64 and 128).
#include "common.cuh"
#include "kernels.h"

namespace sinkattn {

// Backward step 1: delta = rowsum(dO * O) in [h_q, T] and per-chunk partials of
// sum_t exp(S_h - LSE_t) * delta_t. One block = one head x kPreTokens tokens
// (a chunk); kD / 8 lanes share one row, each lane one 16-byte (bf16) or
// 32-byte (fp32) piece of 8 elements. A thread issues the loads of 4 of its
// rows before using any, so every thread keeps 4 rows of O and dO in flight
// (memory-bound step). The head is the grid's x, so the blocks that run at
// the same time read every head of a few consecutive chunks: whole [token,
// head, d] rows of memory, not one head's 128-byte piece out of every
// h_q * 128 bytes. Chunks past the grid's y (more than 65535) loop.
constexpr int kPreTokens = 256;
constexpr int kPreThreads = 256;

// 8 consecutive elements of T as 16-byte words
template <typename T>
struct Piece8 {
    static constexpr int kWords = (int)sizeof(T) * 8 / 16;
    uint4 w[kWords];
};

template <typename T>
__device__ __forceinline__ Piece8<T> load_piece(const T* p) {
    Piece8<T> r;
    const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int i = 0; i < Piece8<T>::kWords; ++i) r.w[i] = __ldg(q + i);
    return r;
}

__device__ __forceinline__ float dot_piece(const Piece8<__nv_bfloat16>& a,
                                           const Piece8<__nv_bfloat16>& b) {
    const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a.w[0]);
    const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b.w[0]);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 u = __bfloat1622float2(x[i]), v = __bfloat1622float2(y[i]);
        s = fmaf(u.x, v.x, s);
        s = fmaf(u.y, v.y, s);
    }
    return s;
}

__device__ __forceinline__ float dot_piece(const Piece8<float>& a, const Piece8<float>& b) {
    const float* x = reinterpret_cast<const float*>(&a.w[0]);
    const float* y = reinterpret_cast<const float*>(&b.w[0]);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s = fmaf(x[i], y[i], s);
    return s;
}

// kLo: o_lo holds the low-order part of O (O - bf16(O), rounded to bf16), and
// delta is formed as dO . (o + o_lo), so D does not inherit the rounding of
// the stored O.
template <typename T, int kD, bool kLo>
__global__ void __launch_bounds__(kPreThreads, sizeof(T) == 2 ? 3 : 1)
preprocess_kernel(int total, int h_q, const T* __restrict__ o, const T* __restrict__ o_lo,
                  const T* __restrict__ dout, const float* __restrict__ lse,
                  const float* __restrict__ sinks, float* __restrict__ delta,
                  float* __restrict__ partial) {
    constexpr int kLanes = kD / 8;  // threads per row, 8 elements each
    constexpr int kPer = 8;
    constexpr int kRowsPerIter = kPreThreads / kLanes;
    constexpr int kIters = kPreTokens / kRowsPerIter;
    constexpr int kBatch = 4;  // rows of a thread in flight at once (3 blocks per SM for bf16)
    static_assert(kIters % kBatch == 0, "row batches");
    pdl_trigger();  // the fixed-order dS_h sum may be scheduled
    __shared__ float warp_sum[kPreThreads / 32];
    const int h = blockIdx.x;
    const int nchunks = (total + kPreTokens - 1) / kPreTokens;
    const int sub = threadIdx.x % kLanes;
    const int r0 = threadIdx.x / kLanes;
    const float sink = __ldg(sinks + h);
    for (int chunk = blockIdx.y; chunk < nchunks; chunk += gridDim.y) {
        const int t0 = chunk * kPreTokens;
        float mine = 0.f;  // this row-group's running sum, added in token order
        for (int b0 = 0; b0 < kIters; b0 += kBatch) {
            Piece8<T> po[kBatch], pd[kBatch], pl[kLo ? kBatch : 1];
            float lz[kBatch];
#pragma unroll
            for (int x = 0; x < kBatch; ++x) {
                const int t = t0 + r0 + (b0 + x) * kRowsPerIter;
                if (t < total) {
                    const size_t off = ((size_t)t * h_q + h) * kD + sub * kPer;
                    po[x] = load_piece(o + off);
                    pd[x] = load_piece(dout + off);
                    if (kLo) pl[kLo ? x : 0] = load_piece(o_lo + off);
                    lz[x] = __ldg(lse + (size_t)h * total + t);
                }
            }
#pragma unroll
            for (int x = 0; x < kBatch; ++x) {
                const int t = t0 + r0 + (b0 + x) * kRowsPerIter;
                float dsum = 0.f;
                if (t < total) {
                    // dO . o_lo first: the smaller term, added before the main one
                    dsum = kLo ? dot_piece(pl[kLo ? x : 0], pd[x]) : 0.f;
                    dsum += dot_piece(po[x], pd[x]);
                }
#pragma unroll
                for (int w = kLanes / 2; w >= 1; w >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, w);
                if (t < total) {
                    if (sub == 0) delta[(size_t)h * total + t] = dsum;
                    mine += expf(sink - lz[x]) * dsum;
                }
            }
        }
        // fixed-order reduction: the first lane of each row group, then warps in order
        if (sub != 0) mine = 0.f;
#pragma unroll
        for (int w = 16; w >= 1; w >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, w);
        if (threadIdx.x % 32 == 0) warp_sum[threadIdx.x / 32] = mine;
        __syncthreads();
        if (threadIdx.x == 0) {
            float acc = 0.f;
            for (int w = 0; w < kPreThreads / 32; ++w) acc += warp_sum[w];
            partial[(size_t)h * nchunks + chunk] = acc;
        }
        __syncthreads();  // warp_sum is rewritten by the next chunk
    }
}

// dsinks[h] = -(sum of the per-chunk partials of head h): one warp per head,
// lane l adds chunks l, l + 32, l + 64, ... in order, then the 32 lane sums
// are combined by a fixed butterfly, so the result is the same on every run.
// clear_flags (nullable): the workspace's device flag word, zeroed here so
// that the backward kernels after this one report their own conditions.
__global__ void dsink_reduce_kernel(int h_q, int nchunks, const float* __restrict__ partial,
                                    float* __restrict__ dsinks, uint32_t* clear_flags) {
    pdl_wait();  // the partials of preprocess_kernel
    if (clear_flags && blockIdx.x == 0 && threadIdx.x == 0) *clear_flags = 0u;
    const int h = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (h >= h_q) return;
    float acc = 0.f;
    for (int c = lane; c < nchunks; c += 32) acc += partial[(size_t)h * nchunks + c];
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    if (lane == 0) dsinks[h] = -acc;
}


int preprocess_chunks(int total) { return (total + kPreTokens - 1) / kPreTokens; }

template <typename T, int kD>
static void launch_preprocess(dim3 grid, cudaStream_t st, const Problem& P, const void* o,
                              const void* o_lo, const void* dout, const float* lse,
                              const float* sinks, float* delta, float* partial) {
    if (o_lo)
        preprocess_kernel<T, kD, true><<<grid, kPreThreads, 0, st>>>(
            P.total, P.h_q, (const T*)o, (const T*)o_lo, (const T*)dout, lse, sinks, delta, partial);
    else
        preprocess_kernel<T, kD, false><<<grid, kPreThreads, 0, st>>>(
            P.total, P.h_q, (const T*)o, nullptr, (const T*)dout, lse, sinks, delta, partial);
}

cudaError_t bwd_preprocess(const Problem& P, bool bf16, const float* sinks, const void* o,
                           const void* o_lo, const float* lse, const void* dout, float* delta,
                           float* dsinks, float* partial, uint32_t* clear_flags, cudaStream_t st) {
    const int nchunks = preprocess_chunks(P.total);
    if (nchunks > 0) {
        dim3 grid(P.h_q, nchunks < 65535 ? nchunks : 65535);
        const bool d128 = P.head_dim == 128;
        if (bf16 && d128)
            launch_preprocess<__nv_bfloat16, 128>(grid, st, P, o, o_lo, dout, lse, sinks, delta, partial);
        else if (bf16)
            launch_preprocess<__nv_bfloat16, 64>(grid, st, P, o, o_lo, dout, lse, sinks, delta, partial);
        else if (d128)
            launch_preprocess<float, 128>(grid, st, P, o, o_lo, dout, lse, sinks, delta, partial);
        else
            launch_preprocess<float, 64>(grid, st, P, o, o_lo, dout, lse, sinks, delta, partial);
        count_launches(1);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // right after preprocess_kernel of this call: it may start while that kernel finishes
    const dim3 grid((P.h_q + 3) / 4), block(128);  // one warp per head
    cudaError_t e = cudaSuccess;
    if (nchunks > 0)
        e = launch_after(dsink_reduce_kernel, grid, block, 0, st, P.h_q, nchunks,
                         (const float*)partial, dsinks, clear_flags);
    else
        dsink_reduce_kernel<<<grid, block, 0, st>>>(P.h_q, nchunks, partial, dsinks, clear_flags);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}


}  // namespace sinkattn
