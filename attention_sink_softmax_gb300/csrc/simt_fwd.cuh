// simt_fwd.cuh - CUDA-core (FFMA) forward for sink attention: the exact fp32
// path, and the general path for shapes the tensor-core kernels do not take.
// Instantiated for head_dim 64 in simt_fwd64.cu and 128 in simt_fwd128_*.cu
// (separate files so that they compile in parallel). The matching backward is
// in simt_bwd.cu, the preprocess step in preprocess.cu.
//
// Forward (page "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、超稳定！", sections
// "GPT-OSS中的带注意力槽的注意力机制" and "数学公式深入解读"): each row keeps a
// running maximum m and denominator l that start from the sink's own term
// (m = S_h, l = exp(S_h - m) = 1), so the sink joins the softmax denominator
// without a value row. Scores are kept in base-2 units (scale * log2 e folded
// into Q) and exponentials use exp2.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace sinkattn {

// Instantiated for head_dim kD = 64 and 128 (a thread keeps rows of kD fp32
// values in registers; at 128 some of them live in local memory).
constexpr int kFwdRows = 128;   // query rows per block (one thread each)
constexpr int kFwdKeys = 32;    // keys per shared-memory tile

template <typename T, int kD>
__global__ void __launch_bounds__(kFwdRows)
simt_fwd_kernel(Problem P, const T* __restrict__ q, const T* __restrict__ k,
                const T* __restrict__ v, const float* __restrict__ sinks,
                T* __restrict__ o, T* __restrict__ o_lo, float* __restrict__ lse, uint32_t* flags) {
    __shared__ float ks[kFwdKeys][kD];
    __shared__ float vs[kFwdKeys][kD];
    const int s = blockIdx.z, h = blockIdx.y;
    int start, L;
    if (!seq_bounds_checked(P, s, start, L, flags)) return;
    if (blockIdx.x == 0 && threadIdx.x == 0 && L > P.max_seqlen) atomicOr(flags, kFlagSeqTooLong);
    const int r0 = blockIdx.x * kFwdRows;
    if (r0 >= L) return;
    const int i = r0 + threadIdx.x;
    const bool valid = i < L;
    const int hk = h / P.group;

    float qr[kD];
    const size_t qoff = ((size_t)(start + (valid ? i : r0)) * P.h_q + h) * kD;
#pragma unroll
    for (int c = 0; c < kD; ++c) qr[c] = valid ? to_f32(q[qoff + c]) * P.scale_log2 : 0.f;

    float m = __ldg(sinks + h) * kLog2e;  // sink-seeded running max (base 2)
    float l = m == -INFINITY ? 0.f : 1.f;   // the sink's own term exp2(S_h - m)
    float acc[kD];
#pragma unroll
    for (int c = 0; c < kD; ++c) acc[c] = 0.f;

    const int jlo = valid ? key_lo(P, i) : 0;
    const int jhi = valid ? key_hi(P, i, L) : 0;
    const int rlast = min(r0 + kFwdRows - 1, L - 1);
    const int jb0 = key_lo(P, r0), jb1 = key_hi(P, rlast, L);

    for (int jt = jb0; jt < jb1; jt += kFwdKeys) {
        __syncthreads();
        for (int e = threadIdx.x; e < kFwdKeys * kD; e += kFwdRows) {
            const int jj = e / kD, c = e % kD, j = jt + jj;
            float kv = 0.f, vv = 0.f;
            if (j < jb1) {
                const size_t off = ((size_t)(start + j) * P.h_kv + hk) * kD + c;
                kv = to_f32(k[off]);
                vv = to_f32(v[off]);
            }
            ks[jj][c] = kv;
            vs[jj][c] = vv;
        }
        __syncthreads();
        float sc[kFwdKeys];
        float tmax = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < kFwdKeys; ++jj) {
            const int j = jt + jj;
            float dot = 0.f;
#pragma unroll
            for (int c = 0; c < kD; ++c) dot = fmaf(qr[c], ks[jj][c], dot);
            sc[jj] = (j >= jlo && j < jhi) ? dot : -INFINITY;
            tmax = fmaxf(tmax, sc[jj]);
        }
        const float mn = fmaxf(m, tmax);
        // reference point for the exponentials; finite unless the sink is -inf
        // and no key has been seen yet (then every term is 0)
        const float mref = mn == -INFINITY ? 0.f : mn;
        const float corr = exp2f(m - mref);
        l *= corr;
#pragma unroll
        for (int c = 0; c < kD; ++c) acc[c] *= corr;
#pragma unroll
        for (int jj = 0; jj < kFwdKeys; ++jj) {
            const float p = exp2f(sc[jj] - mref);
            l += p;
#pragma unroll
            for (int c = 0; c < kD; ++c) acc[c] = fmaf(p, vs[jj][c], acc[c]);
        }
        m = mn;
    }
    if (valid) {
        const float inv = 1.f / l;
#pragma unroll
        for (int c = 0; c < kD; ++c) {
            const float x = acc[c] * inv;
            const T hi = from_f32<T>(x);
            o[qoff + c] = hi;
            // low-order part (bf16 only): what the rounding of O dropped
            if (o_lo) o_lo[qoff + c] = from_f32<T>(x - to_f32(hi));
        }
        lse[(size_t)h * P.total + start + i] = (m + log2f(l)) * kLn2;
    }
}


// ---------------------------------------------------------------------------
// Host launcher.

template <typename T, int kD>
cudaError_t launch_simt_fwd(const Problem& P, const void* q, const void* k, const void* v,
                            const float* sinks, void* o, void* o_lo, float* lse, uint32_t* flags,
                            cudaStream_t st) {
    dim3 grid((P.max_seqlen + kFwdRows - 1) / kFwdRows, P.h_q, P.nseq);
    simt_fwd_kernel<T, kD><<<grid, kFwdRows, 0, st>>>(P, (const T*)q, (const T*)k, (const T*)v,
                                                      sinks, (T*)o, (T*)o_lo, lse, flags);
    count_launches(1);
    return cudaGetLastError();
}

// instantiated in simt_fwd128_bf16.cu and simt_fwd128_f32.cu
extern template cudaError_t launch_simt_fwd<__nv_bfloat16, 128>(
    const Problem&, const void*, const void*, const void*, const float*, void*, void*, float*,
    uint32_t*, cudaStream_t);
extern template cudaError_t launch_simt_fwd<float, 128>(
    const Problem&, const void*, const void*, const void*, const float*, void*, void*, float*,
    uint32_t*, cudaStream_t);

}  // namespace sinkattn
