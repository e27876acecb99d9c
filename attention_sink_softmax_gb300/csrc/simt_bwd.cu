// simt_bwd.cu - CUDA-core (FFMA) backward main step of sink attention: the
// exact fp32 path, and the general path for shapes the tensor-core kernels do
// not take (page "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、超稳定！", section
// "反向传播的实现"): P = exp(S - LSE) needs no sink term since LSE includes it;
// dS = P (dO.V - D) with D_i = dO_i . O_i from the preprocess step.
#include "common.cuh"
#include "kernels.h"

namespace sinkattn {

// Instantiated for head_dim kD = 64 and 128, like the forward.
// Backward step 2 on CUDA cores: dQ by rows, dK/dV by keys (no atomics).
constexpr int kDqRows = 128;
constexpr int kDqKeys = 32;

template <typename T, int kD>
__global__ void __launch_bounds__(kDqRows)
simt_dq_kernel(Problem P, const T* __restrict__ q, const T* __restrict__ k,
               const T* __restrict__ v, const float* __restrict__ lse,
               const float* __restrict__ delta, const T* __restrict__ dout, T* __restrict__ dq,
               uint32_t* flags) {
    __shared__ float ks[kDqKeys][kD];
    __shared__ float vs[kDqKeys][kD];
    const int s = blockIdx.z, h = blockIdx.y;
    int start, L;
    if (!seq_bounds_checked(P, s, start, L, flags)) return;
    const int r0 = blockIdx.x * kDqRows;
    if (r0 >= L) return;
    const int i = r0 + threadIdx.x;
    const bool valid = i < L;
    const int hk = h / P.group;
    const size_t off = ((size_t)(start + (valid ? i : r0)) * P.h_q + h) * kD;
    float qr[kD], dor[kD], acc[kD];
#pragma unroll
    for (int c = 0; c < kD; ++c) {
        qr[c] = valid ? to_f32(q[off + c]) * P.scale_log2 : 0.f;
        dor[c] = valid ? to_f32(dout[off + c]) : 0.f;
        acc[c] = 0.f;
    }
    const size_t rix = (size_t)h * P.total + start + (valid ? i : r0);
    const float lse2 = valid ? lse[rix] * kLog2e : 0.f;
    const float Di = valid ? delta[rix] : 0.f;
    const int jlo = valid ? key_lo(P, i) : 0;
    const int jhi = valid ? key_hi(P, i, L) : 0;
    const int rlast = min(r0 + kDqRows - 1, L - 1);
    const int jb0 = key_lo(P, r0), jb1 = key_hi(P, rlast, L);
    for (int jt = jb0; jt < jb1; jt += kDqKeys) {
        __syncthreads();
        for (int e = threadIdx.x; e < kDqKeys * kD; e += kDqRows) {
            const int jj = e / kD, c = e % kD, j = jt + jj;
            float kv = 0.f, vv = 0.f;
            if (j < jb1) {
                const size_t o2 = ((size_t)(start + j) * P.h_kv + hk) * kD + c;
                kv = to_f32(k[o2]);
                vv = to_f32(v[o2]);
            }
            ks[jj][c] = kv;
            vs[jj][c] = vv;
        }
        __syncthreads();
        for (int jj = 0; jj < kDqKeys; ++jj) {
            const int j = jt + jj;
            if (j < jlo || j >= jhi) continue;
            float sd = 0.f, dp = 0.f;
#pragma unroll
            for (int c = 0; c < kD; ++c) {
                sd = fmaf(qr[c], ks[jj][c], sd);
                dp = fmaf(dor[c], vs[jj][c], dp);
            }
            const float p = exp2f(sd - lse2);
            const float ds = p * (dp - Di);
#pragma unroll
            for (int c = 0; c < kD; ++c) acc[c] = fmaf(ds, ks[jj][c], acc[c]);
        }
    }
    if (valid) {
#pragma unroll
        for (int c = 0; c < kD; ++c) dq[off + c] = from_f32<T>(acc[c] * P.scale);
    }
}

// keys per block (one thread each) and query rows per shared-memory tile,
// sized so that the static shared memory stays under 48 KB
template <int kD> constexpr int kv_keys() { return kD == 64 ? 64 : 32; }
template <int kD> constexpr int kv_rows() { return kD == 64 ? 16 : 8; }

template <typename T, int kD>
__global__ void __launch_bounds__(kv_keys<kD>())
simt_dkdv_kernel(Problem P, const T* __restrict__ q, const T* __restrict__ k,
                 const T* __restrict__ v, const float* __restrict__ lse,
                 const float* __restrict__ delta, const T* __restrict__ dout,
                 T* __restrict__ dk, T* __restrict__ dv, uint32_t* flags) {
    constexpr int kKvKeys = kv_keys<kD>();
    constexpr int kKvRows = kv_rows<kD>();
    __shared__ float kown[kKvKeys][kD + 1];
    __shared__ float vown[kKvKeys][kD + 1];
    __shared__ float qs[kKvRows][kD];
    __shared__ float dos[kKvRows][kD];
    __shared__ float lse2s[kKvRows], ds_[kKvRows];
    const int s = blockIdx.z, hk = blockIdx.y;
    int start, L;
    if (!seq_bounds_checked(P, s, start, L, flags)) return;
    const int j0 = blockIdx.x * kKvKeys;
    if (j0 >= L) return;
    const int j = j0 + threadIdx.x;
    const bool valid = j < L;
    const size_t koff = ((size_t)(start + (valid ? j : j0)) * P.h_kv + hk) * kD;
    for (int c = 0; c < kD; ++c) {
        kown[threadIdx.x][c] = valid ? to_f32(k[koff + c]) * P.scale_log2 : 0.f;
        vown[threadIdx.x][c] = valid ? to_f32(v[koff + c]) : 0.f;
    }
    float dka[kD], dva[kD];
#pragma unroll
    for (int c = 0; c < kD; ++c) dka[c] = dva[c] = 0.f;
    const int ilo = valid ? row_lo(P, j) : 0;
    const int ihi = valid ? row_hi(P, j, L) : 0;
    const int jlast = min(j0 + kKvKeys - 1, L - 1);
    const int ib0 = row_lo(P, j0), ib1 = row_hi(P, jlast, L);
    for (int h = hk * P.group; h < (hk + 1) * P.group; ++h) {
        for (int it = ib0; it < ib1; it += kKvRows) {
            __syncthreads();
            for (int e = threadIdx.x; e < kKvRows * kD; e += kKvKeys) {
                const int ii = e / kD, c = e % kD, i = it + ii;
                float qv = 0.f, dv_ = 0.f;
                if (i < ib1) {
                    const size_t o2 = ((size_t)(start + i) * P.h_q + h) * kD + c;
                    qv = to_f32(q[o2]);
                    dv_ = to_f32(dout[o2]);
                }
                qs[ii][c] = qv;
                dos[ii][c] = dv_;
            }
            if (threadIdx.x < kKvRows) {
                const int i = it + threadIdx.x;
                const size_t rix = (size_t)h * P.total + start + i;
                lse2s[threadIdx.x] = i < ib1 ? lse[rix] * kLog2e : 0.f;
                ds_[threadIdx.x] = i < ib1 ? delta[rix] : 0.f;
            }
            __syncthreads();
            for (int ii = 0; ii < kKvRows; ++ii) {
                const int i = it + ii;
                if (i < ilo || i >= ihi) continue;
                float sd = 0.f, dp = 0.f;
#pragma unroll
                for (int c = 0; c < kD; ++c) {
                    sd = fmaf(qs[ii][c], kown[threadIdx.x][c], sd);
                    dp = fmaf(dos[ii][c], vown[threadIdx.x][c], dp);
                }
                const float p = exp2f(sd - lse2s[ii]);
                const float dsv = p * (dp - ds_[ii]);
#pragma unroll
                for (int c = 0; c < kD; ++c) {
                    dva[c] = fmaf(p, dos[ii][c], dva[c]);
                    dka[c] = fmaf(dsv, qs[ii][c], dka[c]);
                }
            }
        }
    }
    if (valid) {
#pragma unroll
        for (int c = 0; c < kD; ++c) {
            dk[koff + c] = from_f32<T>(dka[c] * P.scale);
            dv[koff + c] = from_f32<T>(dva[c]);
        }
    }
}


template <typename T, int kD>
static cudaError_t launch_bwd_t(const Problem& P, const void* q, const void* k, const void* v,
                                const float* lse, const float* delta, const void* dout, void* dq,
                                void* dk, void* dv, uint32_t* flags, cudaStream_t st) {
    dim3 gq((P.max_seqlen + kDqRows - 1) / kDqRows, P.h_q, P.nseq);
    simt_dq_kernel<T, kD><<<gq, kDqRows, 0, st>>>(P, (const T*)q, (const T*)k, (const T*)v, lse,
                                                  delta, (const T*)dout, (T*)dq, flags);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    constexpr int kKeys = kv_keys<kD>();
    dim3 gk((P.max_seqlen + kKeys - 1) / kKeys, P.h_kv, P.nseq);
    simt_dkdv_kernel<T, kD><<<gk, kKeys, 0, st>>>(P, (const T*)q, (const T*)k, (const T*)v, lse,
                                                  delta, (const T*)dout, (T*)dk, (T*)dv, flags);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t simt_bwd_main(const Problem& P, bool bf16, const void* q, const void* k, const void* v,
                          const float* lse, const float* delta, const void* dout, void* dq,
                          void* dk, void* dv, uint32_t* flags, cudaStream_t st) {
    if (P.nseq == 0 || P.max_seqlen == 0) return cudaSuccess;
    if (P.head_dim == 128)
        return bf16 ? launch_bwd_t<__nv_bfloat16, 128>(P, q, k, v, lse, delta, dout, dq, dk, dv, flags, st)
                    : launch_bwd_t<float, 128>(P, q, k, v, lse, delta, dout, dq, dk, dv, flags, st);
    return bf16 ? launch_bwd_t<__nv_bfloat16, 64>(P, q, k, v, lse, delta, dout, dq, dk, dv, flags, st)
                : launch_bwd_t<float, 64>(P, q, k, v, lse, delta, dout, dq, dk, dv, flags, st);
}


}  // namespace sinkattn
