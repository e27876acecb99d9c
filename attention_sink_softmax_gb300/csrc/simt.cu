// simt.cu - CUDA-core (FFMA) kernels for sink attention: the exact fp32 path,
// and the general path for shapes the tensor-core kernels do not take.
//
// Forward (page "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、超稳定！", sections
// "GPT-OSS中的带注意力槽的注意力机制" and "数学公式深入解读"): each row keeps a
// running maximum m and denominator l that start from the sink's own term
// (m = S_h, l = exp(S_h - m) = 1), so the sink joins the softmax denominator
// without a value row. Scores are kept in base-2 units (scale * log2 e folded
// into Q) and exponentials use exp2.
//
// Backward (section "反向传播的实现"): P = exp(S - LSE) needs no sink term since
// LSE includes it; dS = P (dO.V - D) with D_i = dO_i . O_i; the sink gradient is
// -sum_i exp(S_h - LSE_i) D_i, reduced in a fixed order.
#include "common.cuh"
#include "kernels.h"

namespace sinkattn {

// Every kernel is instantiated for head_dim kD = 64 and 128 (a thread keeps
// rows of kD fp32 values in registers; at 128 some of them live in local
// memory).
constexpr int kFwdRows = 128;   // query rows per block (one thread each)
constexpr int kFwdKeys = 32;    // keys per shared-memory tile

template <typename T, int kD>
__global__ void __launch_bounds__(kFwdRows)
simt_fwd_kernel(Problem P, const T* __restrict__ q, const T* __restrict__ k,
                const T* __restrict__ v, const float* __restrict__ sinks,
                T* __restrict__ o, float* __restrict__ lse, uint32_t* flags) {
    __shared__ float ks[kFwdKeys][kD];
    __shared__ float vs[kFwdKeys][kD];
    const int s = blockIdx.z, h = blockIdx.y;
    int start, L;
    seq_bounds(P, s, start, L);
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
        for (int c = 0; c < kD; ++c) o[qoff + c] = from_f32<T>(acc[c] * inv);
        lse[(size_t)h * P.total + start + i] = (m + log2f(l)) * kLn2;
    }
}

// ---------------------------------------------------------------------------
// Backward step 1: delta = rowsum(dO * O) in [h_q, T] and per-chunk partials of
// sum_t exp(S_h - LSE_t) * delta_t. One block = one head x kPreTokens tokens;
// kD / 8 lanes share one row, each lane one 16-byte (bf16) or 32-byte (fp32)
// piece of 8 elements. A thread issues the loads of 8 of its rows before using
// any, so every thread keeps 8 rows of O and dO in flight (memory-bound step).
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

template <typename T, int kD>
__global__ void __launch_bounds__(kPreThreads)
preprocess_kernel(int total, int h_q, const T* __restrict__ o, const T* __restrict__ dout,
                  const float* __restrict__ lse, const float* __restrict__ sinks,
                  float* __restrict__ delta, float* __restrict__ partial) {
    constexpr int kLanes = kD / 8;  // threads per row, 8 elements each
    constexpr int kPer = 8;
    constexpr int kRowsPerIter = kPreThreads / kLanes;
    constexpr int kIters = kPreTokens / kRowsPerIter;
    constexpr int kBatch = 8;  // rows of a thread in flight at once
    static_assert(kIters % kBatch == 0, "row batches");
    __shared__ float warp_sum[kPreThreads / 32];
    const int h = blockIdx.y;
    const int t0 = blockIdx.x * kPreTokens;
    const int sub = threadIdx.x % kLanes;
    const int r0 = threadIdx.x / kLanes;
    const float sink = __ldg(sinks + h);
    float mine = 0.f;  // this row-group's running sum, added in token order
    for (int b0 = 0; b0 < kIters; b0 += kBatch) {
        Piece8<T> po[kBatch], pd[kBatch];
        float lz[kBatch];
#pragma unroll
        for (int x = 0; x < kBatch; ++x) {
            const int t = t0 + r0 + (b0 + x) * kRowsPerIter;
            if (t < total) {
                const size_t off = ((size_t)t * h_q + h) * kD + sub * kPer;
                po[x] = load_piece(o + off);
                pd[x] = load_piece(dout + off);
                lz[x] = __ldg(lse + (size_t)h * total + t);
            }
        }
#pragma unroll
        for (int x = 0; x < kBatch; ++x) {
            const int t = t0 + r0 + (b0 + x) * kRowsPerIter;
            float dsum = t < total ? dot_piece(po[x], pd[x]) : 0.f;
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
        partial[(size_t)h * gridDim.x + blockIdx.x] = acc;
    }
}

// dsinks[h] = -sum over chunks (in chunk order) of the partials.
__global__ void dsink_reduce_kernel(int h_q, int nchunks, const float* __restrict__ partial,
                                    float* __restrict__ dsinks) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= h_q) return;
    float acc = 0.f;
    for (int c = 0; c < nchunks; ++c) acc += partial[(size_t)h * nchunks + c];
    dsinks[h] = -acc;
}

// ---------------------------------------------------------------------------
// Backward step 2 on CUDA cores: dQ by rows, dK/dV by keys (no atomics).
constexpr int kDqRows = 128;
constexpr int kDqKeys = 32;

template <typename T, int kD>
__global__ void __launch_bounds__(kDqRows)
simt_dq_kernel(Problem P, const T* __restrict__ q, const T* __restrict__ k,
               const T* __restrict__ v, const float* __restrict__ lse,
               const float* __restrict__ delta, const T* __restrict__ dout, T* __restrict__ dq) {
    __shared__ float ks[kDqKeys][kD];
    __shared__ float vs[kDqKeys][kD];
    const int s = blockIdx.z, h = blockIdx.y;
    int start, L;
    seq_bounds(P, s, start, L);
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
                 T* __restrict__ dk, T* __restrict__ dv) {
    constexpr int kKvKeys = kv_keys<kD>();
    constexpr int kKvRows = kv_rows<kD>();
    __shared__ float kown[kKvKeys][kD + 1];
    __shared__ float vown[kKvKeys][kD + 1];
    __shared__ float qs[kKvRows][kD];
    __shared__ float dos[kKvRows][kD];
    __shared__ float lse2s[kKvRows], ds_[kKvRows];
    const int s = blockIdx.z, hk = blockIdx.y;
    int start, L;
    seq_bounds(P, s, start, L);
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

// ---------------------------------------------------------------------------
// Host launchers.

template <typename T, int kD>
static cudaError_t launch_fwd_t(const Problem& P, const void* q, const void* k, const void* v,
                                const float* sinks, void* o, float* lse, uint32_t* flags,
                                cudaStream_t st) {
    dim3 grid((P.max_seqlen + kFwdRows - 1) / kFwdRows, P.h_q, P.nseq);
    simt_fwd_kernel<T, kD><<<grid, kFwdRows, 0, st>>>(P, (const T*)q, (const T*)k, (const T*)v,
                                                      sinks, (T*)o, lse, flags);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t simt_fwd(const Problem& P, bool bf16, const void* q, const void* k, const void* v,
                     const float* sinks, void* o, float* lse, uint32_t* flags, cudaStream_t st) {
    if (P.nseq == 0 || P.max_seqlen == 0) return cudaSuccess;
    if (P.head_dim == 128)
        return bf16 ? launch_fwd_t<__nv_bfloat16, 128>(P, q, k, v, sinks, o, lse, flags, st)
                    : launch_fwd_t<float, 128>(P, q, k, v, sinks, o, lse, flags, st);
    return bf16 ? launch_fwd_t<__nv_bfloat16, 64>(P, q, k, v, sinks, o, lse, flags, st)
                : launch_fwd_t<float, 64>(P, q, k, v, sinks, o, lse, flags, st);
}

int preprocess_chunks(int total) { return (total + kPreTokens - 1) / kPreTokens; }

cudaError_t bwd_preprocess(const Problem& P, bool bf16, const float* sinks, const void* o,
                           const float* lse, const void* dout, float* delta, float* dsinks,
                           float* partial, cudaStream_t st) {
    const int nchunks = preprocess_chunks(P.total);
    if (nchunks > 0) {
        dim3 grid(nchunks, P.h_q);
        const bool d128 = P.head_dim == 128;
        if (bf16 && d128)
            preprocess_kernel<__nv_bfloat16, 128><<<grid, kPreThreads, 0, st>>>(
                P.total, P.h_q, (const __nv_bfloat16*)o, (const __nv_bfloat16*)dout, lse, sinks,
                delta, partial);
        else if (bf16)
            preprocess_kernel<__nv_bfloat16, 64><<<grid, kPreThreads, 0, st>>>(
                P.total, P.h_q, (const __nv_bfloat16*)o, (const __nv_bfloat16*)dout, lse, sinks,
                delta, partial);
        else if (d128)
            preprocess_kernel<float, 128><<<grid, kPreThreads, 0, st>>>(
                P.total, P.h_q, (const float*)o, (const float*)dout, lse, sinks, delta, partial);
        else
            preprocess_kernel<float, 64><<<grid, kPreThreads, 0, st>>>(
                P.total, P.h_q, (const float*)o, (const float*)dout, lse, sinks, delta, partial);
        count_launches(1);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    dsink_reduce_kernel<<<(P.h_q + 127) / 128, 128, 0, st>>>(P.h_q, nchunks, partial, dsinks);
    count_launches(1);
    return cudaGetLastError();
}

template <typename T, int kD>
static cudaError_t launch_bwd_t(const Problem& P, const void* q, const void* k, const void* v,
                                const float* lse, const float* delta, const void* dout, void* dq,
                                void* dk, void* dv, cudaStream_t st) {
    dim3 gq((P.max_seqlen + kDqRows - 1) / kDqRows, P.h_q, P.nseq);
    simt_dq_kernel<T, kD><<<gq, kDqRows, 0, st>>>(P, (const T*)q, (const T*)k, (const T*)v, lse,
                                                  delta, (const T*)dout, (T*)dq);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    constexpr int kKeys = kv_keys<kD>();
    dim3 gk((P.max_seqlen + kKeys - 1) / kKeys, P.h_kv, P.nseq);
    simt_dkdv_kernel<T, kD><<<gk, kKeys, 0, st>>>(P, (const T*)q, (const T*)k, (const T*)v, lse,
                                                  delta, (const T*)dout, (T*)dk, (T*)dv);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t simt_bwd_main(const Problem& P, bool bf16, const void* q, const void* k, const void* v,
                          const float* lse, const float* delta, const void* dout, void* dq,
                          void* dk, void* dv, cudaStream_t st) {
    if (P.nseq == 0 || P.max_seqlen == 0) return cudaSuccess;
    if (P.head_dim == 128)
        return bf16 ? launch_bwd_t<__nv_bfloat16, 128>(P, q, k, v, lse, delta, dout, dq, dk, dv, st)
                    : launch_bwd_t<float, 128>(P, q, k, v, lse, delta, dout, dq, dk, dv, st);
    return bf16 ? launch_bwd_t<__nv_bfloat16, 64>(P, q, k, v, lse, delta, dout, dq, dk, dv, st)
                : launch_bwd_t<float, 64>(P, q, k, v, lse, delta, dout, dq, dk, dv, st);
}

}  // namespace sinkattn
