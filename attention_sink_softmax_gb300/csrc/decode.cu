// decode.cu - single-query (decode / streaming inference) sink attention.
//
// What it computes (page "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、超稳定！"):
// the forward of sections "GPT-OSS中的带注意力槽的注意力机制" and "数学公式深入解读"
// for one query row that is the last token of its context, i.e. row
// kv_len - 1 of the training forward on that context. The sinks exist for
// streaming inference (section "FlashAttentionV3对注意力槽的支持"), and section
// "纠正训练与推理不一致问题" (Fig. 4) is about the training and inference paths
// disagreeing; sink_attn_decode is the inference path of this library.
//
// Split over keys. Query b's allowed keys (its whole context, or the last
// `window` of it) are cut into nsplit chunks; decode_split_kernel computes,
// per (chunk, key/value head, query) and for every query head h of the group,
// the chunk's running max m_c, sum l_c = sum exp(s - m_c) and unnormalised
// o_c = sum exp(s - m_c) v, WITHOUT the sink. decode_merge_kernel then adds
// the sink exactly once:
//   M   = max(S_h, max_c m_c)
//   l   = exp(S_h - M) + sum_c l_c exp(m_c - M)
//   O   = sum_c o_c exp(m_c - M) / l,   LSE = M + ln l.
// Scores are kept in log2 units (scale * log2 e folded into q).
//
// The work is bandwidth-bound (K and V rows are read once per key/value head
// for all g query heads of the group), so it runs on the CUDA cores: a
// 128-key tile of K and of V is staged in shared memory (16-byte global loads;
// rows padded to an odd number of 32-bit words so that a thread per key reads
// its row without bank conflicts), 256 threads form the g x 128 score tile,
// and warp w then owns query heads w, w+8, ...: tile max and sum by warp
// reductions, and the P V product with lane l holding output columns 2l, 2l+1.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace sinkattn {
namespace {

constexpr int kD = 64;
constexpr int kTile = 128;     // keys per tile
constexpr int kThreads = 256;  // 8 warps
constexpr int kPartFloats = 2 + kD;  // m, l, o[64]

// Element access; kStride is the padded shared-memory row length in elements
// (an odd number of 32-bit words: 33 for bf16, 65 for fp32).
template <typename T>
struct Elt;
template <>
struct Elt<float> {
    static constexpr int kStride = 65;
    static __device__ __forceinline__ float2 pair(const float* p) { return make_float2(p[0], p[1]); }
    static __device__ __forceinline__ float one(const float* p) { return *p; }
};
template <>
struct Elt<__nv_bfloat16> {
    static constexpr int kStride = 66;
    static __device__ __forceinline__ float2 pair(const __nv_bfloat16* p) {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
    }
    static __device__ __forceinline__ float one(const __nv_bfloat16* p) { return __bfloat162float(*p); }
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// The query's allowed keys [lo, len) of its context, or false (and a flag) if
// its context is invalid.
__device__ __forceinline__ bool query_keys(const DecodeArgs& a, const int32_t* kv_start,
                                           const int32_t* kv_len, int b, int& start, int& lo,
                                           int& len) {
    start = __ldg(kv_start + b);
    len = __ldg(kv_len + b);
    if (len < 1 || len > a.max_len || start < 0 || (int64_t)start + len > a.total) return false;
    lo = a.window > 0 ? max(0, len - a.window) : 0;
    return true;
}

// grid (nsplit, h_kv, batch); dynamic shared memory: q [g][64] fp32, s [g][128]
// fp32, K and V tiles [128][kStride] of T.
template <typename T>
__global__ void __launch_bounds__(kThreads)
decode_split_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                    const int32_t* __restrict__ kv_start, const int32_t* __restrict__ kv_len,
                    const DecodeArgs a, float* __restrict__ part, uint32_t* flags) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int g = a.group;
    float* qs = reinterpret_cast<float*>(smem);          // [g][64]
    float* ss = qs + g * kD;                              // [g][128]
    constexpr int kS = Elt<T>::kStride;
    T* ks = reinterpret_cast<T*>(ss + g * kTile);         // [128][kS]
    T* vs = ks + kTile * kS;                              // [128][kS]
    const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    int start, lo, len;
    const bool valid = query_keys(a, kv_start, kv_len, b, start, lo, len);
    if (!valid && split == 0 && hk == 0 && threadIdx.x == 0) atomicOr(flags, kFlagSeqTooLong);
    // this chunk's keys [k_begin, k_end) of the context
    int k_begin = 0, k_end = 0;
    if (valid) {
        const int n = len - lo;
        const int chunk = (n + a.nsplit - 1) / a.nsplit;
        k_begin = lo + split * chunk;
        k_end = min(len, k_begin + chunk);
    }

    // q rows of the group, scaled into log2 units
    for (int i = threadIdx.x; i < g * kD; i += kThreads) {
        const int gi = i / kD, c = i % kD;
        qs[i] = Elt<T>::one(q + ((size_t)b * a.h_q + hk * g + gi) * kD + c) * a.scale_log2;
    }
    // per warp: query heads w, w+8, ... ; m, l and two output columns per lane
    constexpr int kMaxHeadsPerWarp = 8;  // group sizes up to 64
    float m[kMaxHeadsPerWarp], l[kMaxHeadsPerWarp], o0[kMaxHeadsPerWarp], o1[kMaxHeadsPerWarp];
#pragma unroll
    for (int x = 0; x < kMaxHeadsPerWarp; ++x) {
        m[x] = -INFINITY;
        l[x] = 0.f;
        o0[x] = 0.f;
        o1[x] = 0.f;
    }
    __syncthreads();

    const int row_elems = a.h_kv * kD;  // elements between consecutive tokens' rows
    for (int t0 = k_begin; t0 < k_end; t0 += kTile) {
        const int nk = min(kTile, k_end - t0);
        // stage K and V rows of this tile (16-byte pieces; rows past the chunk are zero)
        constexpr int kPer16 = 16 / sizeof(T);
        constexpr int kPieces = kTile * kD / kPer16;
        for (int i = threadIdx.x; i < kPieces; i += kThreads) {
            const int j = i / (kD / kPer16), c = (i % (kD / kPer16)) * kPer16;
            uint4 kx = make_uint4(0, 0, 0, 0), vx = make_uint4(0, 0, 0, 0);
            if (j < nk) {
                const size_t off = (size_t)(start + t0 + j) * row_elems + (size_t)hk * kD + c;
                kx = __ldg(reinterpret_cast<const uint4*>(k + off));
                vx = __ldg(reinterpret_cast<const uint4*>(v + off));
            }
            // 4-byte stores: padded rows are only 4-byte aligned
            uint32_t* kw = reinterpret_cast<uint32_t*>(ks + j * kS + c);
            uint32_t* vw = reinterpret_cast<uint32_t*>(vs + j * kS + c);
            kw[0] = kx.x; kw[1] = kx.y; kw[2] = kx.z; kw[3] = kx.w;
            vw[0] = vx.x; vw[1] = vx.y; vw[2] = vx.z; vw[3] = vx.w;
        }
        __syncthreads();
        // scores: thread = (key j, half of the heads)
        {
            const int j = threadIdx.x % kTile, half = threadIdx.x / kTile;
            for (int gi = half; gi < g; gi += 2) {
                float acc = 0.f;
#pragma unroll
                for (int c = 0; c < kD; c += 2) {
                    const float2 kk = Elt<T>::pair(ks + j * kS + c);
                    acc = fmaf(qs[gi * kD + c], kk.x, acc);
                    acc = fmaf(qs[gi * kD + c + 1], kk.y, acc);
                }
                ss[gi * kTile + j] = j < nk ? acc : -INFINITY;
            }
        }
        __syncthreads();
        // online softmax and P V, warp w for heads w, w+8, ...
#pragma unroll
        for (int x = 0; x < kMaxHeadsPerWarp; ++x) {
            const int gi = warp + 8 * x;
            if (gi >= g) break;
            float* srow = ss + gi * kTile;
            float tmax = -INFINITY;
#pragma unroll
            for (int u = 0; u < kTile / 32; ++u) tmax = fmaxf(tmax, srow[lane + 32 * u]);
            tmax = warp_max(tmax);
            const float m_new = fmaxf(m[x], tmax);  // finite: the tile has at least one key
            const float corr = m[x] == -INFINITY ? 0.f : exp2f(m[x] - m_new);
            float psum = 0.f;
#pragma unroll
            for (int u = 0; u < kTile / 32; ++u) {
                const float p = exp2f(srow[lane + 32 * u] - m_new);
                srow[lane + 32 * u] = p;
                psum += p;
            }
            psum = warp_sum(psum);
            l[x] = l[x] * corr + psum;
            m[x] = m_new;
            float a0 = o0[x] * corr, a1 = o1[x] * corr;
            __syncwarp();
            for (int j = 0; j < nk; ++j) {
                const float p = srow[j];
                const float2 vv = Elt<T>::pair(vs + j * kS + 2 * lane);
                a0 = fmaf(p, vv.x, a0);
                a1 = fmaf(p, vv.y, a1);
            }
            o0[x] = a0;
            o1[x] = a1;
        }
        __syncthreads();
    }
    // partial of this chunk for every query head of the group (m = -inf, l = 0 when empty)
#pragma unroll
    for (int x = 0; x < kMaxHeadsPerWarp; ++x) {
        const int gi = warp + 8 * x;
        if (gi >= g) break;
        float* pp = part + (((size_t)split * a.batch + b) * a.h_q + hk * g + gi) * kPartFloats;
        if (lane == 0) {
            pp[0] = m[x];
            pp[1] = l[x];
        }
        *reinterpret_cast<float2*>(pp + 2 + 2 * lane) = make_float2(o0[x], o1[x]);
    }
}

// One warp per (query, head): merges the chunks and adds the sink once.
template <typename T>
__global__ void __launch_bounds__(kThreads)
decode_merge_kernel(const float* __restrict__ part, const float* __restrict__ sinks,
                    const int32_t* __restrict__ kv_start, const int32_t* __restrict__ kv_len,
                    const DecodeArgs a, T* __restrict__ o, float* __restrict__ lse) {
    const int wid = blockIdx.x * (kThreads / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (wid >= a.batch * a.h_q) return;
    const int b = wid / a.h_q, h = wid % a.h_q;
    int start, lo, len;
    const bool valid = query_keys(a, kv_start, kv_len, b, start, lo, len);
    const float sink = __ldg(sinks + h) * kLog2e;
    float M = sink;
    if (valid)
        for (int c = 0; c < a.nsplit; ++c)
            M = fmaxf(M, part[(((size_t)c * a.batch + b) * a.h_q + h) * kPartFloats]);
    float lsum = M == -INFINITY ? 0.f : exp2f(sink - M);
    float acc0 = 0.f, acc1 = 0.f;
    if (valid && M != -INFINITY) {
        for (int c = 0; c < a.nsplit; ++c) {
            const float* pp = part + (((size_t)c * a.batch + b) * a.h_q + h) * kPartFloats;
            const float mc = pp[0];
            if (mc == -INFINITY) continue;  // an empty chunk
            const float wgt = exp2f(mc - M);
            lsum = fmaf(pp[1], wgt, lsum);
            const float2 oc = *reinterpret_cast<const float2*>(pp + 2 + 2 * lane);
            acc0 = fmaf(oc.x, wgt, acc0);
            acc1 = fmaf(oc.y, wgt, acc1);
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    T* dst = o + ((size_t)b * a.h_q + h) * kD + 2 * lane;
    if constexpr (sizeof(T) == 2) {
        *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc0 * inv, acc1 * inv);
    } else {
        *reinterpret_cast<float2*>(dst) = make_float2(acc0 * inv, acc1 * inv);
    }
    if (lane == 0) lse[(size_t)h * a.batch + b] = lsum > 0.f ? (M + log2f(lsum)) * kLn2 : -INFINITY;
}

template <typename T>
cudaError_t launch(const DecodeArgs& a, const void* q, const void* k, const void* v,
                   const float* sinks, const int32_t* kv_start, const int32_t* kv_len, void* o,
                   float* lse, float* part, uint32_t* flags, cudaStream_t st) {
    const size_t smem =
        sizeof(float) * (size_t)a.group * (kD + kTile) + 2 * sizeof(T) * kTile * Elt<T>::kStride;
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.nsplit, a.h_kv, a.batch);
    decode_split_kernel<T><<<grid, kThreads, smem, st>>>((const T*)q, (const T*)k, (const T*)v,
                                                         kv_start, kv_len, a, part, flags);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int warps = a.batch * a.h_q;
    decode_merge_kernel<T><<<(warps + kThreads / 32 - 1) / (kThreads / 32), kThreads, 0, st>>>(
        part, sinks, kv_start, kv_len, a, (T*)o, lse);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

int decode_splits(int batch, int h_kv, int max_len) {
    // about 512 CTAs in the split kernel, at least one 128-key tile per chunk
    const int want = (512 + batch * h_kv - 1) / std::max(1, batch * h_kv);
    const int tiles = std::max(1, (max_len + kTile - 1) / kTile);
    return std::max(1, std::min({want, tiles, kDecodeMaxSplits}));
}

size_t decode_partial_floats(int batch, int h_q) {
    return (size_t)kDecodeMaxSplits * batch * h_q * kPartFloats;
}

cudaError_t decode(const DecodeArgs& a, bool bf16, const void* q, const void* k, const void* v,
                   const float* sinks, const int32_t* kv_start, const int32_t* kv_len, void* o,
                   float* lse, float* part, uint32_t* flags, cudaStream_t st) {
    if (a.batch == 0) return cudaSuccess;
    return bf16 ? launch<__nv_bfloat16>(a, q, k, v, sinks, kv_start, kv_len, o, lse, part, flags, st)
                : launch<float>(a, q, k, v, sinks, kv_start, kv_len, o, lse, part, flags, st);
}

}  // namespace sinkattn
