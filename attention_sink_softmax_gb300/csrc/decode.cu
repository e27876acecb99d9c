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
// `window` of it) are cut into nsplit chunks; a split kernel computes, per
// (chunk, key/value head, query) and for every query head h of the group, the
// chunk's running max m_c, sum l_c = sum exp(s - m_c) and unnormalised
// o_c = sum exp(s - m_c) v, WITHOUT the sink. The merge then adds the sink
// exactly once:
//   M   = max(S_h, max_c m_c)
//   l   = exp(S_h - M) + sum_c l_c exp(m_c - M)
//   O   = sum_c o_c exp(m_c - M) / l,   LSE = M + ln l.
// Scores are kept in log2 units (scale * log2 e applied before exp2).
//
// The work is bandwidth-bound: every K and V row of a key/value head is read
// once for all g query heads of its group, 2 x 64 x 2 bytes per key for
// 4 x 64 x g FLOP. Two split kernels:
//
// decode_mma_kernel (bf16, g <= 16) keeps it near the HBM bound. Per CTA four
// warps, each an independent stream over the chunk's 32-key stages (warp w
// takes stages w, w+4, ...): its lane 0 brings K and V boxes of a stage in by
// TMA (128-byte swizzle) into one of two shared-memory slots of its own,
// completing on the slot's mbarrier, so a warp computes one stage while the
// next one lands. The two products are warp-level mma.sync m16n8k16 tensor
// operations with the keys, not the few query heads, on the 16-row side:
//   S^T [keys x heads] = K [keys x 64] . Q^T       (Q^T fragments held in registers)
//   O^T [64 x heads]  += V^T [64 x keys] . P^T      (V^T by ldmatrix.trans)
// and P^T comes from the S^T accumulator by an 8x8 transpose in registers
// (movmatrix), so nothing of the score tile goes through shared memory. Each
// warp keeps its own running max, sum and O^T; the four are merged through
// shared memory into the CTA's chunk partial, and the last CTA of each
// (query, key/value head) to finish merges the chunks in the same launch.
// tcgen05 is not used here: a tcgen05.mma costs about as long for N = 8..16
// as for N = 128, so products this narrow would be tensor-pipe-bound above
// the HBM time.
//
// decode_split_kernel (fp32 caches, larger groups) runs on the CUDA cores,
// followed by decode_merge_kernel: a 128-key tile of K and of V is staged in
// shared memory (16-byte global loads; rows padded to an odd number of 32-bit
// words so that a thread per key reads its row without bank conflicts), 256
// threads form the g x 128 score tile,
// and warp w then owns query heads w, w+8, ...: tile max and sum by warp
// reductions, and the P V product with lane l holding output columns 2l, 2l+1.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

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

// Merge of query b, head h by one warp: adds the sink once. Lane c (and
// c + 32) holds chunk c's max and sum, so the global max and the weights come
// from two warp reductions; the weighted sum of the chunks' outputs then runs
// with lane l on columns 2l, 2l+1. Partials are read past L1 (other CTAs
// wrote them).
template <typename T>
__device__ __forceinline__ void merge_head(const float* part, const float* __restrict__ sinks,
                                           const DecodeArgs& a, int b, int h, bool valid,
                                           T* __restrict__ o, float* __restrict__ lse, int lane) {
    const float sink = __ldg(sinks + h) * kLog2e;
    const size_t stride = (size_t)a.batch * a.h_q * kPartFloats;  // between chunks
    const float* base = part + ((size_t)b * a.h_q + h) * kPartFloats;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    if (valid) {
        if (lane < a.nsplit) {
            m0 = __ldcg(base + lane * stride);
            l0 = __ldcg(base + lane * stride + 1);
        }
        if (lane + 32 < a.nsplit) {
            m1 = __ldcg(base + (lane + 32) * stride);
            l1 = __ldcg(base + (lane + 32) * stride + 1);
        }
    }
    const float M = fmaxf(sink, warp_max(fmaxf(m0, m1)));
    // an empty chunk (m = -inf), or every term at -inf, weighs nothing
    const float w0 = m0 == -INFINITY ? 0.f : exp2f(m0 - M);
    const float w1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M);
    const float lsum = warp_sum(l0 * w0 + l1 * w1) + (M == -INFINITY ? 0.f : exp2f(sink - M));
    // every chunk's o is written (0 for an empty chunk), so the loads need no
    // guard and stay independent of each other
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 8
    for (int c = 0; c < a.nsplit; ++c) {
        const float wc = __shfl_sync(0xffffffffu, c < 32 ? w0 : w1, c & 31);
        const float2 oc = __ldcg(reinterpret_cast<const float2*>(base + c * stride + 2 + 2 * lane));
        acc0 = fmaf(oc.x, wc, acc0);
        acc1 = fmaf(oc.y, wc, acc1);
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

// ---------------------------------------------------------------- tensor-core split kernel
namespace mmadec {
constexpr int kWarps = 4;
constexpr int kKeys = 32;                     // keys per stage: one TMA box of K and one of V
constexpr int kSlots = 2;                     // stages in flight per warp
constexpr int kBoxBytes = kKeys * kD * 2;     // 4 KB, rows of 128 bytes
constexpr int kStageBytes = 2 * kBoxBytes;
constexpr int kSlotArea = kWarps * kSlots * kStageBytes;
constexpr size_t kSmemBytes = 1024 + kSlotArea + 128;  // alignment slack, slots, barriers + abort word
constexpr int kMB = kKeys / 16;               // 16-key row blocks per stage

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
// D += A B, A 16x16 (row), B 16x8 (col), bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
}  // namespace mmadec

// grid (nsplit, h_kv, batch), 128 threads; NB = ceil(g / 8) blocks of 8 query
// heads (heads past g are zero queries whose results are dropped). The last
// CTA of a (query, key/value head) to finish merges its chunks (a counter per
// pair, zero on entry, reset to zero by that CTA).
template <int NB>
__global__ void __launch_bounds__(mmadec::kWarps * 32)
decode_mma_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                  const __nv_bfloat16* __restrict__ q, const float* __restrict__ sinks,
                  const int32_t* __restrict__ kv_start, const int32_t* __restrict__ kv_len,
                  const DecodeArgs a, float* part, int32_t* counters,
                  __nv_bfloat16* __restrict__ o, float* __restrict__ lse, uint32_t* flags) {
    using namespace mmadec;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSlotArea);  // [kWarps][kSlots]
    volatile int* abort_word = reinterpret_cast<volatile int*>(full + kWarps * kSlots);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int gq = lane / 4, t4 = lane % 4;  // fragment row and column pair
    const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int g = a.group;
    const float c = a.scale_log2;

    int start = 0, lo = 0, len = 0;
    const bool valid = query_keys(a, kv_start, kv_len, b, start, lo, len);
    if (!valid && split == 0 && hk == 0 && threadIdx.x == 0) atomicOr(flags, kFlagSeqTooLong);
    int k_begin = 0, k_end = 0;
    if (valid) {
        const int n = len - lo;
        const int chunk = (n + a.nsplit - 1) / a.nsplit;
        k_begin = min(len, lo + split * chunk);
        k_end = min(len, k_begin + chunk);
    }
    const int nstage = (k_end - k_begin + kKeys - 1) / kKeys;
    const int mine = nstage > warp ? (nstage - warp + kWarps - 1) / kWarps : 0;

    if (threadIdx.x == 0) {
        for (int x = 0; x < kWarps * kSlots; ++x) tc::mbar_init(&full[x], 1);
        *abort_word = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();

    uint8_t* wslots = smem + warp * kSlots * kStageBytes;
    uint64_t* wfull = full + warp * kSlots;
    // own stage j (stage warp + 4 j of the chunk) into slot j % kSlots
    auto issue = [&](int j) {
        uint8_t* dst = wslots + (j % kSlots) * kStageBytes;
        uint64_t* bar = &wfull[j % kSlots];
        const int row = start + k_begin + (warp + j * kWarps) * kKeys;
        tc::mbar_arrive_expect_tx(bar, kStageBytes);
        tc::tma_load_3d(dst, &mk, bar, 0, hk, row);
        tc::tma_load_3d(dst + kBoxBytes, &mv, bar, 0, hk, row);
    };
    if (lane == 0)
        for (int j = 0; j < min(kSlots, mine); ++j) issue(j);

    // Q^T as the B operand of S^T = K Q^T: b0 = Q[head][d 2t4, 2t4+1], b1 = d + 8
    uint32_t qf[NB][4][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int n = nb * 8 + gq;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            qf[nb][ks][0] = qf[nb][ks][1] = 0u;
            if (n < g) {
                const __nv_bfloat16* qp = q + ((size_t)b * a.h_q + hk * g + n) * kD + ks * 16 + 2 * t4;
                qf[nb][ks][0] = __ldg(reinterpret_cast<const unsigned int*>(qp));
                qf[nb][ks][1] = __ldg(reinterpret_cast<const unsigned int*>(qp + 8));
            }
        }
    }

    // running state for heads 8 nb + 2 t4 (+1): max (raw score units), this
    // thread's share of the sum, and O^T fragments oacc[md][nb] (rows d = 16 md + gq, +8)
    float m_run[NB][2], l_run[NB][2], oacc[4][NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        m_run[nb][0] = m_run[nb][1] = -INFINITY;
        l_run[nb][0] = l_run[nb][1] = 0.f;
#pragma unroll
        for (int md = 0; md < 4; ++md) oacc[md][nb][0] = oacc[md][nb][1] = oacc[md][nb][2] = oacc[md][nb][3] = 0.f;
    }

    int done = 0;  // own stages consumed
    for (; done < mine; ++done) {
        const int slot = done % kSlots;
        if (!tc::wait_phase(&wfull[slot], (done / kSlots) & 1, flags, abort_word, a.wait_ns)) break;
        const int nk = min(kKeys, k_end - (k_begin + (warp + done * kWarps) * kKeys));
        uint8_t* kbox = wslots + slot * kStageBytes;
        const uint32_t kb = tc::smem_u32(kbox), vb = kb + kBoxBytes;
        if (nk < kKeys) {
            // rows past the chunk hold another context's values (or anything): zero V there
            uint4* vrows = reinterpret_cast<uint4*>(kbox + kBoxBytes);
            for (int x = nk * 8 + lane; x < kKeys * 8; x += 32) vrows[x] = make_uint4(0u, 0u, 0u, 0u);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
        }
        // S^T: rows = keys 16 mb + gq (+8), columns = heads 8 nb + 2 t4 (+1)
        float s[kMB][NB][4];
#pragma unroll
        for (int mb = 0; mb < kMB; ++mb)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) s[mb][nb][0] = s[mb][nb][1] = s[mb][nb][2] = s[mb][nb][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int mb = 0; mb < kMB; ++mb) {
                uint32_t af[4];
                ldsm_x4(af, kb + swz(mb * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, ks * 2 + (lane >> 4)));
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) mma16816(s[mb][nb], af, qf[nb][ks][0], qf[nb][ks][1]);
            }
        }
        if (nk < kKeys) {
#pragma unroll
            for (int mb = 0; mb < kMB; ++mb)
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    if (mb * 16 + gq >= nk) s[mb][nb][0] = s[mb][nb][1] = -INFINITY;
                    if (mb * 16 + gq + 8 >= nk) s[mb][nb][2] = s[mb][nb][3] = -INFINITY;
                }
        }
        // online softmax per head over this stage's keys
        uint32_t pb[kMB][NB][2];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int mb = 0; mb < kMB; ++mb) {
                mx0 = fmaxf(mx0, fmaxf(s[mb][nb][0], s[mb][nb][2]));
                mx1 = fmaxf(mx1, fmaxf(s[mb][nb][1], s[mb][nb][3]));
            }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            // the stage has at least one key of the chunk, so the new max is finite
            const float mn0 = fmaxf(m_run[nb][0], mx0), mn1 = fmaxf(m_run[nb][1], mx1);
            const float corr0 = fast_exp2((m_run[nb][0] - mn0) * c);
            const float corr1 = fast_exp2((m_run[nb][1] - mn1) * c);
            m_run[nb][0] = mn0;
            m_run[nb][1] = mn1;
            const float neg0 = -mn0 * c, neg1 = -mn1 * c;
            float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
            for (int mb = 0; mb < kMB; ++mb) {
                const float p0 = fast_exp2(fmaf(s[mb][nb][0], c, neg0));
                const float p1 = fast_exp2(fmaf(s[mb][nb][1], c, neg1));
                const float p2 = fast_exp2(fmaf(s[mb][nb][2], c, neg0));
                const float p3 = fast_exp2(fmaf(s[mb][nb][3], c, neg1));
                ps0 += p0 + p2;
                ps1 += p1 + p3;
                // P^T fragment for keys 16 mb .. +15: transpose the two 8x8 halves
                pb[mb][nb][0] = transpose8x8(pack_bf16(p0, p1));
                pb[mb][nb][1] = transpose8x8(pack_bf16(p2, p3));
            }
            l_run[nb][0] = fmaf(l_run[nb][0], corr0, ps0);
            l_run[nb][1] = fmaf(l_run[nb][1], corr1, ps1);
#pragma unroll
            for (int md = 0; md < 4; ++md) {
                oacc[md][nb][0] *= corr0;
                oacc[md][nb][1] *= corr1;
                oacc[md][nb][2] *= corr0;
                oacc[md][nb][3] *= corr1;
            }
        }
        // O^T += V^T P^T
#pragma unroll
        for (int mb = 0; mb < kMB; ++mb) {
#pragma unroll
            for (int md = 0; md < 4; ++md) {
                uint32_t af[4];
                ldsm_x4_trans(af, vb + swz(mb * 16 + (lane & 7) + (lane >> 4) * 8, md * 2 + ((lane >> 3) & 1)));
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) mma16816(oacc[md][nb], af, pb[mb][nb][0], pb[mb][nb][1]);
            }
        }
        __syncwarp();  // every lane's reads of the slot are done before it is refilled
        if (lane == 0 && done + kSlots < mine) issue(done + kSlots);
    }
    // after a timeout: let the copies still in flight land before the CTA leaves
    if (done < mine && lane == 0)
        for (int j = done; j < min(mine, done + kSlots); ++j) tc::drain_phase(&wfull[j % kSlots], (j / kSlots) & 1, a.wait_ns);

#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l_run[nb][0] += __shfl_xor_sync(0xffffffffu, l_run[nb][0], off);
            l_run[nb][1] += __shfl_xor_sync(0xffffffffu, l_run[nb][1], off);
        }
    __syncthreads();  // every warp is done with its slots: reuse them for the merge
    constexpr int kH = NB * 8;
    float* X = reinterpret_cast<float*>(smem);  // [kWarps][kH][2 + 64]: m, l, o
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        float* x0 = X + (warp * kH + nb * 8 + 2 * t4) * kPartFloats;
        float* x1 = x0 + kPartFloats;
        if (gq == 0) {
            x0[0] = m_run[nb][0];
            x0[1] = l_run[nb][0];
            x1[0] = m_run[nb][1];
            x1[1] = l_run[nb][1];
        }
#pragma unroll
        for (int md = 0; md < 4; ++md) {
            x0[2 + md * 16 + gq] = oacc[md][nb][0];
            x1[2 + md * 16 + gq] = oacc[md][nb][1];
            x0[2 + md * 16 + gq + 8] = oacc[md][nb][2];
            x1[2 + md * 16 + gq + 8] = oacc[md][nb][3];
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < g * kD; idx += kWarps * 32) {
        const int h = idx / kD, d = idx % kD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, X[(w * kH + h) * kPartFloats]);
        float lsum = 0.f, acc = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float* xw = X + (w * kH + h) * kPartFloats;
                if (xw[0] == -INFINITY) continue;  // a warp with no keys
                const float wgt = exp2f((xw[0] - M) * c);
                lsum = fmaf(xw[1], wgt, lsum);
                acc = fmaf(xw[2 + d], wgt, acc);
            }
        }
        float* pp = part + (((size_t)split * a.batch + b) * a.h_q + hk * g + h) * kPartFloats;
        pp[2 + d] = acc;
        if (d == 0) {
            pp[0] = M == -INFINITY ? -INFINITY : M * c;  // log2 units, as the merge expects
            pp[1] = lsum;
        }
    }
    // publish this chunk; the last of the pair's nsplit CTAs merges them all
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *abort_word = atomicAdd(counters + (size_t)b * a.h_kv + hk, 1) == a.nsplit - 1 ? 2 : 3;
    __syncthreads();
    if (*abort_word != 2) return;
    __threadfence();
    // merge of the pair's chunks for its g heads: maxima and sums staged in
    // shared memory in one pass, weights per head, then every (head, column
    // pair) sums the chunks' outputs with independent loads
    const int ns = a.nsplit;
    const size_t stride = (size_t)a.batch * a.h_q * kPartFloats;       // between chunks
    const float* pbase = part + ((size_t)b * a.h_q + hk * g) * kPartFloats;  // chunk 0, first head
    float* mw = reinterpret_cast<float*>(smem);  // [g][ns] chunk max, then its weight
    float* ls = mw + g * ns;                      // [g][ns] chunk sum
    float* hinv = ls + g * ns;                    // [g] 1 / l
    for (int idx = threadIdx.x; idx < g * ns; idx += kWarps * 32) {
        const float* pp = pbase + (idx % ns) * stride + (idx / ns) * kPartFloats;
        mw[idx] = valid ? __ldcg(pp) : -INFINITY;
        ls[idx] = valid ? __ldcg(pp + 1) : 0.f;
    }
    __syncthreads();
    if (threadIdx.x < g) {
        const int h = threadIdx.x;
        const float sink = __ldg(sinks + hk * g + h) * kLog2e;
        float M = sink;
        for (int cc = 0; cc < ns; ++cc) M = fmaxf(M, mw[h * ns + cc]);
        float lsum = M == -INFINITY ? 0.f : exp2f(sink - M);
        for (int cc = 0; cc < ns; ++cc) {
            const float mc = mw[h * ns + cc];
            const float wgt = mc == -INFINITY ? 0.f : exp2f(mc - M);  // an empty chunk weighs nothing
            mw[h * ns + cc] = wgt;
            lsum = fmaf(ls[h * ns + cc], wgt, lsum);
        }
        hinv[h] = lsum > 0.f ? 1.f / lsum : 0.f;
        lse[(size_t)(hk * g + h) * a.batch + b] = lsum > 0.f ? (M + log2f(lsum)) * kLn2 : -INFINITY;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < g * 32; idx += kWarps * 32) {
        const int h = idx / 32, cp = idx % 32;
        const float* pp = pbase + h * kPartFloats + 2 + 2 * cp;
        const float* wv = mw + h * ns;
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 8
        for (int cc = 0; cc < ns; ++cc) {
            const float2 oc = __ldcg(reinterpret_cast<const float2*>(pp + cc * stride));
            acc0 = fmaf(oc.x, wv[cc], acc0);
            acc1 = fmaf(oc.y, wv[cc], acc1);
        }
        const float inv = hinv[h];
        *reinterpret_cast<__nv_bfloat162*>(o + ((size_t)b * a.h_q + hk * g + h) * kD + 2 * cp) =
            __floats2bfloat162_rn(acc0 * inv, acc1 * inv);
    }
    if (threadIdx.x == 0) counters[(size_t)b * a.h_kv + hk] = 0;
}

// One warp per (query, head): launched over every pair by the CUDA-core path.
template <typename T>
__global__ void __launch_bounds__(kThreads)
decode_merge_kernel(const float* __restrict__ part, const float* __restrict__ sinks,
                    const int32_t* __restrict__ kv_start, const int32_t* __restrict__ kv_len,
                    const DecodeArgs a, T* __restrict__ o, float* __restrict__ lse) {
    const int wid = blockIdx.x * (kThreads / 32) + threadIdx.x / 32;
    if (wid >= a.batch * a.h_q) return;
    const int b = wid / a.h_q, h = wid % a.h_q;
    int start, lo, len;
    const bool valid = query_keys(a, kv_start, kv_len, b, start, lo, len);
    merge_head<T>(part, sinks, a, b, h, valid, o, lse, threadIdx.x % 32);
}

template <typename T>
cudaError_t launch_merge(const DecodeArgs& a, const float* sinks, const int32_t* kv_start,
                         const int32_t* kv_len, void* o, float* lse, const float* part,
                         cudaStream_t st) {
    const int warps = a.batch * a.h_q;
    decode_merge_kernel<T><<<(warps + kThreads / 32 - 1) / (kThreads / 32), kThreads, 0, st>>>(
        part, sinks, kv_start, kv_len, a, (T*)o, lse);
    count_launches(1);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_simt(const DecodeArgs& a, const void* q, const void* k, const void* v,
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
    return launch_merge<T>(a, sinks, kv_start, kv_len, o, lse, part, st);
}

// Split count for the tensor-core kernel. CTAs come in waves of (SMs x CTAs
// per SM), and every wave pays a pipeline fill at its start and the partial
// write and merge at its end, so a single wave that fills at least 90% of the
// slots is best; otherwise the fewest splits that give at least two waves
// with the last one at least 97% full (else the fullest last wave). Each
// chunk keeps at least two stages per warp.
int mma_splits(int pairs, int keys, int slots) {
    using namespace mmadec;
    const int cap = std::max(1, std::min(kDecodeMaxSplits, keys / (kKeys * kWarps * 2)));
    for (int ns = cap; ns >= 1; --ns) {
        const long ctas = (long)pairs * ns;
        if (ctas <= slots && 10 * ctas >= 9L * slots) return ns;
    }
    int best = 1;
    double best_eff = -1.0;
    for (int ns = 1; ns <= cap; ++ns) {
        const long ctas = (long)pairs * ns;
        const long waves = (ctas + slots - 1) / slots;
        const double eff = (double)ctas / (double)(waves * slots);
        if (ctas >= 2L * slots && eff >= 0.97) return ns;
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = ns;
        }
    }
    return best;
}

template <int NB>
cudaError_t launch_mma(DecodeArgs a, const void* q, const void* k, const void* v,
                       const float* sinks, const int32_t* kv_start, const int32_t* kv_len, void* o,
                       float* lse, float* part, int32_t* counters, uint32_t* flags, cudaStream_t st) {
    using namespace mmadec;
    CUtensorMap mk, mv;
    if (!make_head_tile_map(&mk, k, a.total, a.h_kv, kKeys) ||
        !make_head_tile_map(&mv, v, a.total, a.h_kv, kKeys))
        return cudaErrorInvalidValue;
    static int sms[64] = {0}, per_sm[64] = {0};  // per device, filled on first use
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (sms[dev] == 0) {
        e = cudaFuncSetAttribute(decode_mma_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        int n = 0, r = 0;
        if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, decode_mma_kernel<NB>, kWarps * 32,
                                                                kSmemBytes)) != cudaSuccess)
            return e;
        per_sm[dev] = std::max(1, r);
        sms[dev] = std::max(1, n);
    }
    const int keys = a.window > 0 ? std::min(a.window, a.max_len) : a.max_len;
    a.nsplit = mma_splits(a.batch * a.h_kv, keys, sms[dev] * per_sm[dev]);
    dim3 grid(a.nsplit, a.h_kv, a.batch);
    decode_mma_kernel<NB><<<grid, kWarps * 32, kSmemBytes, st>>>(
        mk, mv, (const __nv_bfloat16*)q, sinks, kv_start, kv_len, a, part, counters,
        (__nv_bfloat16*)o, lse, flags);
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
                   float* lse, float* part, int32_t* counters, uint32_t* flags, cudaStream_t st) {
    if (a.batch == 0) return cudaSuccess;
    if (bf16 && a.total > 0 && a.group <= 16) {
        return a.group <= 8
                   ? launch_mma<1>(a, q, k, v, sinks, kv_start, kv_len, o, lse, part, counters, flags, st)
                   : launch_mma<2>(a, q, k, v, sinks, kv_start, kv_len, o, lse, part, counters, flags, st);
    }
    return bf16 ? launch_simt<__nv_bfloat16>(a, q, k, v, sinks, kv_start, kv_len, o, lse, part, flags, st)
                : launch_simt<float>(a, q, k, v, sinks, kv_start, kv_len, o, lse, part, flags, st);
}

}  // namespace sinkattn
