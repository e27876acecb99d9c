// common.cuh - problem descriptor and small device helpers shared by the
// kernels of libsinkattn (sink attention for sm_103a).
//
// Masks follow the C ABI in include/sink_attn.h: per sequence, positions are
// counted from the sequence start; row i sees keys [lo(i), hi(i)) with
//   causal = 0: [0, L)        causal = 1: [0, i+1)       window W: [max(0, i-W+1), i+1).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sinkattn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device flag bits written into the first word of the workspace.
constexpr uint32_t kFlagTimeout = 1u << 0;    // a bounded wait gave up
constexpr uint32_t kFlagSeqTooLong = 1u << 1;  // a sequence longer than max_seqlen
constexpr uint32_t kFlagBadSeqlens = 1u << 2;  // cu_seqlens is not a non-decreasing run from 0 within T

// Limit of every bounded wait in the tensor-core kernels.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s

struct Problem {
    int nseq;          // number of sequences
    int max_seqlen;    // grid bound on a sequence's length
    int total;         // T
    int h_q, h_kv, group;  // group = h_q / h_kv
    int head_dim;
    int causal, window;
    float scale;       // softmax scale on Q.K
    float scale_log2;  // scale * log2(e): scores in base-2 units
    const int32_t* cu; // device cu_seqlens or nullptr (padded: sequence s = [s*N, s*N+N))
    uint64_t wait_ns;  // limit of each bounded wait (kDefaultWaitNs unless a test lowers it)
    int withhold_load; // test hook: the forward / backward producer stops after its first stage
    int deterministic; // backward: dQ without reduce-adds (the split 64-wide backward)
};

// Decode (one query per entry against a key/value cache), see decode.cu.
constexpr int kDecodeMaxSplits = 64;
struct DecodeArgs {
    int batch;        // queries
    int h_q, h_kv, group;
    int total;        // rows of the cache
    int max_len;      // upper bound on every kv_len
    int window;       // <= 0: whole context; W: its last W keys
    int nsplit;       // chunks of each query's keys
    float scale_log2;
    uint64_t wait_ns; // limit of each bounded wait
};

// Bounds of sequence s, checked: with packed sequences, cu_seqlens comes from
// device memory that the host never reads, so a CTA verifies
// 0 <= cu[s] <= cu[s+1] <= total (and cu[0] == 0 for s = 0) before it touches
// any row. A CTA whose sequence fails returns false and raises
// kFlagBadSeqlens; it must then return before any load, store or barrier.
__device__ __forceinline__ bool seq_bounds_checked(const Problem& P, int s, int& start, int& len,
                                                   uint32_t* flags) {
    if (!P.cu) {
        start = s * P.max_seqlen;
        len = P.max_seqlen;
        return true;
    }
    const int a = __ldg(P.cu + s), b = __ldg(P.cu + s + 1);
    if (a < 0 || b < a || b > P.total || (s == 0 && a != 0)) {
        if (threadIdx.x == 0) atomicOr(flags, kFlagBadSeqlens);
        start = 0;
        len = 0;
        return false;
    }
    start = a;
    len = b - a;
    return true;
}

// This block's (x, y, z) for a grid of (row or key blocks, heads, sequences),
// read from the linear launch index with z (the sequence) slowest, then
// groups of G heads (G = 4 when the head count allows), then x, then the head
// within its group fastest. Blocks are dispatched roughly in linear-index
// order with x fastest; under a causal mask a block's work depends on its x,
// and with x fastest every (head, sequence) slice ran long-to-short in turn,
// so the last slice's longest blocks started late and most SMs idled while
// they finished. With a few heads innermost, the blocks of one sequence run
// longest-first and the last blocks to start are short; grouping the heads
// keeps the Q / dO rows and dQ accumulator lines that run at the same time to
// a part of the sequence's heads, so more of them stay in L2 (an order with x
// slowest over every sequence and head spread that set over all of them).
struct BlockCoord {
    int x, y, z;
};
__device__ __forceinline__ BlockCoord block_seq_x_head() {
    const unsigned lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    const unsigned X = gridDim.x, Y = gridDim.y;
    const unsigned G = Y <= 4 ? Y : (Y % 4 == 0 ? 4 : (Y % 2 == 0 ? 2 : 1));
    const unsigned xy = X * Y;
    const unsigned r = lin % xy;
    const unsigned g = r / (G * X), r2 = r % (G * X);
    return BlockCoord{(int)(r2 / G), (int)(g * G + r2 % G), (int)(lin / xy)};
}

// Programmatic dependent launch. A kernel launched by launch_after() may begin
// while the kernel before it in the stream is finishing (its CTAs take the SMs
// that kernel's last wave leaves, and do their set-up); it calls pdl_wait()
// before it reads anything that kernel wrote, which returns once that kernel
// has completed and its writes are visible (at once in a normal launch). A
// kernel calls pdl_trigger() when the next kernel may be scheduled: every
// kernel that calls it does so as soon as its CTAs start. Only kernels
// launched back to back inside one library call are launched this way, so
// the kernel before one is always this library's.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// First allowed key of row i.
__device__ __forceinline__ int key_lo(const Problem& P, int i) {
    if (!P.causal) return 0;
    if (P.window > 0) return i - P.window + 1 > 0 ? i - P.window + 1 : 0;
    return 0;
}

// One past the last allowed key of row i in a sequence of length L.
__device__ __forceinline__ int key_hi(const Problem& P, int i, int L) {
    return P.causal ? i + 1 : L;
}

// One past the last row that sees key j (sequence length L).
__device__ __forceinline__ int row_hi(const Problem& P, int j, int L) {
    if (P.causal && P.window > 0) return j + P.window < L ? j + P.window : L;
    return L;
}

// First row that sees key j.
__device__ __forceinline__ int row_lo(const Problem& P, int j) {
    return P.causal ? j : 0;
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace sinkattn
