// tc_bwd128.cu - sink-attention backward for 128-wide heads on the sm_103a
// tensor cores.
//
// What it computes (page "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、超稳定！",
// section "反向传播的实现"), with LSE (sink included) from the forward and
// delta_i = dO_i . O_i from the preprocess step:
//   P_ij = exp(S_ij - LSE_i)     dP_ij = dO_i . V_j     dS_ij = P_ij (dP_ij - delta_i)
//   dQ_i = scale sum_j dS_ij K_j      dK_j = scale sum_i dS_ij Q_i      dV_j = sum_i P_ij dO_i
// (the sink's own gradient comes from the preprocess step).
//
// At d = 128 the 64-wide design (one key block holding S, dP, dK, dV, dQ, K,
// V, P and dS in tensor memory) would need 768 of the 512 columns, so the
// work is split in two kernels that each fit:
//
// bwd128_dq_kernel: one CTA = 128 query rows of one head, walking the key
//   blocks that the rows see. Thread r of the first four warps owns row r
//   (tensor-memory lane r), so LSE_r and delta_r are per-thread constants.
//     S  = Q K^T    A = Q  (tensor memory, written once by the row threads)  TS
//     dP = dO V^T   A = dO (shared memory, loaded once)                       SS
//     dQ += dS K    A = dS (tensor memory, from the row threads), B = K MN-major
//   Tensor memory: S 0..127, dP 128..255, dQ 256..383, dS 384..447, Q 448..511.
//
// bwd128_dkdv_kernel: one CTA = 128 keys of one key/value head, walking every
//   (query head of the group, query block) that sees them. Thread = key; the
//   two warpgroups of elementwise warps split the 128 query rows of a step.
//     S^T  = K Q^T    A = K (shared memory, loaded once)   SS
//     dP^T = V dO^T   A = V (shared memory, loaded once)   SS, over S^T once it has been read
//     dV  += P^T dO   A = P^T  (tensor memory), B = dO MN-major
//     dK  += dS^T Q   A = dS^T (tensor memory), B = Q  MN-major
//   The step's LSE and delta rows are staged in shared memory by the producer
//   warp. Tensor memory: S^T/dP^T 0..127, dV 128..255, dK 256..383, P^T
//   384..447, dS^T 448..511.
//
// Tiles of 128 rows x 128 columns are two 128-byte-swizzled atoms of 64
// columns, each filled by its own TMA box. A K-major operand steps through the
// atoms along K; an MN-major operand (N = 128) spans both, 16 KB apart (the
// descriptor's leading byte offset). dQ, dK and dV are written once, in bf16,
// with no atomics. Every mbarrier wait is bounded.
#include <cudaTypedefs.h>

#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tc.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace sinkattn {
namespace {

using namespace tc;

constexpr int kB = 128;                         // rows per query block = keys per key block
constexpr int kD = 128;                         // head dim
constexpr int kAtomCols = 64;                   // columns per 128-byte swizzle atom
constexpr uint32_t kAtomBytes = kB * kAtomCols * 2;  // 16 KB
constexpr uint32_t kTileBytes = kB * kD * 2;         // 32 KB
constexpr uint32_t kSPanel = (uint32_t)(kAtomBytes >> 4);  // atom step in descriptor units

// K step kk (16 columns of d) of a K-major operand: atom kk / 4, 32-byte
// offset kk % 4, both added to the descriptor's start-address field.
__device__ __forceinline__ uint64_t kstep_off(int kk) {
    return (uint64_t)((kk / 4) * kSPanel + 2 * (kk % 4));
}
// K step kk (16 rows) of an MN-major operand in atom a: 16 rows x 128 bytes.
__device__ __forceinline__ uint64_t mnstep_off(int a, int kk) {
    return (uint64_t)(a * kSPanel + ((kk * 16 * 128) >> 4));
}

// ---------------------------------------------------------------- dQ kernel
constexpr int kAStages = 3;
constexpr int kAThreads = 192;  // 4 row warps, producer, MMA issuer
constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 384, kColQ = 448;

struct DqSmem {
    alignas(1024) __nv_bfloat16 dout[kB * kD];
    alignas(1024) __nv_bfloat16 k[kAStages][kB * kD];
    alignas(1024) __nv_bfloat16 v[kAStages][kB * kD];
    uint64_t do_full, q_ready;
    uint64_t k_full[kAStages], v_full[kAStages], kv_empty[kAStages];
    uint64_t s_full, s_loaded, dp_full, dp_loaded, ds_full, dq_done, drained;
    uint32_t tmem_slot;
    int abort_flag;
};
static_assert(sizeof(DqSmem) + 1024 <= 232448, "dQ kernel shared memory");

__global__ void __launch_bounds__(kAThreads, 1)
bwd128_dq_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmDO, const Problem P,
                 const __nv_bfloat16* __restrict__ q, const float* __restrict__ lse,
                 const float* __restrict__ delta, __nv_bfloat16* __restrict__ dq, uint32_t* flags) {
    extern __shared__ uint8_t smem_raw[];
    DqSmem& sm = *reinterpret_cast<DqSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~uintptr_t(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const BlockCoord bc = block_seq_x_head();
    const int rb = gridDim.x - 1 - bc.x;  // longest row blocks first
    const int h = bc.y, seq = bc.z;
    int start, L;
    if (!seq_bounds_checked(P, seq, start, L, flags)) return;
    const int r0 = rb * kB;
    if (r0 >= L) return;  // uniform for the CTA, before any barrier or tensor memory
    int kb_lo = 0, kb_hi = (L - 1) / kB;
    if (P.causal) {
        kb_hi = rb;
        if (P.window > 0) kb_lo = max(0, r0 - P.window + 1) / kB;
    }
    const int nblk = kb_hi - kb_lo + 1;
    const int hk = h / P.group;

    if (threadIdx.x == 0) {
        mbar_init(&sm.do_full, 1);
        mbar_init(&sm.q_ready, 128);
        for (int i = 0; i < kAStages; ++i) {
            mbar_init(&sm.k_full[i], 1);
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.kv_empty[i], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_loaded, 128);
        mbar_init(&sm.dp_full, 1);
        mbar_init(&sm.dp_loaded, 128);
        mbar_init(&sm.ds_full, 128);
        mbar_init(&sm.dq_done, 1);
        mbar_init(&sm.drained, 1);
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc<512>(&sm.tmem_slot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_slot;
    volatile int* abort_word = &sm.abort_flag;

    if (warp < 4) {
        // ------------------------------------------------------------ row threads
        const int r = warp * 32 + lane;
        const int row = r0 + r;
        const bool valid = row < L;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        {
            // Q row into tensor memory: the A operand of S = Q K^T
            uint32_t qw[64];
            const uint4* src = reinterpret_cast<const uint4*>(
                q + ((size_t)(start + (valid ? row : r0)) * P.h_q + h) * kD);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint4 x = valid ? __ldg(src + j) : make_uint4(0u, 0u, 0u, 0u);
                qw[4 * j] = x.x;
                qw[4 * j + 1] = x.y;
                qw[4 * j + 2] = x.z;
                qw[4 * j + 3] = x.w;
            }
            tmem_st64(tmem + lane_off + kColQ, qw);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.q_ready);
        }
        const float sc = P.scale_log2;
        const size_t rix = (size_t)h * P.total + start + (valid ? row : r0);
        const float lse2 = valid ? __ldg(lse + rix) * kLog2e : 0.f;
        const float dlt = valid ? __ldg(delta + rix) : 0.f;
        const uint64_t sc2 = f2_pack(sc, sc);
        const uint64_t nl2 = f2_pack(-lse2, -lse2);
        const int lo = P.causal && P.window > 0 ? row - P.window + 1 : INT_MIN;
        const int hi = P.causal ? min(row, L - 1) : L - 1;
        bool ok = true;
        for (int i = 0; i < nblk; ++i) {
            ok = __all_sync(0xffffffffu, wait_phase(&sm.s_full, i & 1, flags, abort_word, P.wait_ns));
            if (!ok) break;
            tc_fence_after();
            float p[128];
            {
                uint32_t a[128];
                tmem_ld128(tmem + lane_off + kColS, a);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&sm.s_loaded);  // the next block's S may be issued
#pragma unroll
                for (int j = 0; j < 128; ++j) p[j] = __uint_as_float(a[j]);
            }
            const int kp0 = (kb_lo + i) * kB;
            const bool need_mask = P.causal ? (kp0 + kB - 1 > r0 || (P.window > 0 && kp0 < r0 + kB - P.window))
                                            : (kp0 + kB > L);
            if (need_mask) {
#pragma unroll
                for (int j = 0; j < 128; ++j) {
                    const int kp = kp0 + j;
                    if (kp < lo || kp > hi) p[j] = -INFINITY;
                }
            }
            // P = exp2(S * scale * log2 e - LSE * log2 e)
#pragma unroll
            for (int j = 0; j < 128; j += 2) {
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(p[j], p[j + 1]), sc2, nl2), x0, x1);
                p[j] = fast_exp2(x0);
                p[j + 1] = fast_exp2(x1);
            }
            ok = __all_sync(0xffffffffu, wait_phase(&sm.dp_full, i & 1, flags, abort_word, P.wait_ns));
            if (!ok) break;
            tc_fence_after();
            uint32_t dsw[64];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t d[64];
                tmem_ld64(tmem + lane_off + kColDP + half * 64, d);
                tmem_ld_wait();
                if (half == 1) {
                    tc_fence_before();
                    mbar_arrive(&sm.dp_loaded);  // the next block's dP may be issued
                }
#pragma unroll
                for (int j = 0; j < 64; j += 2) {
                    const float ds0 = p[half * 64 + j] * (__uint_as_float(d[j]) - dlt);
                    const float ds1 = p[half * 64 + j + 1] * (__uint_as_float(d[j + 1]) - dlt);
                    dsw[half * 32 + j / 2] = pack_bf16x2(ds0, ds1);
                }
            }
            if (i > 0) {
                // dQ of the previous block has read the dS columns
                ok = __all_sync(0xffffffffu, wait_phase(&sm.dq_done, (i - 1) & 1, flags, abort_word, P.wait_ns));
                if (!ok) break;
                tc_fence_after();
            }
            tmem_st64(tmem + lane_off + kColDS, dsw);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.ds_full);
        }
        if (ok) ok = __all_sync(0xffffffffu, wait_phase(&sm.dq_done, (nblk - 1) & 1, flags, abort_word, P.wait_ns));
        if (ok) {
            tc_fence_after();
            uint4* dst = reinterpret_cast<uint4*>(dq + ((size_t)(start + row) * P.h_q + h) * kD);
            const float s = P.scale;
#pragma unroll
            for (int c0 = 0; c0 < kD; c0 += 64) {
                uint32_t a[64];
                tmem_ld64(tmem + lane_off + kColDQ + c0, a);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(a[8 * j + 0]) * s, __uint_as_float(a[8 * j + 1]) * s);
                        w.y = pack_bf16x2(__uint_as_float(a[8 * j + 2]) * s, __uint_as_float(a[8 * j + 3]) * s);
                        w.z = pack_bf16x2(__uint_as_float(a[8 * j + 4]) * s, __uint_as_float(a[8 * j + 5]) * s);
                        w.w = pack_bf16x2(__uint_as_float(a[8 * j + 6]) * s, __uint_as_float(a[8 * j + 7]) * s);
                        dst[c0 / 8 + j] = w;
                    }
                }
            }
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmDO);
            mbar_arrive_expect_tx(&sm.do_full, kTileBytes);
            for (int a = 0; a < 2; ++a)
                tma_load_3d(sm.dout + a * kB * kAtomCols, &tmDO, &sm.do_full, a * kAtomCols, h, start + r0);
            int issued = 0;
            for (int i = 0; i < nblk; ++i) {
                const int st = i % kAStages;
                if (i >= kAStages &&
                    !wait_phase(&sm.kv_empty[st], ((i / kAStages) - 1) & 1, flags, abort_word, P.wait_ns))
                    break;
                const int kpos = start + (kb_lo + i) * kB;
                mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
                for (int a = 0; a < 2; ++a)
                    tma_load_3d(sm.k[st] + a * kB * kAtomCols, &tmK, &sm.k_full[st], a * kAtomCols, hk, kpos);
                mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
                for (int a = 0; a < 2; ++a)
                    tma_load_3d(sm.v[st] + a * kB * kAtomCols, &tmV, &sm.v_full[st], a * kAtomCols, hk, kpos);
                issued = i + 1;
            }
            // copies still in flight must land before the CTA's shared memory goes away
            drain_phase(&sm.do_full, 0, P.wait_ns);
            for (int i = max(0, issued - kAStages); i < issued; ++i) {
                const int st = i % kAStages;
                drain_phase(&sm.k_full[st], (i / kAStages) & 1, P.wait_ns);
                drain_phase(&sm.v_full[st], (i / kAStages) & 1, P.wait_ns);
            }
        }
    } else if (lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idSq = idesc_bf16(kB, kB, 0, 0);         // S, dP: B K-major
        constexpr uint32_t idQ = idesc_bf16(kB, kD, 0, 1);          // dQ: B = K MN-major, N = 128
        const uint64_t ddo = smem_desc_sw128(smem_u32(sm.dout), 16, 1024);
        auto s_product = [&](int st) {
            const uint64_t dk = smem_desc_sw128(smem_u32(sm.k[st]), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
                mma_ts(tmem + kColS, tmem + kColQ + kk * 8, dk + kstep_off(kk), idSq, kk > 0);
        };
        auto dp_product = [&](int st) {
            const uint64_t dv = smem_desc_sw128(smem_u32(sm.v[st]), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
                mma_ss(tmem + kColDP, ddo + kstep_off(kk), dv + kstep_off(kk), idSq, kk > 0);
        };
        auto dq_product = [&](int st, bool acc) {
            const uint64_t dk = smem_desc_sw128(smem_u32(sm.k[st]), kAtomBytes, 1024);
#pragma unroll
            for (int kk = 0; kk < kB / 16; ++kk)
                mma_ts(tmem + kColDQ, tmem + kColDS + kk * 8, dk + mnstep_off(0, kk), idQ, acc || kk > 0);
        };
        bool ok = wait_phase(&sm.q_ready, 0, flags, abort_word, P.wait_ns) &&
                  wait_phase(&sm.k_full[0], 0, flags, abort_word, P.wait_ns);
        if (ok) {
            tc_fence_after();
            s_product(0);
            mma_commit(&sm.s_full);
            ok = wait_phase(&sm.do_full, 0, flags, abort_word, P.wait_ns) &&
                 wait_phase(&sm.v_full[0], 0, flags, abort_word, P.wait_ns);
        }
        if (ok) {
            tc_fence_after();
            dp_product(0);
            mma_commit(&sm.dp_full);
        }
        for (int i = 0; ok && i < nblk; ++i) {
            const int st = i % kAStages, st1 = (i + 1) % kAStages;
            if (i + 1 < nblk) {
                // S(i+1) once S(i) is read, dP(i+1) once dP(i) is read: both ahead of dQ(i)
                if (!(ok = wait_phase(&sm.s_loaded, i & 1, flags, abort_word, P.wait_ns))) break;
                if (!(ok = wait_phase(&sm.k_full[st1], ((i + 1) / kAStages) & 1, flags, abort_word, P.wait_ns))) break;
                tc_fence_after();
                s_product(st1);
                mma_commit(&sm.s_full);
                if (!(ok = wait_phase(&sm.dp_loaded, i & 1, flags, abort_word, P.wait_ns))) break;
                if (!(ok = wait_phase(&sm.v_full[st1], ((i + 1) / kAStages) & 1, flags, abort_word, P.wait_ns))) break;
                tc_fence_after();
                dp_product(st1);
                mma_commit(&sm.dp_full);
            }
            if (!(ok = wait_phase(&sm.ds_full, i & 1, flags, abort_word, P.wait_ns))) break;
            tc_fence_after();
            dq_product(st, i > 0);
            mma_commit(&sm.dq_done);
            mma_commit(&sm.kv_empty[st]);  // K(i) and V(i) are no longer read
        }
        mma_commit(&sm.drained);
        drain_phase(&sm.drained, 0, P.wait_ns);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<512>(tmem);
    }
}

// ---------------------------------------------------------------- dK / dV kernel
constexpr int kBStages = 2;
constexpr int kBThreads = 320;  // 8 key warps, producer, MMA issuer
constexpr uint32_t kColSP = 0, kColDV = 128, kColDK = 256, kColPT = 384, kColDST = 448;

struct DkvSmem {
    alignas(1024) __nv_bfloat16 k[kB * kD];
    alignas(1024) __nv_bfloat16 v[kB * kD];
    alignas(1024) __nv_bfloat16 q[kBStages][kB * kD];
    alignas(1024) __nv_bfloat16 dout[kBStages][kB * kD];
    alignas(16) float lse2[kBStages][kB];  // LSE * log2 e of the step's rows (0 past the sequence)
    alignas(16) float dlt[kBStages][kB];   // delta of the step's rows
    uint64_t kv_full;
    uint64_t q_full[kBStages], q_empty[kBStages], rows_full[kBStages];
    uint64_t s_full, s_loaded, dp_full, dp_loaded, ds_full, pd_free, acc_done, drained;
    uint32_t tmem_slot;
    int abort_flag;
};
static_assert(sizeof(DkvSmem) + 1024 <= 232448, "dK/dV kernel shared memory");

__global__ void __launch_bounds__(kBThreads, 1)
bwd128_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                   const Problem P, const float* __restrict__ lse, const float* __restrict__ delta,
                   __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, uint32_t* flags) {
    extern __shared__ uint8_t smem_raw[];
    DkvSmem& sm = *reinterpret_cast<DkvSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const BlockCoord bc = block_seq_x_head();  // key block 0 (the longest) first
    const int kb = bc.x, hk = bc.y, seq = bc.z;
    int start, L;
    if (!seq_bounds_checked(P, seq, start, L, flags)) return;
    const int j0 = kb * kB;
    if (j0 >= L) return;  // uniform for the CTA
    // query blocks that see some key of this block
    int qb_lo = 0, qb_hi = (L - 1) / kB;
    if (P.causal) {
        qb_lo = kb;
        if (P.window > 0) qb_hi = min(qb_hi, (j0 + kB - 1 + P.window - 1) / kB);
    }
    const int nqb = qb_hi - qb_lo + 1;
    const int nsteps = P.group * nqb;

    if (threadIdx.x == 0) {
        mbar_init(&sm.kv_full, 1);
        for (int i = 0; i < kBStages; ++i) {
            mbar_init(&sm.q_full[i], 1);
            mbar_init(&sm.q_empty[i], 1);
            mbar_init(&sm.rows_full[i], 32);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_loaded, 256);
        mbar_init(&sm.dp_full, 1);
        mbar_init(&sm.dp_loaded, 256);
        mbar_init(&sm.ds_full, 256);
        mbar_init(&sm.pd_free, 1);
        mbar_init(&sm.acc_done, 1);
        mbar_init(&sm.drained, 1);
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc<512>(&sm.tmem_slot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_slot;
    volatile int* abort_word = &sm.abort_flag;

    if (warp < 8) {
        // ------------------------------------------------------------ key threads
        const int g = warp / 4;   // query rows [64 g, 64 g + 64) of each step
        const int wq = warp % 4;  // keys [32 wq, 32 wq + 32)
        const int key = j0 + wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const float sc = P.scale_log2;
        const uint64_t sc2 = f2_pack(sc, sc);
        bool ok = true;
        for (int i = 0; i < nsteps; ++i) {
            const int st = i % kBStages;
            const int qb = qb_lo + i % nqb;
            const int rbase = qb * kB + g * 64;  // first query row of this thread's columns
            ok = __all_sync(0xffffffffu, wait_phase(&sm.rows_full[st], (i / kBStages) & 1, flags, abort_word, P.wait_ns));
            if (!ok) break;
            ok = __all_sync(0xffffffffu, wait_phase(&sm.s_full, i & 1, flags, abort_word, P.wait_ns));
            if (!ok) break;
            tc_fence_after();
            float p[64];
            {
                uint32_t a[64];
                tmem_ld64(tmem + lane_off + kColSP + g * 64, a);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&sm.s_loaded);  // dP^T may be written over S^T
                // the rows' LSE as 16-byte broadcast loads (every lane reads the same row values)
                const float4* l4 = reinterpret_cast<const float4*>(sm.lse2[st] + g * 64);
#pragma unroll
                for (int c = 0; c < 64; c += 4) {
                    const float4 l = l4[c / 4];
                    float x0, x1, x2, x3;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(a[c]), __uint_as_float(a[c + 1])), sc2,
                                     f2_pack(-l.x, -l.y)),
                              x0, x1);
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(a[c + 2]), __uint_as_float(a[c + 3])), sc2,
                                     f2_pack(-l.z, -l.w)),
                              x2, x3);
                    p[c] = fast_exp2(x0);
                    p[c + 1] = fast_exp2(x1);
                    p[c + 2] = fast_exp2(x2);
                    p[c + 3] = fast_exp2(x3);
                }
            }
            // rows that do not see this key (causal diagonal block, window edge,
            // rows past the sequence end) take no part
            const bool need_mask = (P.causal && (rbase < j0 + kB ||
                                                 (P.window > 0 && rbase + 63 > j0 + P.window - 1))) ||
                                   rbase + 64 > L;
            if (need_mask) {
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const int row = rbase + c;
                    const bool seen = row < L && (!P.causal || (row >= key &&
                                                   (P.window <= 0 || row <= key + P.window - 1)));
                    if (!seen) p[c] = 0.f;
                }
            }
            ok = __all_sync(0xffffffffu, wait_phase(&sm.dp_full, i & 1, flags, abort_word, P.wait_ns));
            if (!ok) break;
            tc_fence_after();
            uint32_t pw[32], dw[32];
            {
                uint32_t d[64];
                tmem_ld64(tmem + lane_off + kColSP + g * 64, d);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&sm.dp_loaded);  // the next step's S^T may be issued
                const float4* d4 = reinterpret_cast<const float4*>(sm.dlt[st] + g * 64);
#pragma unroll
                for (int c = 0; c < 64; c += 4) {
                    const float4 dl = d4[c / 4];
                    pw[c / 2] = pack_bf16x2(p[c], p[c + 1]);
                    pw[c / 2 + 1] = pack_bf16x2(p[c + 2], p[c + 3]);
                    dw[c / 2] = pack_bf16x2(p[c] * (__uint_as_float(d[c]) - dl.x),
                                            p[c + 1] * (__uint_as_float(d[c + 1]) - dl.y));
                    dw[c / 2 + 1] = pack_bf16x2(p[c + 2] * (__uint_as_float(d[c + 2]) - dl.z),
                                                p[c + 3] * (__uint_as_float(d[c + 3]) - dl.w));
                }
            }
            if (i > 0) {
                // dV and dK of the previous step have read P^T and dS^T
                ok = __all_sync(0xffffffffu, wait_phase(&sm.pd_free, (i - 1) & 1, flags, abort_word, P.wait_ns));
                if (!ok) break;
                tc_fence_after();
            }
            tmem_st32(tmem + lane_off + kColPT + g * 32, pw);
            tmem_st32(tmem + lane_off + kColDST + g * 32, dw);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.ds_full);
        }
        if (ok) ok = __all_sync(0xffffffffu, wait_phase(&sm.acc_done, 0, flags, abort_word, P.wait_ns));
        if (ok) {
            tc_fence_after();
            // warpgroup g writes columns [64 g, 64 g + 64) of dV and dK
            uint32_t a[64];
            const size_t off = ((size_t)(start + key) * P.h_kv + hk) * kD + g * 64;
            tmem_ld64(tmem + lane_off + kColDV + g * 64, a);
            tmem_ld_wait();
            if (key < L) {
                uint4* dst = reinterpret_cast<uint4*>(dv + off);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(a[8 * j + 0]), __uint_as_float(a[8 * j + 1]));
                    w.y = pack_bf16x2(__uint_as_float(a[8 * j + 2]), __uint_as_float(a[8 * j + 3]));
                    w.z = pack_bf16x2(__uint_as_float(a[8 * j + 4]), __uint_as_float(a[8 * j + 5]));
                    w.w = pack_bf16x2(__uint_as_float(a[8 * j + 6]), __uint_as_float(a[8 * j + 7]));
                    dst[j] = w;
                }
            }
            tmem_ld64(tmem + lane_off + kColDK + g * 64, a);
            tmem_ld_wait();
            if (key < L) {
                const float s = P.scale;
                uint4* dst = reinterpret_cast<uint4*>(dk + off);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(a[8 * j + 0]) * s, __uint_as_float(a[8 * j + 1]) * s);
                    w.y = pack_bf16x2(__uint_as_float(a[8 * j + 2]) * s, __uint_as_float(a[8 * j + 3]) * s);
                    w.z = pack_bf16x2(__uint_as_float(a[8 * j + 4]) * s, __uint_as_float(a[8 * j + 5]) * s);
                    w.w = pack_bf16x2(__uint_as_float(a[8 * j + 6]) * s, __uint_as_float(a[8 * j + 7]) * s);
                    dst[j] = w;
                }
            }
        }
    } else if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmDO);
            mbar_arrive_expect_tx(&sm.kv_full, 2 * kTileBytes);
            for (int a = 0; a < 2; ++a) {
                tma_load_3d(sm.k + a * kB * kAtomCols, &tmK, &sm.kv_full, a * kAtomCols, hk, start + j0);
                tma_load_3d(sm.v + a * kB * kAtomCols, &tmV, &sm.kv_full, a * kAtomCols, hk, start + j0);
            }
        }
        int issued = 0;
        for (int i = 0; i < nsteps; ++i) {
            const int st = i % kBStages;
            if (i >= kBStages &&
                !__all_sync(0xffffffffu, wait_phase(&sm.q_empty[st], ((i / kBStages) - 1) & 1, flags,
                                                    abort_word, P.wait_ns)))
                break;
            const int hq = hk * P.group + i / nqb;
            const int r0 = (qb_lo + i % nqb) * kB;
            if (lane == 0) {
                mbar_arrive_expect_tx(&sm.q_full[st], 2 * kTileBytes);
                for (int a = 0; a < 2; ++a) {
                    tma_load_3d(sm.q[st] + a * kB * kAtomCols, &tmQ, &sm.q_full[st], a * kAtomCols, hq,
                                start + r0);
                    tma_load_3d(sm.dout[st] + a * kB * kAtomCols, &tmDO, &sm.q_full[st], a * kAtomCols,
                                hq, start + r0);
                }
            }
            for (int c = lane; c < kB; c += 32) {
                const int row = r0 + c;
                const size_t rix = (size_t)hq * P.total + start + row;
                sm.lse2[st][c] = row < L ? __ldg(lse + rix) * kLog2e : 0.f;
                sm.dlt[st][c] = row < L ? __ldg(delta + rix) : 0.f;
            }
            mbar_arrive(&sm.rows_full[st]);
            issued = i + 1;
        }
        if (lane == 0) {
            drain_phase(&sm.kv_full, 0, P.wait_ns);
            for (int i = max(0, issued - kBStages); i < issued; ++i)
                drain_phase(&sm.q_full[i % kBStages], (i / kBStages) & 1, P.wait_ns);
        }
    } else if (lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idS = idesc_bf16(kB, kB, 0, 0);         // S^T, dP^T: A, B K-major
        constexpr uint32_t idG = idesc_bf16(kB, kD, 0, 1);         // dV, dK: B MN-major, N = 128
        const uint64_t dkey = smem_desc_sw128(smem_u32(sm.k), 16, 1024);
        const uint64_t dval = smem_desc_sw128(smem_u32(sm.v), 16, 1024);
        auto st_product = [&](int st) {
            const uint64_t dqk = smem_desc_sw128(smem_u32(sm.q[st]), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
                mma_ss(tmem + kColSP, dkey + kstep_off(kk), dqk + kstep_off(kk), idS, kk > 0);
        };
        auto dpt_product = [&](int st) {
            const uint64_t ddo = smem_desc_sw128(smem_u32(sm.dout[st]), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
                mma_ss(tmem + kColSP, dval + kstep_off(kk), ddo + kstep_off(kk), idS, kk > 0);
        };
        auto grads = [&](int st, bool acc) {
            const uint64_t ddo = smem_desc_sw128(smem_u32(sm.dout[st]), kAtomBytes, 1024);
            const uint64_t dqm = smem_desc_sw128(smem_u32(sm.q[st]), kAtomBytes, 1024);
#pragma unroll
            for (int kk = 0; kk < kB / 16; ++kk)
                mma_ts(tmem + kColDV, tmem + kColPT + kk * 8, ddo + mnstep_off(0, kk), idG, acc || kk > 0);
#pragma unroll
            for (int kk = 0; kk < kB / 16; ++kk)
                mma_ts(tmem + kColDK, tmem + kColDST + kk * 8, dqm + mnstep_off(0, kk), idG, acc || kk > 0);
        };
        bool ok = wait_phase(&sm.kv_full, 0, flags, abort_word, P.wait_ns) &&
                  wait_phase(&sm.q_full[0], 0, flags, abort_word, P.wait_ns);
        if (ok) {
            tc_fence_after();
            st_product(0);
            mma_commit(&sm.s_full);
            ok = wait_phase(&sm.s_loaded, 0, flags, abort_word, P.wait_ns);
        }
        if (ok) {
            tc_fence_after();
            dpt_product(0);
            mma_commit(&sm.dp_full);
        }
        for (int i = 0; ok && i < nsteps; ++i) {
            const int st = i % kBStages, st1 = (i + 1) % kBStages;
            if (i + 1 < nsteps) {
                // S^T(i+1) over dP^T(i) once that has been read, ahead of dV/dK(i)
                if (!(ok = wait_phase(&sm.dp_loaded, i & 1, flags, abort_word, P.wait_ns))) break;
                if (!(ok = wait_phase(&sm.q_full[st1], ((i + 1) / kBStages) & 1, flags, abort_word, P.wait_ns))) break;
                tc_fence_after();
                st_product(st1);
                mma_commit(&sm.s_full);
            }
            if (!(ok = wait_phase(&sm.ds_full, i & 1, flags, abort_word, P.wait_ns))) break;
            tc_fence_after();
            grads(st, i > 0);
            mma_commit(&sm.pd_free);
            mma_commit(&sm.q_empty[st]);
            if (i + 1 < nsteps) {
                if (!(ok = wait_phase(&sm.s_loaded, (i + 1) & 1, flags, abort_word, P.wait_ns))) break;
                tc_fence_after();
                dpt_product(st1);
                mma_commit(&sm.dp_full);
            }
        }
        mma_commit(&sm.acc_done);
        mma_commit(&sm.drained);
        drain_phase(&sm.drained, 0, P.wait_ns);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<512>(tmem);
    }
}

}  // namespace

bool tc_bwd128_supported(const Problem& P, bool bf16) {
    return bf16 && P.head_dim == kD && P.total > 0;
}

cudaError_t tc_bwd128(const Problem& P, const void* q, const void* k, const void* v,
                      const float* lse, const float* delta, const void* dout, void* dq, void* dk,
                      void* dv, uint32_t* flags, cudaStream_t st) {
    if (P.nseq == 0 || P.max_seqlen == 0) return cudaSuccess;
    CUtensorMap mq, mk, mv, mdo;
    if (!make_head_tile_map(&mq, q, P.total, P.h_q, kB, kD) ||
        !make_head_tile_map(&mk, k, P.total, P.h_kv, kB, kD) ||
        !make_head_tile_map(&mv, v, P.total, P.h_kv, kB, kD) ||
        !make_head_tile_map(&mdo, dout, P.total, P.h_q, kB, kD))
        return cudaErrorInvalidValue;
    const int nblocks = (P.max_seqlen + kB - 1) / kB;
    const size_t smem_a = sizeof(DqSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(bwd128_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_a);
    if (e != cudaSuccess) return e;
    bwd128_dq_kernel<<<dim3(nblocks, P.h_q, P.nseq), kAThreads, smem_a, st>>>(
        mk, mv, mdo, P, (const __nv_bfloat16*)q, lse, delta, (__nv_bfloat16*)dq, flags);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t smem_b = sizeof(DkvSmem) + 1024;
    e = cudaFuncSetAttribute(bwd128_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_b);
    if (e != cudaSuccess) return e;
    bwd128_dkdv_kernel<<<dim3(nblocks, P.h_kv, P.nseq), kBThreads, smem_b, st>>>(
        mq, mk, mv, mdo, P, lse, delta, (__nv_bfloat16*)dk, (__nv_bfloat16*)dv, flags);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace sinkattn
