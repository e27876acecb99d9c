// tc_bwd_dq.cu - the dQ half of the 64-wide sink-attention backward on the
// sm_103a tensor cores, one query block per CTA, with no atomics.
//
// What it computes (page "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、超稳定！",
// section "反向传播的实现"), with LSE (sink included) from the forward and
// delta_i = dO_i . O_i from the preprocess step:
//   P_ij = exp(S_ij - LSE_i)   dP_ij = dO_i . V_j   dS_ij = P_ij (dP_ij - delta_i)
//   dQ_i = scale sum_j dS_ij K_j
// dK and dV come from the key-owning kernel (tc_bwd.cu without its dQ part).
//
// One CTA = 128 query rows of one head, walking the key blocks those rows see.
// Warpgroup w (warps 4w..4w+3) takes keys [64w, 64w + 64) of each block, and
// its thread r owns row r (tensor-memory lane r), so LSE_r and delta_r are
// per-thread constants; two warpgroups keep two warps per sub-partition on the
// exponentials. Every product takes its A operand from tensor memory:
//   S  = Q K^T     A = Q  (written once by the row threads, f16)  B = K (f16, K-major)
//   dP = dO V^T    A = dO (written once, bf16)                    B = V (bf16, K-major)
//   dQ += dS K     A = dS (from the row threads, f16)             B = K (f16, MN-major)
// dQ accumulates in tensor memory over the key blocks and is written once, in
// bf16, so it is reproducible bit for bit. dS and the operands it meets are
// f16: with large logits bf16's 8 bits of dS would put dQ out of tolerance.
// Q and K are read from the f16 copies that the launcher writes first.
// Tensor memory: S 0..127, dP 128..255, dQ 256..319, dS 320..383, Q 384..415,
// dO 416..447. Warps: 0-7 row threads, 8 TMA producer (K and V tiles through a
// kStages ring), 9 MMA issuer. Every mbarrier wait is bounded.
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

constexpr int kB = 128;  // query rows per CTA = keys per block
constexpr int kD = 64;
constexpr int kStages = 3;
constexpr int kThreads = 320;
constexpr uint32_t kTileBytes = kB * kD * 2;  // 16 KB: one 128-byte-swizzled atom
constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 320, kColQ = 384,
                   kColDO = 416;

struct DqSmem {
    alignas(1024) __nv_bfloat16 k[kStages][kB * kD];
    alignas(1024) __nv_bfloat16 v[kStages][kB * kD];
    uint64_t rows_ready;
    uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
    uint64_t s_full, s_loaded, dp_full, dp_loaded, ds_full, dq_done, drained;
    uint32_t tmem_slot;
    int abort_flag;
};
static_assert(sizeof(DqSmem) + 1024 <= 232448, "dQ kernel shared memory");

__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const Problem P, const __nv_bfloat16* __restrict__ q16,
              const __nv_bfloat16* __restrict__ dout, const float* __restrict__ lse,
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
    if (L > P.max_seqlen) {
        // as in the forward: rows and keys past max_seqlen are not computed
        if (bc.x == 0 && threadIdx.x == 0) atomicOr(flags, kFlagSeqTooLong);
        L = P.max_seqlen;
    }
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
        mbar_init(&sm.rows_ready, 256);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.k_full[i], 1);
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.kv_empty[i], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_loaded, 256);
        mbar_init(&sm.dp_full, 1);
        mbar_init(&sm.dp_loaded, 256);
        mbar_init(&sm.ds_full, 256);
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

    if (warp < 8) {
        // ------------------------------------------------------------ row threads
        const int w = warp / 4;           // key half of each block: keys [64w, 64w + 64)
        const int r = (warp % 4) * 32 + lane;
        const int row = r0 + r;
        const bool valid = row < L;
        const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
        {
            // this row's Q (f16, warpgroup 0) or dO (bf16, warpgroup 1): the A
            // operands of S and dP
            const size_t off = ((size_t)(start + (valid ? row : r0)) * P.h_q + h) * kD;
            uint32_t rw[32];
            const uint4* src = reinterpret_cast<const uint4*>((w == 0 ? q16 : dout) + off);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 x = valid ? __ldg(src + j) : make_uint4(0u, 0u, 0u, 0u);
                rw[4 * j] = x.x;
                rw[4 * j + 1] = x.y;
                rw[4 * j + 2] = x.z;
                rw[4 * j + 3] = x.w;
            }
            tmem_st32(tmem + lane_off + (w == 0 ? kColQ : kColDO), rw);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.rows_ready);
        }
        const float sc = P.scale_log2;
        const size_t rix = (size_t)h * P.total + start + (valid ? row : r0);
        const float lse2 = valid ? __ldg(lse + rix) * kLog2e : 0.f;
        const float dlt = valid ? __ldg(delta + rix) : 0.f;
        const uint64_t sc2 = f2_pack(sc, sc);
        const uint64_t nl2 = f2_pack(-lse2, -lse2);
        const uint64_t nd2 = f2_pack(-dlt, -dlt);
        const int lo = P.causal && P.window > 0 ? row - P.window + 1 : INT_MIN;
        const int hi = P.causal ? min(row, L - 1) : L - 1;
        bool ok = true;
        for (int i = 0; i < nblk; ++i) {
            ok = __all_sync(0xffffffffu, wait_phase(&sm.s_full, i & 1, flags, abort_word, P.wait_ns));
            if (!ok) break;
            tc_fence_after();
            float p[64];
            {
                uint32_t a[64];
                tmem_ld64(tmem + lane_off + kColS + 64 * w, a);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&sm.s_loaded);  // the next block's S may be issued
#pragma unroll
                for (int j = 0; j < 64; ++j) p[j] = __uint_as_float(a[j]);
            }
            const int kp0 = (kb_lo + i) * kB + 64 * w;  // first key of this thread's half
            const int bk0 = (kb_lo + i) * kB;
            const bool need_mask = P.causal ? (bk0 + kB - 1 > r0 || (P.window > 0 && bk0 < r0 + kB - P.window))
                                            : (bk0 + kB > L);
            if (need_mask) {
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const int kp = kp0 + j;
                    if (kp < lo || kp > hi) p[j] = -INFINITY;
                }
            }
            // P = exp2(S scale log2 e - LSE log2 e), two columns per paired FMA
#pragma unroll
            for (int j = 0; j < 64; j += 2) {
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(p[j], p[j + 1]), sc2, nl2), x0, x1);
                p[j] = fast_exp2(x0);
                p[j + 1] = fast_exp2(x1);
            }
            ok = __all_sync(0xffffffffu, wait_phase(&sm.dp_full, i & 1, flags, abort_word, P.wait_ns));
            if (!ok) break;
            tc_fence_after();
            uint32_t dsw[32];  // dS of this row's key half as f16 pairs
            {
                uint32_t d[64];
                tmem_ld64(tmem + lane_off + kColDP + 64 * w, d);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&sm.dp_loaded);  // the next block's dP may be issued
#pragma unroll
                for (int j = 0; j < 64; j += 2) {
                    float y0, y1;
                    const uint64_t t = f2_add(f2_pack(__uint_as_float(d[j]), __uint_as_float(d[j + 1])), nd2);
                    f2_unpack(f2_mul(f2_pack(p[j], p[j + 1]), t), y0, y1);
                    dsw[j / 2] = pack_f16x2(y0, y1);
                }
            }
            if (i > 0) {
                // dQ of the previous block has read the dS columns
                ok = __all_sync(0xffffffffu, wait_phase(&sm.dq_done, (i - 1) & 1, flags, abort_word, P.wait_ns));
                if (!ok) break;
                tc_fence_after();
            }
            tmem_st32(tmem + lane_off + kColDS + 32 * w, dsw);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.ds_full);
        }
        if (ok) ok = __all_sync(0xffffffffu, wait_phase(&sm.dq_done, (nblk - 1) & 1, flags, abort_word, P.wait_ns));
        if (ok) {
            // warpgroup w writes dQ columns [32w, 32w + 32) of the row
            tc_fence_after();
            uint32_t a[32];
            tmem_ld32(tmem + lane_off + kColDQ + 32 * w, a);
            tmem_ld_wait();
            if (valid) {
                uint4* dst = reinterpret_cast<uint4*>(dq + ((size_t)(start + row) * P.h_q + h) * kD) + 4 * w;
                const float s = P.scale;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    dst[j] = make_uint4(pack_bf16x2(__uint_as_float(a[8 * j]) * s, __uint_as_float(a[8 * j + 1]) * s),
                                        pack_bf16x2(__uint_as_float(a[8 * j + 2]) * s, __uint_as_float(a[8 * j + 3]) * s),
                                        pack_bf16x2(__uint_as_float(a[8 * j + 4]) * s, __uint_as_float(a[8 * j + 5]) * s),
                                        pack_bf16x2(__uint_as_float(a[8 * j + 6]) * s, __uint_as_float(a[8 * j + 7]) * s));
            }
        }
    } else if (warp == 8) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            int issued = 0;
            for (int i = 0; i < nblk; ++i) {
                const int st = i % kStages;
                if (i >= kStages &&
                    !wait_phase(&sm.kv_empty[st], ((i / kStages) - 1) & 1, flags, abort_word, P.wait_ns))
                    break;
                const int kpos = start + (kb_lo + i) * kB;
                mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
                tma_load_3d(sm.k[st], &tmK, &sm.k_full[st], 0, hk, kpos);
                mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
                tma_load_3d(sm.v[st], &tmV, &sm.v_full[st], 0, hk, kpos);
                issued = i + 1;
            }
            // copies still in flight must land before the CTA's shared memory goes away
            for (int i = max(0, issued - kStages); i < issued; ++i) {
                const int st = i % kStages;
                drain_phase(&sm.k_full[st], (i / kStages) & 1, P.wait_ns);
                drain_phase(&sm.v_full[st], (i / kStages) & 1, P.wait_ns);
            }
        }
    } else if (warp == 9 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idS = idesc_f16(kB, kB, 0, 0);    // S: Q (tmem), K K-major, f16
        constexpr uint32_t idDP = idesc_bf16(kB, kB, 0, 0);  // dP: dO (tmem), V K-major, bf16
        constexpr uint32_t idQ = idesc_f16(kB, kD, 0, 1);    // dQ: dS (tmem), K MN-major, f16
        auto s_product = [&](int st) {
            const uint64_t dk = smem_desc_sw128(smem_u32(sm.k[st]), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
                mma_ts(tmem + kColS, tmem + kColQ + kk * 8, dk + 2 * kk, idS, kk > 0);
        };
        auto dp_product = [&](int st) {
            const uint64_t dv = smem_desc_sw128(smem_u32(sm.v[st]), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
                mma_ts(tmem + kColDP, tmem + kColDO + kk * 8, dv + 2 * kk, idDP, kk > 0);
        };
        auto dq_product = [&](int st, bool acc) {
            const uint64_t dk = smem_desc_sw128(smem_u32(sm.k[st]), 1024, 1024);
#pragma unroll
            for (int kk = 0; kk < kB / 16; ++kk)
                mma_ts(tmem + kColDQ, tmem + kColDS + kk * 8, dk + (uint64_t)((kk * 2048) >> 4), idQ,
                       acc || kk > 0);
        };
        bool ok = wait_phase(&sm.rows_ready, 0, flags, abort_word, P.wait_ns) &&
                  wait_phase(&sm.k_full[0], 0, flags, abort_word, P.wait_ns);
        if (ok) {
            tc_fence_after();
            s_product(0);
            mma_commit(&sm.s_full);
            ok = wait_phase(&sm.v_full[0], 0, flags, abort_word, P.wait_ns);
        }
        if (ok) {
            tc_fence_after();
            dp_product(0);
            mma_commit(&sm.dp_full);
        }
        for (int i = 0; ok && i < nblk; ++i) {
            const int st = i % kStages, st1 = (i + 1) % kStages;
            if (i + 1 < nblk) {
                // S(i+1) once S(i) is read, dP(i+1) once dP(i) is read: both ahead of dQ(i)
                if (!(ok = wait_phase(&sm.s_loaded, i & 1, flags, abort_word, P.wait_ns))) break;
                if (!(ok = wait_phase(&sm.k_full[st1], ((i + 1) / kStages) & 1, flags, abort_word, P.wait_ns))) break;
                tc_fence_after();
                s_product(st1);
                mma_commit(&sm.s_full);
                if (!(ok = wait_phase(&sm.dp_loaded, i & 1, flags, abort_word, P.wait_ns))) break;
                if (!(ok = wait_phase(&sm.v_full[st1], ((i + 1) / kStages) & 1, flags, abort_word, P.wait_ns))) break;
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

}  // namespace

cudaError_t tc_bwd_dq64(const Problem& P, const CUtensorMap& mk16, const CUtensorMap& mv,
                        const void* q16, const void* dout, const float* lse, const float* delta,
                        void* dq, uint32_t* flags, cudaStream_t st) {
    const size_t smem = sizeof(DqSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int nblocks = (P.max_seqlen + kB - 1) / kB;
    bwd_dq_kernel<<<dim3(nblocks, P.h_q, P.nseq), kThreads, smem, st>>>(
        mk16, mv, P, (const __nv_bfloat16*)q16, (const __nv_bfloat16*)dout, lse, delta,
        (__nv_bfloat16*)dq, flags);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace sinkattn
