// tc_bwd.cu - sink-attention backward main loop on the sm_103a tensor cores.
//
// What it computes (page "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、超稳定！",
// section "反向传播的实现"): with the forward's logsumexp LSE (sink included)
// and delta_i = dO_i . O_i from the preprocess step,
//   P_ij  = exp(S_ij - LSE_i)                (the sink needs no term: LSE has it)
//   dV_j  = sum_i P_ij dO_i                  dP_ij = dO_i . V_j
//   dS_ij = P_ij (dP_ij - delta_i)
//   dK_j  = scale sum_i dS_ij Q_i            dQ_i  = scale sum_j dS_ij K_j
// dK and dV sum over the query heads of each key/value head. The sink's own
// gradient is formed by the preprocess step.
//
// One CTA = one key block of 128 keys of one key/value head of one sequence;
// it walks every (query head of the group, query block of 128 rows) that can
// see the block, accumulating dK and dV in tensor memory, and adds each dQ
// block into an fp32 accumulator in the workspace.
//   warps 0-7    two elementwise warpgroups: thread = key (tensor-memory lane),
//                warpgroup w takes query rows [64w, 64w+64) of the block.
//                P^T goes to tensor memory (A operand of dV), dS^T to shared
//                memory in a layout that is the K-major A operand of dK and,
//                read the other way, the MN-major A operand of dQ.
//   warp 8       TMA producer: K, V once; Q, dO (+ LSE, delta) per step through
//                a 2-deep ring.
//   warp 9       MMA issuer (one thread): S^T = K Q^T and dP^T = V dO^T for the
//                next step as soon as the elementwise warps have read the
//                current ones, then dV += P^T dO, dK += dS^T Q, dQ = dS K.
//   warps 12-15  dQ drain: tensor memory -> fp32 vector atomics.
// Tensor memory: S^T 0..127, dP^T 128..255, dV 256..319, dK 320..383,
// dQ 384..447, P^T (bf16 pairs) 448..511.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace sinkattn {
namespace {

using namespace tc;

constexpr int kBN = 128;  // keys per CTA
constexpr int kBM = 128;  // query rows per step
constexpr int kD = 64;
constexpr int kQStages = 2;
constexpr uint32_t kTileBytes = kBM * kD * 2;
constexpr int kThreads = 512;
// Register split (launch: 512 threads x 128): 2 elementwise warpgroups x 128
// x 176 + producer/MMA warpgroup x 128 x 56 + dQ warpgroup x 128 x 96
// = 45056 + 7168 + 12288 = 64512 <= 65536.
constexpr int kLaunchRegs = 128;
constexpr int kEltRegs = 176;
constexpr int kCtlRegs = 56;
constexpr int kDqRegs = 96;
static_assert(2 * 128 * kEltRegs + 128 * kCtlRegs + 128 * kDqRegs <= kThreads * kLaunchRegs,
              "register split");

constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 320, kColDQ = 384, kColP = 448;

struct BwdSmem {
    alignas(1024) __nv_bfloat16 k[kBN * kD];
    alignas(1024) __nv_bfloat16 v[kBN * kD];
    alignas(1024) __nv_bfloat16 q[kQStages][kBM * kD];
    alignas(1024) __nv_bfloat16 dout[kQStages][kBM * kD];
    // dS^T: two 16 KB atoms (query rows 0..63 and 64..127), each 128 keys x 128 bytes
    alignas(1024) uint8_t ds[2][kBN * 128];
    float lse2[kQStages][kBM];  // LSE * log2(e); +inf marks rows outside the sequence
    float delta[kQStages][kBM];
    uint64_t kv_full;
    uint64_t q_full[kQStages], q_empty[kQStages];
    uint64_t sdp_full, s_consumed, ds_full, grads_done, dq_consumed, drained;
    uint32_t tmem_slot;
    int abort_flag;
};

// byte offset of (row r, byte b) inside a tile of 128-byte rows with the 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int r, int b) {
    return (uint32_t)(r * 128 + (((b >> 4) ^ (r & 7)) << 4) + (b & 15));
}

__device__ __forceinline__ uint4 pack8(const uint32_t* a, float f) {
    return make_uint4(pack_bf16x2(__uint_as_float(a[0]) * f, __uint_as_float(a[1]) * f),
                      pack_bf16x2(__uint_as_float(a[2]) * f, __uint_as_float(a[3]) * f),
                      pack_bf16x2(__uint_as_float(a[4]) * f, __uint_as_float(a[5]) * f),
                      pack_bf16x2(__uint_as_float(a[6]) * f, __uint_as_float(a[7]) * f));
}

__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              const Problem P, const float* __restrict__ lse, const float* __restrict__ delta,
              float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dk,
              __nv_bfloat16* __restrict__ dv, uint32_t* flags) {
    extern __shared__ uint8_t smem_raw[];
    BwdSmem& sm = *reinterpret_cast<BwdSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int kb = blockIdx.x;  // key block; block 0 sees the most rows under a causal mask
    const int hk = blockIdx.y;
    const int seq = blockIdx.z;
    int start, L;
    seq_bounds(P, seq, start, L);
    const int k0 = kb * kBN;
    if (k0 >= L) return;  // uniform for the CTA, before any barrier or TMEM use

    // query blocks that can see keys [k0, k0 + 128)
    const int nrb = (L + kBM - 1) / kBM;
    int qb_lo = 0, qb_hi = nrb - 1;
    if (P.causal) {
        qb_lo = kb;
        if (P.window > 0) qb_hi = min(nrb - 1, (k0 + kBN - 1 + P.window - 1) / kBM);
    }
    const int nq = qb_hi - qb_lo + 1;
    const int nsteps = nq * P.group;

    if (threadIdx.x == 0) {
        mbar_init(&sm.kv_full, 1);
        for (int i = 0; i < kQStages; ++i) {
            mbar_init(&sm.q_full[i], 1 + 32);
            mbar_init(&sm.q_empty[i], 1);
        }
        mbar_init(&sm.sdp_full, 1);
        mbar_init(&sm.s_consumed, 256);
        mbar_init(&sm.ds_full, 256);
        mbar_init(&sm.grads_done, 1);
        mbar_init(&sm.dq_consumed, 128);
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
        // ------------------------------------------------------------ elementwise
        regs_increase<kEltRegs>();
        const int w = warp / 4;         // query-row half of the block
        const int wq = warp % 4;
        const int kr = wq * 32 + lane;  // key within the block (tensor-memory lane)
        const int kp = k0 + kr;         // key position in the sequence
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const float sc = P.scale_log2;
        bool ok = true;
        for (int it = 0; it < nsteps; ++it) {
            const int st = it % kQStages;
            const int q0 = (qb_lo + it % nq) * kBM;
            ok = __all_sync(0xffffffffu, wait_phase(&sm.sdp_full, it & 1, flags, abort_word));
            if (!ok) break;
            tc_fence_after();
            const bool need_mask =
                P.causal ? (k0 + kBN - 1 > q0 || (P.window > 0 && k0 < q0 + kBM - P.window))
                         : (k0 + kBN > L);
            uint32_t pp[32], pd[32];  // packed bf16 pairs of P^T and dS^T, 64 rows
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                const int c0 = 64 * w + 32 * ch;  // first query row of the chunk
                uint32_t sraw[32], draw[32];
                tmem_ld32(tmem + lane_off + kColS + c0, sraw);
                tmem_ld32(tmem + lane_off + kColDP + c0, draw);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    float p2[2], d2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int c = c0 + j + u;
                        float p = fast_exp2(fmaf(__uint_as_float(sraw[j + u]), sc, -sm.lse2[st][c]));
                        if (need_mask) {
                            const int ip = q0 + c;
                            const bool allowed =
                                P.causal ? (kp <= ip && (P.window <= 0 || kp > ip - P.window))
                                         : kp < L;
                            p = allowed ? p : 0.f;
                        }
                        p2[u] = p;
                        d2[u] = p * (__uint_as_float(draw[j + u]) - sm.delta[st][c]);
                    }
                    pp[16 * ch + j / 2] = pack_bf16x2(p2[0], p2[1]);
                    pd[16 * ch + j / 2] = pack_bf16x2(d2[0], d2[1]);
                }
            }
            // S^T and dP^T have been read: the next step's products may overwrite them
            tc_fence_before();
            mbar_arrive(&sm.s_consumed);
            // the previous step's gradient products read P^T and dS^T: wait for them
            if (it > 0) {
                ok = __all_sync(0xffffffffu,
                                wait_phase(&sm.grads_done, (it - 1) & 1, flags, abort_word));
                if (!ok) break;
            }
            tc_fence_after();
            tmem_st32(tmem + lane_off + kColP + 32 * w, pp);
            // dS^T row of this key: 64 query rows = 128 bytes of atom w
            uint8_t* atom = sm.ds[w];
#pragma unroll
            for (int c16 = 0; c16 < 8; ++c16) {
                const uint4 val = make_uint4(pd[4 * c16], pd[4 * c16 + 1], pd[4 * c16 + 2], pd[4 * c16 + 3]);
                *reinterpret_cast<uint4*>(atom + sw128(kr, c16 * 16)) = val;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.ds_full);
        }
        // epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK (scaled)
        if (ok)
            ok = __all_sync(0xffffffffu,
                            wait_phase(&sm.grads_done, (nsteps - 1) & 1, flags, abort_word));
        if (ok) {
            tc_fence_after();
            uint32_t a[32], b[32];
            const uint32_t col = w == 0 ? kColDV : kColDK;
            tmem_ld32(tmem + lane_off + col, a);
            tmem_ld32(tmem + lane_off + col + 32, b);
            tmem_ld_wait();
            if (kp < L) {
                const float f = w == 0 ? 1.f : P.scale;
                __nv_bfloat16* dst = (w == 0 ? dv : dk) + ((size_t)(start + kp) * P.h_kv + hk) * kD;
                uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                for (int j = 0; j < 4; ++j) d4[j] = pack8(a + 8 * j, f);
#pragma unroll
                for (int j = 0; j < 4; ++j) d4[4 + j] = pack8(b + 8 * j, f);
            }
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ dQ drain
        regs_decrease<kDqRegs>();
        const int wq = warp - 12;
        const int r = wq * 32 + lane;  // query row within the block (tensor-memory lane)
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        for (int it = 0; it < nsteps; ++it) {
            const int h = hk * P.group + it / nq;
            const int qb = qb_lo + it % nq;
            if (!__all_sync(0xffffffffu, wait_phase(&sm.grads_done, it & 1, flags, abort_word)))
                break;
            tc_fence_after();
            uint32_t a[32], b[32];
            tmem_ld32(tmem + lane_off + kColDQ, a);
            tmem_ld32(tmem + lane_off + kColDQ + 32, b);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&sm.dq_consumed);
            const int ip = qb * kBM + r;
            if (ip < L) {
                float4* dst = reinterpret_cast<float4*>(dq_acc + ((size_t)(start + ip) * P.h_q + h) * kD);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    atomicAdd(dst + j, make_float4(__uint_as_float(a[4 * j]), __uint_as_float(a[4 * j + 1]),
                                                   __uint_as_float(a[4 * j + 2]), __uint_as_float(a[4 * j + 3])));
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    atomicAdd(dst + 8 + j, make_float4(__uint_as_float(b[4 * j]), __uint_as_float(b[4 * j + 1]),
                                                       __uint_as_float(b[4 * j + 2]), __uint_as_float(b[4 * j + 3])));
            }
        }
    } else {
        regs_decrease<kCtlRegs>();
        if (warp == 8) {
            // -------------------------------------------------------- producer
            if (lane == 0) {
                tma_prefetch_desc(&tmQ);
                tma_prefetch_desc(&tmK);
                tma_prefetch_desc(&tmV);
                tma_prefetch_desc(&tmDO);
                mbar_arrive_expect_tx(&sm.kv_full, 2 * kTileBytes);
                tma_load_3d(sm.k, &tmK, &sm.kv_full, 0, hk, start + k0);
                tma_load_3d(sm.v, &tmV, &sm.kv_full, 0, hk, start + k0);
            }
            int issued = 0;
            for (int it = 0; it < nsteps; ++it) {
                const int st = it % kQStages;
                const int h = hk * P.group + it / nq;
                const int q0 = (qb_lo + it % nq) * kBM;
                if (it >= kQStages &&
                    !__all_sync(0xffffffffu, wait_phase(&sm.q_empty[st], ((it / kQStages) - 1) & 1,
                                                        flags, abort_word)))
                    break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sm.q_full[st], 2 * kTileBytes);
                    tma_load_3d(sm.q[st], &tmQ, &sm.q_full[st], 0, h, start + q0);
                    tma_load_3d(sm.dout[st], &tmDO, &sm.q_full[st], 0, h, start + q0);
                }
#pragma unroll
                for (int u = 0; u < kBM / 32; ++u) {
                    const int c = lane * (kBM / 32) + u;
                    const int ip = q0 + c;
                    const size_t ix = (size_t)h * P.total + start + ip;
                    sm.lse2[st][c] = ip < L ? lse[ix] * kLog2e : INFINITY;
                    sm.delta[st][c] = ip < L ? delta[ix] : 0.f;
                }
                mbar_arrive(&sm.q_full[st]);
                issued = it + 1;
            }
            if (lane == 0) {
                drain_phase(&sm.kv_full, 0);
                for (int it = max(0, issued - kQStages); it < issued; ++it)
                    drain_phase(&sm.q_full[it % kQStages], (it / kQStages) & 1);
            }
        } else if (warp == 9 && lane == 0) {
            // -------------------------------------------------------- MMA issuer
            constexpr uint32_t idSS = idesc_bf16(kBN, kBM, 0, 0);  // S^T, dP^T: K-major A and B
            constexpr uint32_t idG = idesc_bf16(kBN, kD, 0, 1);    // dV, dK: B MN-major
            constexpr uint32_t idQ = idesc_bf16(kBM, kD, 1, 1);    // dQ: A and B MN-major
            const uint64_t dK_ = smem_desc_sw128(smem_u32(sm.k), 16, 1024);
            const uint64_t dV_ = smem_desc_sw128(smem_u32(sm.v), 16, 1024);
            const uint64_t dKmn = smem_desc_sw128(smem_u32(sm.k), 1024, 1024);
            bool ok = wait_phase(&sm.kv_full, 0, flags, abort_word) &&
                      wait_phase(&sm.q_full[0], 0, flags, abort_word);
            auto issue_sdp = [&](int st) {
                tc_fence_after();
                const uint64_t dq_ = smem_desc_sw128(smem_u32(sm.q[st]), 16, 1024);
                const uint64_t ddo = smem_desc_sw128(smem_u32(sm.dout[st]), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    mma_ss(tmem + kColS, dK_ + 2 * kk, dq_ + 2 * kk, idSS, kk > 0);
                    mma_ss(tmem + kColDP, dV_ + 2 * kk, ddo + 2 * kk, idSS, kk > 0);
                }
                mma_commit(&sm.sdp_full);
            };
            if (ok) issue_sdp(0);
            for (int it = 0; ok && it < nsteps; ++it) {
                const int st = it % kQStages;
                if (it + 1 < nsteps) {
                    const int st1 = (it + 1) % kQStages;
                    if (!(ok = wait_phase(&sm.q_full[st1], ((it + 1) / kQStages) & 1, flags, abort_word)))
                        break;
                    if (!(ok = wait_phase(&sm.s_consumed, it & 1, flags, abort_word))) break;
                    issue_sdp(st1);
                }
                if (!(ok = wait_phase(&sm.ds_full, it & 1, flags, abort_word))) break;
                tc_fence_after();
                const uint64_t ddo_mn = smem_desc_sw128(smem_u32(sm.dout[st]), 1024, 1024);
                const uint64_t dq_mn = smem_desc_sw128(smem_u32(sm.q[st]), 1024, 1024);
                const bool acc = it > 0;
#pragma unroll
                for (int kk = 0; kk < kBM / 16; ++kk) {
                    // dV += P^T dO   (A = P^T from tensor memory, K = query rows)
                    mma_ts(tmem + kColDV, tmem + kColP + kk * 8, ddo_mn + (uint64_t)((kk * 2048) >> 4),
                           idG, acc || kk > 0);
                    // dK += dS^T Q   (A = dS^T, K-major: atom kk/4, 32 bytes per 16 rows)
                    const uint64_t da = smem_desc_sw128(smem_u32(sm.ds[kk / 4]) + (kk % 4) * 32, 16, 1024);
                    mma_ss(tmem + kColDK, da, dq_mn + (uint64_t)((kk * 2048) >> 4), idG, acc || kk > 0);
                }
                if (it > 0) {
                    if (!(ok = wait_phase(&sm.dq_consumed, (it - 1) & 1, flags, abort_word))) break;
                    tc_fence_after();
                }
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    // dQ = dS K   (A = dS, MN-major: query rows contiguous, 2 atoms of 64)
                    const uint64_t da = smem_desc_sw128(smem_u32(sm.ds[0]) + kk * 2048, kBN * 128, 1024);
                    mma_ss(tmem + kColDQ, da, dKmn + (uint64_t)((kk * 2048) >> 4), idQ, kk > 0);
                }
                mma_commit(&sm.grads_done);
                mma_commit(&sm.q_empty[st]);
            }
            // every MMA issued above must finish before tensor memory is released
            mma_commit(&sm.drained);
            drain_phase(&sm.drained, 0);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<512>(tmem);
    }
}

// dq = scale * dq_acc, fp32 -> bf16, 4 elements per thread
__global__ void dq_convert_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq, size_t n4,
                                  float scale) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x) {
        const float4 a = acc[i];
        dq[i] = make_uint2(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale));
    }
}

}  // namespace

bool tc_bwd_supported(const Problem& P, bool bf16) {
    return bf16 && P.head_dim == kD && P.total > 0;
}

size_t tc_bwd_workspace_bytes(const Problem& P, bool bf16) {
    if (!bf16 || P.head_dim != kD) return 0;
    return sizeof(float) * (size_t)P.total * P.h_q * kD;  // dQ accumulator
}

cudaError_t tc_bwd(const Problem& P, const void* q, const void* k, const void* v,
                   const float* lse, const float* delta, const void* dout, void* dq, void* dk,
                   void* dv, uint32_t* flags, void* workspace, cudaStream_t st) {
    if (P.nseq == 0 || P.max_seqlen == 0) return cudaSuccess;
    CUtensorMap mq, mk, mv, mdo;
    if (!make_head_tile_map(&mq, q, P.total, P.h_q, kBM) ||
        !make_head_tile_map(&mk, k, P.total, P.h_kv, kBN) ||
        !make_head_tile_map(&mv, v, P.total, P.h_kv, kBN) ||
        !make_head_tile_map(&mdo, dout, P.total, P.h_q, kBM))
        return cudaErrorInvalidValue;
    // the register split is only safe at exactly this launch value
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, bwd_tc_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    const size_t smem = sizeof(BwdSmem) + 1024;
    e = cudaFuncSetAttribute(bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    float* acc = static_cast<float*>(workspace);
    const size_t n = (size_t)P.total * P.h_q * kD;
    e = cudaMemsetAsync(acc, 0, n * sizeof(float), st);
    if (e != cudaSuccess) return e;
    dim3 grid((P.max_seqlen + kBN - 1) / kBN, P.h_kv, P.nseq);
    bwd_tc_kernel<<<grid, kThreads, smem, st>>>(mq, mk, mv, mdo, P, lse, delta, acc,
                                                (__nv_bfloat16*)dk, (__nv_bfloat16*)dv, flags);
    count_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t n4 = n / 4;
    const int blocks = (int)std::min<size_t>((n4 + 255) / 256, 152 * 32);
    dq_convert_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(acc),
                                              reinterpret_cast<uint2*>(dq), n4, P.scale);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace sinkattn
