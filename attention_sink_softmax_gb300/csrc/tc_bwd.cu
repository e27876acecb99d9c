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
// see the block ("steps"), accumulating dK and dV in tensor memory, and adds
// each step's dQ block into an fp32 accumulator in the workspace.
//
// Operand placement. On this tensor core an MMA whose A operand comes from
// tensor memory issues about twice as fast as one reading A from shared
// memory, so every product whose A operand can live in tensor memory does:
//   S^T  = K Q^T     A = K    (tensor memory, loaded once)    B = Q  (smem)
//   dP^T = V dO^T    A = V    (tensor memory, loaded once)    B = dO (smem)
//   dV  += P^T dO    A = P^T  (tensor memory, from registers) B = dO
//   dK  += dS^T Q    A = dS^T (tensor memory, from registers) B = Q
//   dQ   = dS K      A = dS   (smem: needs query rows as M)   B = K  (smem)
// dS feeds dQ and dK in f16 (with large logits bf16's 8 bits of dS push dQ and
// dK out of tolerance), so their B operands K and Q are f16 too: tc_bwd first
// writes f16 copies of Q and K into the workspace (convert.cu), the tiles are
// loaded from them, and S^T = K Q^T runs in f16 as well. dP^T and dV stay
// bf16. bf16 -> f16 is exact for magnitudes within f16's range.
// S^T and dP^T share one 128-column region: the elementwise warps read S^T
// into registers, then dP^T is computed into the same columns while they
// exponentiate. Two threads issue MMAs: one issues S^T and dP^T, the other
// dV, dK and dQ, so the tensor pipe always has one stream's products queued
// while the other thread waits on a barrier. The elementwise work of step i
// overlaps the gradient products of step i-1. The P^T / dS^T columns are
// released as soon as dV and dK of step i-1 are done, and dS goes to one of
// two shared-memory buffers, so step i's stores never wait for the dQ product
// of step i-1. A Q / dO stage is refilled once both issuers are done with it.
//
// Warps: 0-7 elementwise (thread = key = tensor-memory lane; warpgroup w takes
// query rows [64w, 64w+64) of the step); 8 producer (TMA for K, Q, dO, and the
// step's LSE and delta rows written as the B tiles of the extra K step, through
// a kQStages ring); 9 and 10 MMA issuers (one thread each); 12-15 dQ drain
// (tensor memory -> shared staging, 32 columns at a time -> TMA bulk
// reduce-add). Tensor memory: S^T/dP^T 0..127, dV
// 128..191, dK 192..255, dQ 256..319, K 320..351, V 352..383, P^T 384..447,
// dS^T 448..511.
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
constexpr int kQStages = 3;
constexpr uint32_t kTileBytes = kBM * kD * 2;
constexpr int kThreads = 512;
// Register split (launch: 512 threads x 128): 2 elementwise warpgroups x 128
// x 192 + producer/MMA warpgroup x 128 x 64 + dQ warpgroup x 128 x 64
// = 49152 + 8192 + 8192 = 65536.
constexpr int kLaunchRegs = 128;
constexpr int kEltRegs = 192;
constexpr int kCtlRegs = 64;
constexpr int kDqRegs = 64;
static_assert(2 * 128 * kEltRegs + 128 * kCtlRegs + 128 * kDqRegs <= kThreads * kLaunchRegs,
              "register split");

constexpr uint32_t kColSdP = 0, kColDV = 128, kColDK = 192, kColDQ = 256, kColK = 320,
                   kColV = 352, kColP = 384, kColDS = 448;

// LSE and delta reach the elementwise warps through the MMAs: one extra K = 16
// step is appended to S^T = K Q^T and to dP^T = V dO^T, whose A operand holds
// 1 in k = 0, 1, 2 of every key row and whose B operand holds, per query row,
// -LSE / scale (resp. -delta) split into three bf16 parts (hi + mid + lo carry
// about 24 bits). The accumulators then hold S - LSE / scale and dP - delta,
// so P = exp2(S' * scale * log2 e) and dS = P dP' need no per-column loads.
// The tiles are 128 rows x 16 bf16 without swizzle: element (r, k) at
// aug_off(r) + (k / 8) * 128 + (k % 8) * 2.
constexpr uint32_t kAugTile = 128 * 16 * 2;
constexpr uint32_t kAugLBO = 128, kAugSBO = 256;
__device__ __forceinline__ uint32_t aug_off(int r) { return (uint32_t)((r & 7) * 16 + (r >> 3) * 256); }

// three bf16 parts whose sum is v to about 24 bits, packed (k = 0, 1, 2, 3 = 0)
__device__ __forceinline__ uint2 split3_bf16(float v) {
    const __nv_bfloat16 a = __float2bfloat16_rn(v);
    float r = v - __bfloat162float(a);
    const __nv_bfloat16 b = __float2bfloat16_rn(r);
    r -= __bfloat162float(b);
    const __nv_bfloat16 c = __float2bfloat16_rn(r);
    return make_uint2((uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16),
                      (uint32_t)__bfloat16_as_ushort(c));
}

struct BwdSmem {
    alignas(1024) __nv_bfloat16 k[kBN * kD];  // B operand of dQ (converted to f16 in place)
    alignas(1024) __nv_bfloat16 q[kQStages][kBM * kD];
    alignas(1024) __nv_bfloat16 dout[kQStages][kBM * kD];
    // dS, double-buffered by step parity: two 16 KB atoms (query rows 0..63 and
    // 64..127), each 128 keys x 128 bytes
    alignas(1024) uint8_t ds[2][2][kBN * 128];
    // half a dQ block (32 columns) staged for the bulk reduce, 128 rows x 128 bytes
    alignas(1024) uint8_t dq_stage[kBM * 128];
    alignas(128) uint8_t aug_ones[kAugTile];              // A of the extra K step
    alignas(128) uint8_t aug_lse[kQStages][kAugTile];     // B: -LSE / scale, per query row
    alignas(128) uint8_t aug_delta[kQStages][kAugTile];   // B: -delta, per query row
    uint64_t k_full, kv_tmem;
    uint64_t q_full[kQStages], q_empty[kQStages];
    uint64_t s_full, s_loaded, dp_full, dp_loaded, ds_full, pd_free, ds_free[2], grads_done,
        dq_consumed, acc_done, drained[2];
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

// kDq = false: the same kernel without its dQ part (no dS in shared memory, no
// dQ product, the drain warps idle): the key-owning half of the split
// backward, whose dQ comes from tc_bwd_dq.cu.
template <bool kDq>
__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ CUtensorMap tmDQ,
              const Problem P, const __nv_bfloat16* __restrict__ kg,
              const __nv_bfloat16* __restrict__ vg, const float* __restrict__ lse,
              const float* __restrict__ delta, __nv_bfloat16* __restrict__ dk,
              __nv_bfloat16* __restrict__ dv, uint32_t* flags) {
    extern __shared__ uint8_t smem_raw[];
    BwdSmem& sm = *reinterpret_cast<BwdSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const BlockCoord bc = block_seq_x_head();
    const int kb = bc.x;  // key block; block 0 sees the most rows under a causal mask
    const int hk = bc.y;
    const int seq = bc.z;
    int start, L;
    if (!seq_bounds_checked(P, seq, start, L, flags)) return;
    if (L > P.max_seqlen) {
        // as in the forward: rows and keys past max_seqlen are not computed
        if (kb == 0 && threadIdx.x == 0) atomicOr(flags, kFlagSeqTooLong);
        L = P.max_seqlen;
    }
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

    // The elementwise threads fetch their key's K row (warpgroup 0, from the
    // f16 copy) or V row (warpgroup 1) now, and the producer thread
    // initialises the barriers and starts the K tile's load, so both are in
    // flight while warp 0 allocates tensor memory.
    uint32_t kv_row[32];
    if (warp < 8) {
        const int kp = k0 + (warp % 4) * 32 + lane;
        const __nv_bfloat16* src = (warp < 4 ? kg : vg) + ((size_t)(start + kp) * P.h_kv + hk) * kD;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 x = kp < L ? __ldg(reinterpret_cast<const uint4*>(src) + j) : make_uint4(0, 0, 0, 0);
            kv_row[4 * j] = x.x;
            kv_row[4 * j + 1] = x.y;
            kv_row[4 * j + 2] = x.z;
            kv_row[4 * j + 3] = x.w;
        }
    }
    if (threadIdx.x == 8 * 32) {
        mbar_init(&sm.k_full, 1);
        mbar_init(&sm.kv_tmem, 256);
        for (int i = 0; i < kQStages; ++i) {
            mbar_init(&sm.q_full[i], 1 + 32);
            mbar_init(&sm.q_empty[i], 2);  // one commit from each MMA issuer
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_loaded, 256);
        mbar_init(&sm.dp_full, 1);
        mbar_init(&sm.dp_loaded, 256);
        mbar_init(&sm.ds_full, 256);
        mbar_init(&sm.pd_free, 1);
        mbar_init(&sm.ds_free[0], 1);
        mbar_init(&sm.ds_free[1], 1);
        mbar_init(&sm.grads_done, 1);
        mbar_init(&sm.dq_consumed, 128);
        mbar_init(&sm.acc_done, 1);
        mbar_init(&sm.drained[0], 1);
        mbar_init(&sm.drained[1], 1);
        sm.abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmDO);
        mbar_arrive_expect_tx(&sm.k_full, kTileBytes);
        tma_load_3d(sm.k, &tmK, &sm.k_full, 0, hk, start + k0);
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
        const int w = warp / 4;         // query-row half of the step (and K or V at start)
        const int wq = warp % 4;
        const int kr = wq * 32 + lane;  // key within the block (tensor-memory lane)
        const int kp = k0 + kr;         // key position in the sequence
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const float sc = P.scale_log2;
        {
            // A operands of S^T and dP^T: warpgroup 0 places this key's K row (f16),
            // warpgroup 1 its V row (bf16), loaded above; zeros past the sequence
            tmem_st32(tmem + lane_off + (w == 0 ? kColK : kColV), kv_row);
            if (w == 0) {
                // A of the extra K step: 1 in k = 0, 1, 2 of this key's row
                uint8_t* ones = sm.aug_ones + aug_off(kr);
                *reinterpret_cast<uint4*>(ones) = make_uint4(0x3F803F80u, 0x00003F80u, 0u, 0u);
                *reinterpret_cast<uint4*>(ones + 128) = make_uint4(0u, 0u, 0u, 0u);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.kv_tmem);
        }
        bool ok = true;
        bool s_ready = false;  // S^T of this step seen complete by an early poll
        for (int it = 0; it < nsteps; ++it) {
            const int q0 = (qb_lo + it % nq) * kBM;
            ok = __all_sync(0xffffffffu, s_ready || wait_phase(&sm.s_full, it & 1, flags, abort_word, P.wait_ns));
            if (!ok) break;
            tc_fence_after();
            float p[64];  // P^T for this key and query rows [64w, 64w+64)
            {
                uint32_t sv[64];
                tmem_ld64(tmem + lane_off + kColSdP + 64 * w, sv);
                tmem_ld_wait();
                // S^T is in registers: dP^T may now be written into the same columns
                tc_fence_before();
                mbar_arrive(&sm.s_loaded);
                // P = exp2((S - LSE / scale) * scale * log2 e), two columns per paired op
                const uint64_t sc2 = f2_pack(sc, sc);
#pragma unroll
                for (int j = 0; j < 64; j += 4) {
                    const uint32_t* src = sv + j;
                    const uint64_t a01 = f2_mul(f2_pack(__uint_as_float(src[0]), __uint_as_float(src[1])), sc2);
                    const uint64_t a23 = f2_mul(f2_pack(__uint_as_float(src[2]), __uint_as_float(src[3])), sc2);
                    float x0, x1, x2, x3;
                    f2_unpack(a01, x0, x1);
                    f2_unpack(a23, x2, x3);
                    p[j] = fast_exp2(x0);
                    p[j + 1] = fast_exp2(x1);
                    p[j + 2] = fast_exp2(x2);
                    p[j + 3] = fast_exp2(x3);
                }
            }
            // masks (boundary steps only): causal / window / past the sequence
            if (q0 + kBM > L ||
                (P.causal ? (k0 + kBN - 1 > q0 || (P.window > 0 && k0 < q0 + kBM - P.window))
                          : (k0 + kBN > L))) {
                // this key is seen by the query rows ip with ip >= kp (causal),
                // ip < kp + window and ip < L: as offsets j = ip - base from this
                // thread's first row, the interval [lo, hi), two compares per element
                const int base = q0 + 64 * w;
                int lo = 0, hi = L - base;
                if (P.causal) {
                    lo = kp - base;
                    if (P.window > 0) hi = min(hi, kp + P.window - base);
                } else if (kp >= L) {
                    hi = lo;
                }
                // which bounds can cut into this half step's 64 rows for some key
                // of the block (uniform over the warpgroup): on a window layer
                // most half steps need only one of them
                const bool need_lo = !P.causal || base < k0 + kBN - 1;
                const bool need_hi = !P.causal || base + 63 >= L ||
                                     (P.window > 0 && base + 63 >= k0 + P.window);
                if (need_lo && need_hi) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) p[j] = (j >= lo && j < hi) ? p[j] : 0.f;
                } else if (need_lo) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) p[j] = j >= lo ? p[j] : 0.f;
                } else if (need_hi) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) p[j] = j < hi ? p[j] : 0.f;
                }
            }
            // packed pairs: P^T in bf16 (tensor memory, A of dV), dS^T in f16 (tensor
            // memory, A of dK, and shared memory, A of dQ; their B operands Q and K
            // are f16 too): f16's 11 bits keep dQ and dK within tolerance when logits
            // are large
            uint32_t pp[32], pd[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) pp[j] = pack_bf16x2(p[2 * j], p[2 * j + 1]);
            ok = __all_sync(0xffffffffu, wait_phase(&sm.dp_full, it & 1, flags, abort_word, P.wait_ns));
            if (!ok) break;
            tc_fence_after();
            {
                uint32_t dv64[64];
                tmem_ld64(tmem + lane_off + kColSdP + 64 * w, dv64);
                // P^T and dS^T are read by the previous step's dV and dK products, and
                // this step's dS buffer by the dQ product of two steps back: poll their
                // barriers now, while the loads are in flight, and wait below if needed
                const bool pd_ready = it == 0 || mbar_test_wait(&sm.pd_free, (it - 1) & 1);
                const bool ds_ready = !kDq || it <= 1 || mbar_test_wait(&sm.ds_free[it & 1], ((it >> 1) - 1) & 1);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 64; j += 4) {
                    // dS = P (dP - delta), two columns per paired op (the MMA subtracted delta)
                    const uint32_t* d = dv64 + j;
                    const uint64_t t01 = f2_pack(__uint_as_float(d[0]), __uint_as_float(d[1]));
                    const uint64_t t23 = f2_pack(__uint_as_float(d[2]), __uint_as_float(d[3]));
                    float y0, y1, y2, y3;
                    f2_unpack(f2_mul(f2_pack(p[j], p[j + 1]), t01), y0, y1);
                    f2_unpack(f2_mul(f2_pack(p[j + 2], p[j + 3]), t23), y2, y3);
                    pd[j / 2] = pack_f16x2(y0, y1);
                    pd[j / 2 + 1] = pack_f16x2(y2, y3);
                }
                // dP^T has been read: the next step's S^T may overwrite the columns
                tc_fence_before();
                mbar_arrive(&sm.dp_loaded);
                if (it > 0) {
                    ok = __all_sync(0xffffffffu, pd_ready || wait_phase(&sm.pd_free, (it - 1) & 1, flags,
                                                                        abort_word, P.wait_ns));
                    if (!ok) break;
                }
                if (kDq && it > 1) {
                    ok = __all_sync(0xffffffffu, ds_ready || wait_phase(&sm.ds_free[it & 1],
                                                                        ((it >> 1) - 1) & 1, flags,
                                                                        abort_word, P.wait_ns));
                    if (!ok) break;
                }
            }
            // dS row of this key (f16): 64 query rows = 128 bytes of atom w (A operand
            // of dQ); written before the tensor-memory stores so that the proxy fence
            // below finds them done
            if (kDq) {
                uint8_t* atom = sm.ds[it & 1][w];
#pragma unroll
                for (int c16 = 0; c16 < 8; ++c16) {
                    const uint4 val = make_uint4(pd[4 * c16], pd[4 * c16 + 1], pd[4 * c16 + 2], pd[4 * c16 + 3]);
                    *reinterpret_cast<uint4*>(atom + sw128(kr, c16 * 16)) = val;
                }
            }
            tc_fence_after();
            tmem_st32(tmem + lane_off + kColP + 32 * w, pp);
            tmem_st32(tmem + lane_off + kColDS + 32 * w, pd);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            // poll the next step's S^T while the stores drain
            s_ready = it + 1 < nsteps && mbar_test_wait(&sm.s_full, (it + 1) & 1);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.ds_full);
        }
        // epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK (scaled). These
        // warps do not wait on every phase of grads_done, so a parity wait on it
        // could match a phase two steps back: the single-phase acc_done is used.
        if (ok) ok = __all_sync(0xffffffffu, wait_phase(&sm.acc_done, 0, flags, abort_word, P.wait_ns));
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
        if (kDq) {
        const int wq = warp - 12;
        const int r = wq * 32 + lane;  // query row within the step (tensor-memory lane)
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const bool issuer = warp == 12 && lane == 0;
        for (int it = 0; it < nsteps; ++it) {
            const int h = hk * P.group + it / nq;
            const int q0 = (qb_lo + it % nq) * kBM;
            // one decision for all four drain warps (they meet at named barriers below)
            if (!vote_all_128(1, wait_phase(&sm.grads_done, it & 1, flags, abort_word, P.wait_ns))) break;
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                // the previous reduce must have read the staging buffer
                if (issuer) bulk_wait_read<0>();
                named_barrier_sync(1, 128);
                uint32_t a[32];
                tmem_ld32(tmem + lane_off + kColDQ + 32 * half, a);
                tmem_ld_wait();
                if (half == 1) {
                    // the dQ columns have been read: the next dQ product may overwrite them
                    tc_fence_before();
                    mbar_arrive(&sm.dq_consumed);
                }
#pragma unroll
                for (int c16 = 0; c16 < 8; ++c16)
                    *reinterpret_cast<uint4*>(sm.dq_stage + sw128(r, c16 * 16)) =
                        make_uint4(a[4 * c16], a[4 * c16 + 1], a[4 * c16 + 2], a[4 * c16 + 3]);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                named_barrier_sync(1, 128);
                if (issuer) {
                    // rows past the sequence carry exact zeros (their dS is 0), so adding
                    // them into the next sequence's rows changes nothing
                    tma_reduce_add_3d(&tmDQ, sm.dq_stage, 32 * half, h, start + q0);
                    bulk_commit();
                }
            }
        }
        if (issuer) bulk_wait_all<0>();
        }  // kDq
    } else {
        regs_decrease<kCtlRegs>();
        if (warp == 8) {
            // -------------------------------------------------------- producer
            // (the K tile's load went out before the CTA barrier)
            // B tiles of the extra K step: only k = 0..3 of each row are rewritten per step
            for (int i = lane; i < (int)(kQStages * kAugTile / 16); i += 32) {
                reinterpret_cast<uint4*>(sm.aug_lse)[i] = make_uint4(0u, 0u, 0u, 0u);
                reinterpret_cast<uint4*>(sm.aug_delta)[i] = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();  // every lane's zeros land before any lane writes a row
            const float neg_inv_scale = -1.f / P.scale;
            int issued = 0;
            for (int it = 0; it < nsteps; ++it) {
                const int st = it % kQStages;
                const int h = hk * P.group + it / nq;
                const int q0 = (qb_lo + it % nq) * kBM;
                // test hook (off unless a test sets it): no load after the first step,
                // so the consumers' bounded waits run out
                if (P.withhold_load && it == 1) break;
                if (it >= kQStages &&
                    !__all_sync(0xffffffffu, wait_phase(&sm.q_empty[st], ((it / kQStages) - 1) & 1,
                                                        flags, abort_word, P.wait_ns)))
                    break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sm.q_full[st], 2 * kTileBytes);
                    tma_load_3d(sm.q[st], &tmQ, &sm.q_full[st], 0, h, start + q0);
                    tma_load_3d(sm.dout[st], &tmDO, &sm.q_full[st], 0, h, start + q0);
                }
                float lv[kBM / 32], dv_[kBM / 32];
#pragma unroll
                for (int u = 0; u < kBM / 32; ++u) {
                    const int c = lane * (kBM / 32) + u;
                    const int ip = min(q0 + c, L - 1);  // rows past the sequence are masked
                    const size_t ix = (size_t)h * P.total + start + ip;
                    lv[u] = __ldg(lse + ix);
                    dv_[u] = __ldg(delta + ix);
                }
#pragma unroll
                for (int u = 0; u < kBM / 32; ++u) {
                    const int c = lane * (kBM / 32) + u;
                    *reinterpret_cast<uint2*>(sm.aug_lse[st] + aug_off(c)) = split3_bf16(lv[u] * neg_inv_scale);
                    *reinterpret_cast<uint2*>(sm.aug_delta[st] + aug_off(c)) = split3_bf16(-dv_[u]);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(&sm.q_full[st]);
                issued = it + 1;
            }
            if (lane == 0) {
                drain_phase(&sm.k_full, 0, P.wait_ns);
                for (int it = max(0, issued - kQStages); it < issued; ++it)
                    drain_phase(&sm.q_full[it % kQStages], (it / kQStages) & 1, P.wait_ns);
            }
        } else if (warp == 9 && lane == 0) {
            // -------------------------------------------------------- MMA issuer 1: S^T, dP^T
            constexpr uint32_t idSS = idesc_bf16(kBN, kBM, 0, 0);  // A tmem, B K-major: bf16
            constexpr uint32_t idS16 = idesc_f16(kBN, kBM, 0, 0);  // the same in f16 (K, Q)
            const uint64_t dones = smem_desc_noswizzle(smem_u32(sm.aug_ones), kAugLBO, kAugSBO);
            bool ok = wait_phase(&sm.kv_tmem, 0, flags, abort_word, P.wait_ns) &&
                      wait_phase(&sm.q_full[0], 0, flags, abort_word, P.wait_ns);
            auto issue_s = [&](int st) {  // S^T - LSE / scale = K Q^T + ones (-LSE / scale)^T
                tc_fence_after();
                const uint64_t dq_ = smem_desc_sw128(smem_u32(sm.q[st]), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    mma_ts(tmem + kColSdP, tmem + kColK + kk * 8, dq_ + 2 * kk, idS16, kk > 0);
                mma_ss(tmem + kColSdP, dones, smem_desc_noswizzle(smem_u32(sm.aug_lse[st]), kAugLBO, kAugSBO),
                       idSS, 1);
                mma_commit(&sm.s_full);
            };
            if (ok) issue_s(0);
            for (int it = 0; ok && it < nsteps; ++it) {
                const int st = it % kQStages;
                const int st1 = (it + 1) % kQStages;
                // early poll of the next step's Q / dO stage (answer used after dP)
                const bool q_ready = it + 1 >= nsteps || mbar_test_wait(&sm.q_full[st1], ((it + 1) / kQStages) & 1);
                if (!(ok = wait_phase(&sm.s_loaded, it & 1, flags, abort_word, P.wait_ns))) break;
                // dP^T - delta = V dO^T + ones (-delta)^T, into the columns S^T was read from
                tc_fence_after();
                const uint64_t ddo = smem_desc_sw128(smem_u32(sm.dout[st]), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    mma_ts(tmem + kColSdP, tmem + kColV + kk * 8, ddo + 2 * kk, idSS, kk > 0);
                mma_ss(tmem + kColSdP, dones, smem_desc_noswizzle(smem_u32(sm.aug_delta[st]), kAugLBO, kAugSBO),
                       idSS, 1);
                mma_commit(&sm.dp_full);
                mma_commit(&sm.q_empty[st]);  // this issuer's last read of the step's Q / dO stage
                if (it + 1 < nsteps) {
                    if (!(ok = q_ready || wait_phase(&sm.q_full[st1], ((it + 1) / kQStages) & 1, flags,
                                                     abort_word, P.wait_ns)))
                        break;
                    if (!(ok = wait_phase(&sm.dp_loaded, it & 1, flags, abort_word, P.wait_ns))) break;
                    issue_s(st1);
                }
            }
            // every MMA issued above must finish before tensor memory is released
            mma_commit(&sm.drained[0]);
            drain_phase(&sm.drained[0], 0, P.wait_ns);
        } else if (warp == 10 && lane == 0) {
            // -------------------------------------------------------- MMA issuer 2: dV, dK, dQ
            constexpr uint32_t idG = idesc_bf16(kBN, kD, 0, 1);    // dV: A tmem, B MN-major, bf16
            constexpr uint32_t idG16 = idesc_f16(kBN, kD, 0, 1);   // dK: the same in f16
            constexpr uint32_t idQ = idesc_f16(kBM, kD, 1, 1);  // dQ: f16, A and B MN-major (smem)
            const uint64_t dKmn = smem_desc_sw128(smem_u32(sm.k), 1024, 1024);
            bool ok = wait_phase(&sm.k_full, 0, flags, abort_word, P.wait_ns);
            for (int j = 0; ok && j < nsteps; ++j) {
                const int st = j % kQStages;
                // dV += P^T dO, dK += dS^T Q  (K = query rows)
                if (!(ok = wait_phase(&sm.ds_full, j & 1, flags, abort_word, P.wait_ns))) break;
                tc_fence_after();
                const uint64_t ddo_mn = smem_desc_sw128(smem_u32(sm.dout[st]), 1024, 1024);
                const uint64_t dq_mn = smem_desc_sw128(smem_u32(sm.q[st]), 1024, 1024);
#pragma unroll
                for (int kk = 0; kk < kBM / 16; ++kk) {
                    const uint64_t boff = (uint64_t)((kk * 2048) >> 4);
                    mma_ts(tmem + kColDV, tmem + kColP + kk * 8, ddo_mn + boff, idG, j > 0 || kk > 0);
                    mma_ts(tmem + kColDK, tmem + kColDS + kk * 8, dq_mn + boff, idG16, j > 0 || kk > 0);
                }
                // P^T, dS^T and the step's Q / dO stage are no longer read
                mma_commit(&sm.pd_free);
                mma_commit(&sm.q_empty[st]);
                if (kDq) {
                    // dQ = dS K  (A = dS, MN-major: query rows contiguous, 2 atoms of 64)
                    if (j > 0) {
                        if (!(ok = wait_phase(&sm.dq_consumed, (j - 1) & 1, flags, abort_word, P.wait_ns))) break;
                        tc_fence_after();
                    }
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk) {
                        const uint64_t da = smem_desc_sw128(smem_u32(sm.ds[j & 1][0]) + kk * 2048, kBN * 128, 1024);
                        mma_ss(tmem + kColDQ, da, dKmn + (uint64_t)((kk * 2048) >> 4), idQ, kk > 0);
                    }
                    mma_commit(&sm.ds_free[j & 1]);
                    mma_commit(&sm.grads_done);
                }
            }
            if (ok) mma_commit(&sm.acc_done);
            mma_commit(&sm.drained[1]);
            drain_phase(&sm.drained[1], 0, P.wait_ns);
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

// The deterministic mode (Problem::deterministic) runs the split backward: this
// kernel without its dQ part for dK and dV, and the row-owning dQ kernel
// (tc_bwd_dq.cu), which sums each dQ row over its key blocks in tensor memory
// in a fixed order and writes it once, so dQ is reproducible bit for bit. It
// recomputes S and dP for dQ and is slower than the fused kernel, whose dQ
// blocks meet by reduce-adds in a run-dependent order.
static bool split_bwd(const Problem& P) { return P.deterministic != 0; }

// [dQ accumulator fp32 [T, h_q, 64] (fused only)][Q in f16 [T, h_q, 64]][K in f16 [T, h_kv, 64]]
// The accumulator's region is reserved in both backward modes (the split one
// does not add into it), so the workspace layout does not depend on the
// reproducible-dQ setting: a workspace prepared under one setting is laid out
// as the main call under the other expects.
static size_t acc_bytes(const Problem& P) { return sizeof(float) * (size_t)P.total * P.h_q * kD; }
static size_t q16_bytes(const Problem& P) { return 2 * (size_t)P.total * P.h_q * kD; }
static size_t k16_bytes(const Problem& P) { return 2 * (size_t)P.total * P.h_kv * kD; }

size_t tc_bwd_workspace_bytes(const Problem& P, bool bf16) {
    if (!bf16 || P.head_dim != kD) return 0;
    return acc_bytes(P) + q16_bytes(P) + k16_bytes(P);
}

template <bool kDq>
static cudaError_t launch_bwd_kernel(const Problem& P, const CUtensorMap& mq, const CUtensorMap& mk,
                                     const CUtensorMap& mdo, const CUtensorMap& mdq, const void* k16,
                                     const void* v, const float* lse, const float* delta, void* dk,
                                     void* dv, uint32_t* flags, cudaStream_t st) {
    // the register split is only safe at exactly this launch value
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, bwd_tc_kernel<kDq>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    const size_t smem = sizeof(BwdSmem) + 1024;
    e = cudaFuncSetAttribute(bwd_tc_kernel<kDq>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((P.max_seqlen + kBN - 1) / kBN, P.h_kv, P.nseq);
    bwd_tc_kernel<kDq><<<grid, kThreads, smem, st>>>(mq, mk, mdo, mdq, P, (const __nv_bfloat16*)k16,
                                                     (const __nv_bfloat16*)v, lse, delta,
                                                     (__nv_bfloat16*)dk, (__nv_bfloat16*)dv, flags);
    count_launches(1);
    return cudaGetLastError();
}

// Workspace of the 64-wide backward: [fp32 dQ accumulator][Q in f16][K in f16].
static void bwd_regions(const Problem& P, void* workspace, float*& acc, void*& q16, void*& k16) {
    acc = static_cast<float*>(workspace);
    q16 = static_cast<char*>(workspace) + acc_bytes(P);
    k16 = static_cast<char*>(q16) + q16_bytes(P);
}

// f16 copies of Q and K for the f16 products (the same 2-byte layout) and the
// fp32 dQ accumulator zeroed (only the fused kernel adds into it: zero_acc),
// in one memory-bound pass
static cudaError_t prepare_pass(const Problem& P, const void* q, const void* k, void* workspace,
                                bool zero_acc, cudaStream_t st) {
    float* acc;
    void *q16, *k16;
    bwd_regions(P, workspace, acc, q16, k16);
    const size_t n = (size_t)P.total * P.h_q * kD;
    return bwd_prepare(q, q16, n, k, k16, (size_t)P.total * P.h_kv * kD, acc, zero_acc ? n : 0, st);
}

// The pass on its own (sink_attn_bwd_prepare): the accumulator is zeroed
// whatever the reproducible-dQ setting, so the setting may change before the
// main call without leaving it dirty.
cudaError_t tc_bwd_prepare(const Problem& P, const void* q, const void* k, void* workspace,
                           cudaStream_t st) {
    if (P.nseq == 0 || P.max_seqlen == 0) return cudaSuccess;
    return prepare_pass(P, q, k, workspace, true, st);
}

cudaError_t tc_bwd(const Problem& P, const void* q, const void* k, const void* v,
                   const float* lse, const float* delta, const void* dout, void* dq, void* dk,
                   void* dv, uint32_t* flags, void* workspace, bool prepared, cudaStream_t st) {
    if (P.nseq == 0 || P.max_seqlen == 0) return cudaSuccess;
    const bool split = split_bwd(P);
    float* acc;
    void *q16, *k16;
    bwd_regions(P, workspace, acc, q16, k16);
    const size_t n = (size_t)P.total * P.h_q * kD;
    cudaError_t e = cudaSuccess;
    if (!prepared && (e = prepare_pass(P, q, k, workspace, !split, st)) != cudaSuccess) return e;
    CUtensorMap mq, mk, mv, mdo, mdq;
    if (!make_head_tile_map(&mq, q16, P.total, P.h_q, kBM) ||
        !make_head_tile_map(&mk, k16, P.total, P.h_kv, kBN) ||
        !make_head_tile_map(&mdo, dout, P.total, P.h_q, kBM))
        return cudaErrorInvalidValue;
    if (split) {
        if (!make_head_tile_map(&mv, v, P.total, P.h_kv, kBN)) return cudaErrorInvalidValue;
        e = launch_bwd_kernel<false>(P, mq, mk, mdo, mdo, k16, v, lse, delta, dk, dv, flags, st);
        if (e != cudaSuccess) return e;
        return tc_bwd_dq64(P, mk, mv, q16, dout, lse, delta, dq, flags, st);
    }
    if (!make_f32_head_half_map(&mdq, acc, P.total, P.h_q, kBM)) return cudaErrorInvalidValue;
    e = launch_bwd_kernel<true>(P, mq, mk, mdo, mdq, k16, v, lse, delta, dk, dv, flags, st);
    if (e != cudaSuccess) return e;
    const size_t n4 = n / 4;
    const int blocks = (int)std::min<size_t>((n4 + 255) / 256, 152 * 32);
    dq_convert_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(acc),
                                              reinterpret_cast<uint2*>(dq), n4, P.scale);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace sinkattn
