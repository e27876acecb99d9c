// tc_fwd.cu - sink-attention forward on the sm_103a tensor cores.
//
// What it computes (page "惊爆！GPT-OSS-20B强化学习，训练速度狂飙、超稳定！",
// sections "GPT-OSS中的带注意力槽的注意力机制" and "数学公式深入解读"): per row,
// softmax over the allowed scores plus the head's sink logit S_h, the sink
// column dropped before the product with V; plus the row's logsumexp with the
// sink included.
//
// Structure of one CTA: NT query tiles of 128 rows that share a key/value
// head (NT = 2 query heads of one GQA group when the group size is even), so
// every K/V tile fetched serves NT tiles.
//   warp 4*NT      TMA producer: Q tiles once, then K and V tiles of 128 keys
//                  through a kStages-deep ring of shared-memory buffers.
//   warp 4*NT+1+t  MMA issuer of tile t (one thread): S_t = Q_t K^T (SS, M=128
//                  N=128 K=64) into tensor memory, then O_t += P_t V (A = P_t
//                  read from tensor memory, M=128 N=64 K=128). S_t of the next
//                  key block is issued as soon as the softmax has read S_t
//                  into registers, so each tile's softmax runs back to back
//                  while the tensor pipe works on the next block and the other
//                  tile. One issuer per tile keeps a wait on one tile from
//                  holding back the other tile's products; a K/V stage is
//                  refilled once every tile's issuer is done with it.
//   warps 4t..4t+3 softmax of tile t: thread r owns row r (tensor-memory lane
//                  r). An online softmax over the keys (running max and sum);
//                  once every key is seen, the sink's term joins the
//                  denominator relative to the larger of the keys' max and the
//                  sink logit (fold_sink), and it contributes no value row.
//                  The max is only moved (and O rescaled in tensor memory)
//                  when it grows by more than kRescaleLog2 in log2 units; P
//                  values then stay below 2^kRescaleLog2 and the final O / l
//                  is unchanged.
// P V runs in f16, not bf16: P lies in [0, 2^kRescaleLog2], where f16 keeps
// 11 bits against bf16's 8, and the product's rounding of P is what limits the
// accuracy of O (and of D = dO . O in the backward) when logits are large. One
// product's A and B share a format, so V is read from an f16 copy that
// tc_fwd writes into the workspace first (convert.cu; exact for |V| <= 65504).
// Tensor memory (512 columns): S_t at t*128, O_t at 256 + t*64, P_t (f16
// pairs) at 384 + t*64. Every mbarrier wait is bounded; a wait that gives up
// sets the timeout flag and the CTA winds down without further work.
//
// Head dim D = 64 or 128. A tile of D columns is held as D/64 swizzle atoms
// of 128 rows x 64 (128-byte rows), each filled by its own TMA box; S takes
// D/16 K steps across the atoms, and P V is one N = D product per K step.
// At D = 128 a CTA holds one tile (NT = 1): S 128 + O 128 + P 64 columns.
//
// Two kernels share this structure. fwd_tc_kernel runs one row tile per
// query head of the CTA. fwd_tc_tiles_kernel (causal layers, D = 64) runs
// several consecutive row tiles per CTA, a count chosen per launch (two
// without a short window, 4 to 16 with a window of at most 256 keys); it
// writes each whole tile's O and o_lo through shared memory with one TMA
// store each, and tests per key block only the mask bound that can cut in.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace sinkattn {
namespace {

using namespace tc;

constexpr int kBM = 128;           // query rows per tile
constexpr int kBN = 128;           // keys per block
constexpr int kAtomCols = 64;      // head-dim columns per 128-byte swizzle atom
constexpr uint32_t kAtomBytes = kBM * kAtomCols * 2;  // 16 KB (kBM == kBN)
constexpr int kStages = 3;         // K/V ring depth
template <int D>
constexpr uint32_t tile_bytes() { return kBM * D * 2; }
constexpr float kRescaleLog2 = 8.0f;
// Register split for two tiles (384 threads launched at kLaunchRegs each):
// 2 softmax warpgroups x 128 x kSoftmaxRegs + 1 warpgroup x 128 x kOtherRegs
// = 53248 + 11264 = 64512 = 384 x 168.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 208;
constexpr int kOtherRegs = 88;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kOtherRegs <= 384 * kLaunchRegs, "register split");

template <int NT>
constexpr int fwd_threads() { return NT * 128 + 128; }

// Eight consecutive O values of a row, scaled by 1 / l: their bf16 (hi) and
// the bf16 of what that rounding dropped (lo = O - bf16(O), exact in fp32), so
// that o + o_lo carries about 16 bits of O.
__device__ __forceinline__ void pack_o8(const uint32_t* a, float inv, uint4& hi_out, uint4& lo_out) {
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = __uint_as_float(a[j]) * inv;
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) hi[j] = pack_bf16x2(x[2 * j], x[2 * j + 1]);
#pragma unroll
    for (int j = 0; j < 4; ++j)
        lo[j] = pack_bf16x2(x[2 * j] - __uint_as_float(hi[j] << 16),
                            x[2 * j + 1] - __uint_as_float(hi[j] & 0xFFFF0000u));
    hi_out = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    lo_out = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// Eight consecutive O values of a row, scaled by 1 / l, stored as bf16 at dst;
// when dst_lo is given, the bf16 of what that rounding dropped goes to dst_lo.
__device__ __forceinline__ void store_o8(uint4* dst, uint4* dst_lo, const uint32_t* a, float inv) {
    uint4 hi, lo;
    pack_o8(a, inv, hi, lo);
    *dst = hi;
    if (dst_lo) *dst_lo = lo;
}

// Byte offset of 16-byte chunk c of row r in a 128-row tile of 128-byte rows
// with the 128-byte swizzle (the layout of a TMA box of 64 bf16 x 128 rows).
__device__ __forceinline__ uint32_t sw128_chunk(int r, int c) {
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// The sink's term joins the row's denominator once every key has been seen:
// with the keys' running max m and sum l (log2 units, l relative to m) and the
// sink logit s2 = S_h log2 e, both parts are taken relative to M = max(m, s2):
//   l_tot = l 2^(m - M) + 2^(s2 - M),  O = acc 2^(m - M) / l_tot,
//   LSE = (M + log2 l_tot) ln 2.
// The sink adds no value row. Keeping it out of the running max keeps P (the
// operand of the f16 P V product) relative to the largest key, so a row whose
// sink dominates every key (P_ij ~ e^-30) still has P values f16 can hold.
// Returns the factor that turns acc into O; writes the row's LSE to *lse_out.
__device__ __forceinline__ float fold_sink(float m, float l, float s2, float* lse_out) {
    const float M = fmaxf(m, s2);
    const float a = m == -INFINITY ? 0.f : fast_exp2(m - M);
    const float st = s2 == -INFINITY ? 0.f : fast_exp2(s2 - M);
    const float lt = l * a + st;
    *lse_out = (M + __log2f(lt)) * kLn2;
    return lt > 0.f ? a / lt : 0.f;
}

template <int NT, int D>
struct FwdSmem {
    alignas(1024) __nv_bfloat16 q[NT][kBM * D];  // D/64 atoms of 128 rows x 64
    alignas(1024) __nv_bfloat16 k[kStages][kBN * D];
    alignas(1024) __nv_bfloat16 v[kStages][kBN * D];
    uint64_t q_full;
    uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
    uint64_t s_full[NT], s_loaded[NT], p_full[NT], o_done[NT];
    uint64_t exp_turn[NT];  // the two tiles' exponentials take turns (NT = 2)
    uint64_t drained[NT];
    uint32_t tmem_slot;
    int abort_flag;
};

static_assert(sizeof(FwdSmem<1, 128>) + 1024 <= 232448, "shared memory of the D = 128 forward");
static_assert(sizeof(FwdSmem<2, 64>) + 1024 <= 232448, "shared memory of the D = 64 forward");

template <int NT, int D>
__global__ void __launch_bounds__(fwd_threads<NT>(), 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const Problem P,
              const float* __restrict__ sinks, __nv_bfloat16* __restrict__ out,
              __nv_bfloat16* __restrict__ out_lo, float* __restrict__ lse, uint32_t* flags) {
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(D == 64 || NT == 1, "tensor memory holds one D = 128 tile");
    constexpr int kAtoms = D / kAtomCols;
    constexpr uint32_t kTileBytes = tile_bytes<D>();
    extern __shared__ uint8_t smem_raw[];
    FwdSmem<NT, D>& sm = *reinterpret_cast<FwdSmem<NT, D>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int rb = gridDim.x - 1 - blockIdx.x;  // longest tiles first
    const int seq = blockIdx.z;
    const int h0 = blockIdx.y * NT;
    int start, L;
    if (!seq_bounds_checked(P, seq, start, L, flags)) return;
    if (blockIdx.x == 0 && threadIdx.x == 0 && L > P.max_seqlen) atomicOr(flags, kFlagSeqTooLong);
    const int r0 = rb * kBM;
    if (r0 >= L) return;  // uniform for the whole CTA, before any barrier or TMEM use

    int kb_lo = 0, kb_hi = (L - 1) / kBN;
    if (P.causal) {
        kb_hi = rb;
        if (P.window > 0) kb_lo = max(0, r0 - P.window + 1) / kBN;
    }
    const int nblk = kb_hi - kb_lo + 1;
    const int hk = h0 / P.group;

    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.k_full[i], 1);
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.kv_empty[i], NT);  // one commit from each tile's MMA issuer
        }
        for (int t = 0; t < NT; ++t) {
            mbar_init(&sm.s_full[t], 1);
            mbar_init(&sm.s_loaded[t], 128);
            mbar_init(&sm.p_full[t], 128);
            mbar_init(&sm.o_done[t], 1);
            mbar_init(&sm.exp_turn[t], 128);
        }
        for (int t = 0; t < NT; ++t) mbar_init(&sm.drained[t], 1);
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc<512>(&sm.tmem_slot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // launched right after this call's conversion of V: its f16 copy is read below
    pdl_wait();
    const uint32_t tmem = sm.tmem_slot;
    volatile int* abort_word = &sm.abort_flag;

    if (warp < 4 * NT) {
        if (NT == 2) regs_increase<kSoftmaxRegs>();
        // ------------------------------------------------------------ softmax warpgroup t
        const int t = warp / 4;
        const int wq = warp % 4;
        const int r = wq * 32 + lane;
        const int h = h0 + t;
        const int row = r0 + r;
        const bool valid = row < L;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * 128;
        const uint32_t tO = tmem + lane_off + 256 + t * 64;
        const uint32_t tP = tmem + lane_off + 384 + t * 64;
        const float sc = P.scale_log2;
        const float sink2 = __ldg(sinks + h) * kLog2e;  // S_h in log2 units
        float m = -INFINITY;  // the keys' running max in log2 units
        float l = 0.f;        // the keys' running sum relative to m (the sink joins at the end)
        bool ok = true;
        for (int i = 0; i < nblk; ++i) {
            ok = __all_sync(0xffffffffu, wait_phase(&sm.s_full[t], i & 1, flags, abort_word, P.wait_ns));
            if (!ok) break;
            tc_fence_after();
            float s[128];
            {
                uint32_t a[128];
                tmem_ld128(tS, a);
                tmem_ld_wait();
                // S_t is in registers: the next block's S_t product may be issued
                tc_fence_before();
                mbar_arrive(&sm.s_loaded[t]);
#pragma unroll
                for (int j = 0; j < 128; ++j) s[j] = __uint_as_float(a[j]);
            }
            const int kp0 = (kb_lo + i) * kBN;  // first key position of the block
            const bool need_mask =
                P.causal ? (kp0 + kBN - 1 > r0 ||
                            (P.window > 0 && kp0 < r0 + kBM - P.window))
                         : (kp0 + kBN > L);
            if (need_mask) {
                const int lo = P.causal && P.window > 0 ? row - P.window + 1 : INT_MIN;
                const int hi = P.causal ? min(row, L - 1) : L - 1;
#pragma unroll
                for (int j = 0; j < 128; ++j) {
                    const int kp = kp0 + j;
                    if (kp < lo || kp > hi) s[j] = -INFINITY;
                }
            }
            // row max: three-input max, four independent chains
            float mx4[4] = {fmaxf(s[0], s[1]), fmaxf(s[2], s[3]), fmaxf(s[4], s[5]), fmaxf(s[6], s[7])};
#pragma unroll
            for (int j = 8; j < 128; j += 8) {
                mx4[0] = max3f(mx4[0], s[j], s[j + 1]);
                mx4[1] = max3f(mx4[1], s[j + 2], s[j + 3]);
                mx4[2] = max3f(mx4[2], s[j + 4], s[j + 5]);
                mx4[3] = max3f(mx4[3], s[j + 6], s[j + 7]);
            }
            const float smax = max3f(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]);
            const float mx = smax * sc;
            const bool upd = i == 0 ? mx > m : mx > m + kRescaleLog2;
            const float m_new = upd ? mx : m;
            const float corr = upd ? (m == -INFINITY ? 0.f : fast_exp2(m - m_new)) : 1.f;
            const float mref = m_new == -INFINITY ? 0.f : m_new;
            // p = exp2(s * sc - mref), two columns per paired op; row sum in pairs
            const uint64_t sc2 = f2_pack(sc, sc);
            const uint64_t nm2 = f2_pack(-mref, -mref);
            uint64_t rs2[4] = {0, 0, 0, 0};
            // With two tiles the exponentials alternate (tile 0 block i, tile 1 block
            // i, tile 0 block i+1, ...), so one tile's exp2 loop overlaps the other
            // tile's loads, max and stores instead of both competing for the
            // special-function units at once.
            if (NT == 2 && (t == 1 || i > 0)) {
                const int ph = t == 0 ? i - 1 : i;
                ok = __all_sync(0xffffffffu, wait_phase(&sm.exp_turn[t], ph & 1, flags, abort_word, P.wait_ns));
                if (!ok) break;
            }
            // P into registers first (f16 pairs): the exponentials overlap the
            // previous block's P V product, which still reads P_t and writes O_t
            uint32_t pk[64];
#pragma unroll
            for (int j = 0; j < 128; j += 2) {
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(s[j], s[j + 1]), sc2, nm2), x0, x1);
                const float p0 = fast_exp2(x0);
                const float p1 = fast_exp2(x1);
                rs2[(j >> 1) & 3] = f2_add(rs2[(j >> 1) & 3], f2_pack(p0, p1));
                pk[j >> 1] = pack_f16x2(p0, p1);
            }
            if (NT == 2) mbar_arrive(&sm.exp_turn[(1 - t) % NT]);
            if (i > 0) {
                ok = __all_sync(0xffffffffu,
                                wait_phase(&sm.o_done[t], (i - 1) & 1, flags, abort_word, P.wait_ns));
                if (!ok) break;
                tc_fence_after();
            }
            tmem_st64(tP, pk);
            float r0, r1, r2, r3, r4, r5, r6, r7;
            f2_unpack(rs2[0], r0, r1);
            f2_unpack(rs2[1], r2, r3);
            f2_unpack(rs2[2], r4, r5);
            f2_unpack(rs2[3], r6, r7);
            const float rs = ((r0 + r1) + (r2 + r3)) + ((r4 + r5) + (r6 + r7));
            if (i > 0 && __any_sync(0xffffffffu, upd)) {
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 64) {
                    uint32_t oa[32], ob[32];
                    tmem_ld32(tO + c0, oa);
                    tmem_ld32(tO + c0 + 32, ob);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        oa[j] = __float_as_uint(__uint_as_float(oa[j]) * corr);
                        ob[j] = __float_as_uint(__uint_as_float(ob[j]) * corr);
                    }
                    tmem_st32(tO + c0, oa);
                    tmem_st32(tO + c0 + 32, ob);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.p_full[t]);
            l = l * corr + rs;
            m = m_new;
        }
        if (ok)
            ok = __all_sync(0xffffffffu,
                            wait_phase(&sm.o_done[t], (nblk - 1) & 1, flags, abort_word, P.wait_ns));
        if (ok) {
            tc_fence_after();
            float row_lse;
            const float inv = fold_sink(m, l, sink2, &row_lse);
            const size_t ooff = ((size_t)(start + row) * P.h_q + h) * D;
            uint4* dst = reinterpret_cast<uint4*>(out + ooff);
            uint4* dst_lo = out_lo ? reinterpret_cast<uint4*>(out_lo + ooff) : nullptr;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 64) {
                // both loads complete before any register they write is read
                uint32_t oa[32], ob[32];
                tmem_ld32(tO + c0, oa);
                tmem_ld32(tO + c0 + 32, ob);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        store_o8(dst + c0 / 8 + j, dst_lo ? dst_lo + c0 / 8 + j : nullptr, oa + 8 * j, inv);
                        store_o8(dst + c0 / 8 + 4 + j, dst_lo ? dst_lo + c0 / 8 + 4 + j : nullptr, ob + 8 * j, inv);
                    }
                }
            }
            if (valid) lse[(size_t)h * P.total + start + row] = row_lse;
        }
        } else {
        if (NT == 2) regs_decrease<kOtherRegs>();
        if (warp == 4 * NT) {
            // ------------------------------------------------------------ TMA producer
            if (lane == 0) {
                tma_prefetch_desc(&tmQ);
                tma_prefetch_desc(&tmK);
                tma_prefetch_desc(&tmV);
                mbar_arrive_expect_tx(&sm.q_full, NT * kTileBytes);
                for (int t = 0; t < NT; ++t)
                    for (int a = 0; a < kAtoms; ++a)
                        tma_load_3d(sm.q[t] + a * kBM * kAtomCols, &tmQ, &sm.q_full, a * kAtomCols,
                                    h0 + t, start + r0);
                int issued = 0;
                for (int i = 0; i < nblk; ++i) {
                    const int st = i % kStages;
                    // test hook (off unless a test sets it): no load after the first
                    // stage, so the consumers' bounded waits run out
                    if (P.withhold_load && i == 1) break;
                    if (i >= kStages &&
                        !wait_phase(&sm.kv_empty[st], ((i / kStages) - 1) & 1, flags, abort_word, P.wait_ns))
                        break;
                    const int kpos = start + (kb_lo + i) * kBN;
                    mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
                    for (int a = 0; a < kAtoms; ++a)
                        tma_load_3d(sm.k[st] + a * kBN * kAtomCols, &tmK, &sm.k_full[st], a * kAtomCols,
                                    hk, kpos);
                    mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
                    for (int a = 0; a < kAtoms; ++a)
                        tma_load_3d(sm.v[st] + a * kBN * kAtomCols, &tmV, &sm.v_full[st], a * kAtomCols,
                                    hk, kpos);
                    issued = i + 1;
                }
                // copies still in flight must land before the CTA's shared memory goes away
                drain_phase(&sm.q_full, 0, P.wait_ns);
                for (int i = max(0, issued - kStages); i < issued; ++i) {
                    const int st = i % kStages;
                    drain_phase(&sm.k_full[st], (i / kStages) & 1, P.wait_ns);
                    drain_phase(&sm.v_full[st], (i / kStages) & 1, P.wait_ns);
                }
            }
        } else if (warp >= 4 * NT + 1 && warp <= 4 * NT + NT && lane == 0) {
            // ------------------------------------------------------------ MMA issuer of tile t
            const int t = warp - (4 * NT + 1);
            constexpr uint32_t idS = idesc_bf16(kBM, kBN, 0, 0);       // Q, K both K-major
            // P from TMEM, V MN-major with N = D: at D = 128 the two 64-column
            // atoms are 16 KB apart (the descriptor's leading byte offset)
            constexpr uint32_t idO = idesc_f16(kBM, D, 0, 1);  // P and V in f16
            const uint32_t tS = tmem + t * 128, tO = tmem + 256 + t * 64, tP = tmem + 384 + t * 64;
            // K step kk of S reads atom kk / 4 at byte offset 32 (kk % 4); both are
            // added to the descriptors' start-address field (16-byte units)
            const uint64_t dq = smem_desc_sw128(smem_u32(sm.q[t]), 16, 1024);
            auto s_product = [&](int stage) {
                const uint64_t dk = smem_desc_sw128(smem_u32(sm.k[stage]), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk / 4) * kAtomBytes) >> 4) + 2 * (kk % 4);
                    mma_ss(tS, dq + off, dk + off, idS, kk > 0);
                }
            };
            bool ok = wait_phase(&sm.q_full, 0, flags, abort_word, P.wait_ns) &&
                      wait_phase(&sm.k_full[0], 0, flags, abort_word, P.wait_ns);
            if (ok) {
                tc_fence_after();
                s_product(0);
                mma_commit(&sm.s_full[t]);
            }
            for (int i = 0; ok && i < nblk; ++i) {
                const int st = i % kStages;
                const int st1 = (i + 1) % kStages;
                if (i + 1 < nblk) {
                    // S_t(i+1) = Q_t K(i+1)^T as soon as S_t(i) has been read
                    if (!(ok = wait_phase(&sm.s_loaded[t], i & 1, flags, abort_word, P.wait_ns))) break;
                    if (!(ok = wait_phase(&sm.k_full[st1], ((i + 1) / kStages) & 1, flags, abort_word, P.wait_ns)))
                        break;
                    tc_fence_after();
                    s_product(st1);
                    mma_commit(&sm.s_full[t]);
                }
                // O_t += P_t(i) V(i)
                if (!(ok = wait_phase(&sm.p_full[t], i & 1, flags, abort_word, P.wait_ns))) break;
                if (!(ok = wait_phase(&sm.v_full[st], (i / kStages) & 1, flags, abort_word, P.wait_ns))) break;
                tc_fence_after();
                const uint64_t dv = smem_desc_sw128(smem_u32(sm.v[st]), kAtomBytes, 1024);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_ts(tO, tP + kk * 8, dv + (uint64_t)((kk * 16 * 128) >> 4), idO, (i > 0 || kk > 0));
                mma_commit(&sm.o_done[t]);
                // this tile's last reads of stage st (K(i) by S_t(i), V(i) by the product above)
                mma_commit(&sm.kv_empty[st]);
            }
            // every MMA issued above must finish before tensor memory is released
            mma_commit(&sm.drained[t]);
            drain_phase(&sm.drained[t], 0, P.wait_ns);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<512>(tmem);
    }
}

// ---------------------------------------------------------------- several row tiles per CTA
// A short window (at most 256 keys) leaves each row tile one or two key
// blocks, too little work to hide a CTA's start-up (tensor-memory allocation,
// first loads, pipeline fill) and its epilogue. fwd_tc_tiles_kernel runs
// several consecutive row tiles of the same query heads in one CTA (a launch
// parameter, fwd_tiles_per_cta below): the
// next tile's Q is loaded into the second Q buffer while the current tile
// computes, the K/V ring and the barrier phases run on across tiles (a block
// counter g), and each tile's first P V waits until the softmax has read the
// previous tile's O (o_free). It is the kernel above generalised to several
// tiles, for causal layers (with or without a window) at d = 64; with two
// tiles per CTA it is also faster than the one-tile kernel on a full causal
// layer of moderate length (one CTA's start-up and epilogue per two tiles).
// The one-tile kernel serves the other cases (no causal mask, an odd group,
// rows longer than kTwoTileMaxRows).

template <int NT>
struct FwdTilesSmem {
    alignas(1024) __nv_bfloat16 q[2][NT][kBM * 64];
    alignas(1024) __nv_bfloat16 k[kStages][kBN * 64];
    alignas(1024) __nv_bfloat16 v[kStages][kBN * 64];
    // tile t's normalised O and o_lo, staged for one TMA store each
    alignas(1024) __nv_bfloat16 o_stage[NT][2][kBM * 64];
    uint64_t q_full[2], q_empty[2];
    uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
    uint64_t s_full[NT], s_loaded[NT], p_full[NT], o_done[NT];
    uint64_t o_free[NT];    // the softmax has read O_t of its tile: the next tile may overwrite it
    uint64_t exp_turn[NT];  // the two tiles' exponentials take turns (NT = 2)
    uint64_t drained[NT];
    uint32_t tmem_slot;
    int abort_flag;
};
static_assert(sizeof(FwdTilesSmem<2>) + 1024 <= 232448, "shared memory of the multi-tile forward");

template <int NT>
__global__ void __launch_bounds__(fwd_threads<NT>(), 1)
fwd_tc_tiles_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
              const __grid_constant__ CUtensorMap tmOlo, const Problem P,
              const float* __restrict__ sinks, __nv_bfloat16* __restrict__ out,
              __nv_bfloat16* __restrict__ out_lo, float* __restrict__ lse, uint32_t* flags,
              const int tiles_per_cta) {
    constexpr int D = 64;
    constexpr int kQBufs = 2;
    constexpr int kAtoms = D / kAtomCols;
    constexpr uint32_t kTileBytes = tile_bytes<D>();
    extern __shared__ uint8_t smem_raw[];
    FwdTilesSmem<NT>& sm = *reinterpret_cast<FwdTilesSmem<NT>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cb = gridDim.x - 1 - blockIdx.x;  // longest tiles first
    const int seq = blockIdx.z;
    const int h0 = blockIdx.y * NT;
    int start, L;
    if (!seq_bounds_checked(P, seq, start, L, flags)) return;
    if (blockIdx.x == 0 && threadIdx.x == 0 && L > P.max_seqlen) atomicOr(flags, kFlagSeqTooLong);
    // this CTA's row tiles: row blocks rb0 .. rb0 + ntile - 1 of the sequence
    const int rb0 = cb * tiles_per_cta;
    const int ntile = min(tiles_per_cta, (L + kBM - 1) / kBM - rb0);
    if (rb0 * kBM >= L) return;  // uniform for the whole CTA, before any barrier or TMEM use
    // first row, first key block and number of key blocks of tile k
    auto tile_blocks = [&](int k, int& r0, int& kb_lo, int& nblk) {
        const int rb = rb0 + k;
        r0 = rb * kBM;
        kb_lo = 0;
        int kb_hi = (L - 1) / kBN;
        if (P.causal) {
            kb_hi = rb;
            if (P.window > 0) kb_lo = max(0, r0 - P.window + 1) / kBN;
        }
        nblk = kb_hi - kb_lo + 1;
    };
    const int hk = h0 / P.group;

    if (threadIdx.x == 0) {
        for (int b = 0; b < kQBufs; ++b) {
            mbar_init(&sm.q_full[b], 1);
            mbar_init(&sm.q_empty[b], NT);  // one commit from each tile's MMA issuer
        }
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.k_full[i], 1);
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.kv_empty[i], NT);  // one commit from each tile's MMA issuer
        }
        for (int t = 0; t < NT; ++t) {
            mbar_init(&sm.s_full[t], 1);
            mbar_init(&sm.s_loaded[t], 128);
            mbar_init(&sm.p_full[t], 128);
            mbar_init(&sm.o_done[t], 1);
            mbar_init(&sm.exp_turn[t], 128);
            mbar_init(&sm.o_free[t], 128);
        }
        for (int t = 0; t < NT; ++t) mbar_init(&sm.drained[t], 1);
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc<512>(&sm.tmem_slot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // launched right after this call's conversion of V: its f16 copy is read below
    pdl_wait();
    const uint32_t tmem = sm.tmem_slot;
    volatile int* abort_word = &sm.abort_flag;

    if (warp < 4 * NT) {
        if (NT == 2) regs_increase<kSoftmaxRegs>();
        // ------------------------------------------------------------ softmax warpgroup t
        const int t = warp / 4;
        const int wq = warp % 4;
        const int r = wq * 32 + lane;
        const int h = h0 + t;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * 128;
        const uint32_t tO = tmem + lane_off + 256 + t * 64;
        const uint32_t tP = tmem + lane_off + 384 + t * 64;
        const float sc = P.scale_log2;
        const float sink2 = __ldg(sinks + h) * kLog2e;
        bool ok = true;
        int g = 0;  // key blocks of this CTA so far: the barrier phases run on across its tiles
        for (int k = 0; ok && k < ntile; ++k) {
        int r0, kb_lo, nblk;
        tile_blocks(k, r0, kb_lo, nblk);
        const int row = r0 + r;
        const bool valid = row < L;
        float m = -INFINITY;  // the keys' running max in log2 units
        float l = 0.f;        // the keys' running sum relative to m (the sink joins at the end)
        for (int i = 0; i < nblk; ++i, ++g) {
            ok = __all_sync(0xffffffffu, wait_phase(&sm.s_full[t], g & 1, flags, abort_word, P.wait_ns));
            if (!ok) break;
            tc_fence_after();
            float s[128];
            {
                uint32_t a[128];
                tmem_ld128(tS, a);
                tmem_ld_wait();
                // S_t is in registers: the next block's S_t product may be issued
                tc_fence_before();
                mbar_arrive(&sm.s_loaded[t]);
#pragma unroll
                for (int j = 0; j < 128; ++j) s[j] = __uint_as_float(a[j]);
            }
            const int kp0 = (kb_lo + i) * kBN;  // first key position of the block
            const bool need_mask =
                P.causal ? (kp0 + kBN - 1 > r0 ||
                            (P.window > 0 && kp0 < r0 + kBM - P.window))
                         : (kp0 + kBN > L);
            if (need_mask) {
                // (this kernel runs causal layers only) a block needs the causal
                // bound only if it reaches past the tile's first row, and the
                // window bound only if it starts before the last row's window: on
                // a window layer most blocks need one of the two, tested alone
                const int lo = P.window > 0 ? row - P.window + 1 : INT_MIN;
                const int hi = min(row, L - 1);
                const bool need_hi = kp0 + kBN - 1 > r0;
                const bool need_lo = P.window > 0 && kp0 < r0 + kBM - P.window;
                if (need_hi && need_lo) {
#pragma unroll
                    for (int j = 0; j < 128; ++j)
                        if (kp0 + j < lo || kp0 + j > hi) s[j] = -INFINITY;
                } else if (need_hi) {
                    const int jh = hi - kp0;
#pragma unroll
                    for (int j = 0; j < 128; ++j)
                        if (j > jh) s[j] = -INFINITY;
                } else {
                    const int jl = lo - kp0;
#pragma unroll
                    for (int j = 0; j < 128; ++j)
                        if (j < jl) s[j] = -INFINITY;
                }
            }
            // row max: three-input max, four independent chains
            float mx4[4] = {fmaxf(s[0], s[1]), fmaxf(s[2], s[3]), fmaxf(s[4], s[5]), fmaxf(s[6], s[7])};
#pragma unroll
            for (int j = 8; j < 128; j += 8) {
                mx4[0] = max3f(mx4[0], s[j], s[j + 1]);
                mx4[1] = max3f(mx4[1], s[j + 2], s[j + 3]);
                mx4[2] = max3f(mx4[2], s[j + 4], s[j + 5]);
                mx4[3] = max3f(mx4[3], s[j + 6], s[j + 7]);
            }
            const float smax = max3f(fmaxf(mx4[0], mx4[1]), mx4[2], mx4[3]);
            const float mx = smax * sc;
            const bool upd = i == 0 ? mx > m : mx > m + kRescaleLog2;
            const float m_new = upd ? mx : m;
            const float corr = upd ? (m == -INFINITY ? 0.f : fast_exp2(m - m_new)) : 1.f;
            const float mref = m_new == -INFINITY ? 0.f : m_new;
            // p = exp2(s * sc - mref), two columns per paired op; row sum in pairs
            const uint64_t sc2 = f2_pack(sc, sc);
            const uint64_t nm2 = f2_pack(-mref, -mref);
            uint64_t rs2[4] = {0, 0, 0, 0};
            // With two tiles the exponentials alternate (tile 0 block i, tile 1 block
            // i, tile 0 block i+1, ...), so one tile's exp2 loop overlaps the other
            // tile's loads, max and stores instead of both competing for the
            // special-function units at once.
            if (NT == 2 && (t == 1 || g > 0)) {
                const int ph = t == 0 ? g - 1 : g;
                ok = __all_sync(0xffffffffu, wait_phase(&sm.exp_turn[t], ph & 1, flags, abort_word, P.wait_ns));
                if (!ok) break;
            }
            // P into registers first (f16 pairs): the exponentials overlap the
            // previous block's P V product, which still reads P_t and writes O_t
            uint32_t pk[64];
#pragma unroll
            for (int j = 0; j < 128; j += 2) {
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(s[j], s[j + 1]), sc2, nm2), x0, x1);
                const float p0 = fast_exp2(x0);
                const float p1 = fast_exp2(x1);
                rs2[(j >> 1) & 3] = f2_add(rs2[(j >> 1) & 3], f2_pack(p0, p1));
                pk[j >> 1] = pack_f16x2(p0, p1);
            }
            if (NT == 2) mbar_arrive(&sm.exp_turn[(1 - t) % NT]);
            if (g > 0) {
                // P_t V of the previous block (possibly the previous tile's) is done with P_t
                ok = __all_sync(0xffffffffu,
                                wait_phase(&sm.o_done[t], (g - 1) & 1, flags, abort_word, P.wait_ns));
                if (!ok) break;
                tc_fence_after();
            }
            tmem_st64(tP, pk);
            float r0, r1, r2, r3, r4, r5, r6, r7;
            f2_unpack(rs2[0], r0, r1);
            f2_unpack(rs2[1], r2, r3);
            f2_unpack(rs2[2], r4, r5);
            f2_unpack(rs2[3], r6, r7);
            const float rs = ((r0 + r1) + (r2 + r3)) + ((r4 + r5) + (r6 + r7));
            if (i > 0 && __any_sync(0xffffffffu, upd)) {
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 64) {
                    uint32_t oa[32], ob[32];
                    tmem_ld32(tO + c0, oa);
                    tmem_ld32(tO + c0 + 32, ob);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        oa[j] = __float_as_uint(__uint_as_float(oa[j]) * corr);
                        ob[j] = __float_as_uint(__uint_as_float(ob[j]) * corr);
                    }
                    tmem_st32(tO + c0, oa);
                    tmem_st32(tO + c0 + 32, ob);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&sm.p_full[t]);
            l = l * corr + rs;
            m = m_new;
        }
        // One decision for the tile's four warps, each of which reaches this
        // point even when it gave up inside the block loop: they meet at the
        // named barrier 1 + t below.
        ok = vote_all_128(1 + t, ok && wait_phase(&sm.o_done[t], (g - 1) & 1, flags, abort_word,
                                                  P.wait_ns));
        if (!ok) break;
        {
            tc_fence_after();
            float row_lse;
            const float inv = fold_sink(m, l, sink2, &row_lse);
            static_assert(D == 64, "the multi-tile forward is 64 wide");
            // both loads complete before any register they write is read
            uint32_t oa[32], ob[32];
            tmem_ld32(tO, oa);
            tmem_ld32(tO + 32, ob);
            tmem_ld_wait();
            // O_t is in registers: the next tile's first P V may overwrite it
            tc_fence_before();
            mbar_arrive(&sm.o_free[t]);
            if (r0 + kBM <= L) {
                // a whole tile of the sequence: O and o_lo through shared memory
                // and one TMA store each (rows leave as whole 128-byte lines
                // instead of a 16-byte piece per thread per row)
                uint8_t* so = reinterpret_cast<uint8_t*>(sm.o_stage[t][0]);
                uint8_t* sl = reinterpret_cast<uint8_t*>(sm.o_stage[t][1]);
                if (r == 0) bulk_wait_read<0>();  // the previous tile's stores have read them
                named_barrier_sync(1 + t, 128);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint4 hi, lo;
                    pack_o8(j < 4 ? oa + 8 * j : ob + 8 * (j - 4), inv, hi, lo);
                    *reinterpret_cast<uint4*>(so + sw128_chunk(r, j)) = hi;
                    *reinterpret_cast<uint4*>(sl + sw128_chunk(r, j)) = lo;
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                named_barrier_sync(1 + t, 128);
                if (r == 0) {
                    tma_store_3d(&tmO, so, 0, h, start + r0);
                    if (out_lo) tma_store_3d(&tmOlo, sl, 0, h, start + r0);
                    bulk_commit();
                }
                lse[(size_t)h * P.total + start + row] = row_lse;
            } else if (valid) {
                const size_t ooff = ((size_t)(start + row) * P.h_q + h) * D;
                uint4* dst = reinterpret_cast<uint4*>(out + ooff);
                uint4* dst_lo = out_lo ? reinterpret_cast<uint4*>(out_lo + ooff) : nullptr;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    store_o8(dst + j, dst_lo ? dst_lo + j : nullptr, oa + 8 * j, inv);
                    store_o8(dst + 4 + j, dst_lo ? dst_lo + 4 + j : nullptr, ob + 8 * j, inv);
                }
                lse[(size_t)h * P.total + start + row] = row_lse;
            }
        }
        }  // tiles
        // the staged tiles' stores complete before the CTA's shared memory goes away
        if (r == 0) bulk_wait_all<0>();
        } else {
        if (NT == 2) regs_decrease<kOtherRegs>();
        if (warp == 4 * NT) {
            // ------------------------------------------------------------ TMA producer
            if (lane == 0) {
                tma_prefetch_desc(&tmQ);
                tma_prefetch_desc(&tmK);
                tma_prefetch_desc(&tmV);
                int g = 0, issued = 0, q_issued = 0;
                bool ok = true;
                for (int k = 0; ok && k < ntile; ++k) {
                    int r0, kb_lo, nblk;
                    tile_blocks(k, r0, kb_lo, nblk);
                    const int qb = k % kQBufs;
                    // the buffer's previous tile: every S product that read it has completed
                    if (k >= kQBufs &&
                        !wait_phase(&sm.q_empty[qb], ((k / kQBufs) - 1) & 1, flags, abort_word, P.wait_ns))
                        break;
                    mbar_arrive_expect_tx(&sm.q_full[qb], NT * kTileBytes);
                    for (int t = 0; t < NT; ++t)
                        for (int a = 0; a < kAtoms; ++a)
                            tma_load_3d(sm.q[qb][t] + a * kBM * kAtomCols, &tmQ, &sm.q_full[qb],
                                        a * kAtomCols, h0 + t, start + r0);
                    q_issued = k + 1;
                    for (int i = 0; i < nblk; ++i, ++g) {
                        const int st = g % kStages;
                        // test hook (off unless a test sets it): no load after the
                        // CTA's first K/V stage, so the consumers' bounded waits run out
                        if (P.withhold_load && g == 1) {
                            ok = false;
                            break;
                        }
                        if (g >= kStages &&
                            !wait_phase(&sm.kv_empty[st], ((g / kStages) - 1) & 1, flags, abort_word, P.wait_ns)) {
                            ok = false;
                            break;
                        }
                        const int kpos = start + (kb_lo + i) * kBN;
                        mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
                        for (int a = 0; a < kAtoms; ++a)
                            tma_load_3d(sm.k[st] + a * kBN * kAtomCols, &tmK, &sm.k_full[st], a * kAtomCols,
                                        hk, kpos);
                        mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
                        for (int a = 0; a < kAtoms; ++a)
                            tma_load_3d(sm.v[st] + a * kBN * kAtomCols, &tmV, &sm.v_full[st], a * kAtomCols,
                                        hk, kpos);
                        issued = g + 1;
                    }
                }
                // copies still in flight must land before the CTA's shared memory goes away
                for (int k = max(0, q_issued - kQBufs); k < q_issued; ++k)
                    drain_phase(&sm.q_full[k % kQBufs], (k / kQBufs) & 1, P.wait_ns);
                for (int j = max(0, issued - kStages); j < issued; ++j) {
                    const int st = j % kStages;
                    drain_phase(&sm.k_full[st], (j / kStages) & 1, P.wait_ns);
                    drain_phase(&sm.v_full[st], (j / kStages) & 1, P.wait_ns);
                }
            }
        } else if (warp >= 4 * NT + 1 && warp <= 4 * NT + NT && lane == 0) {
            // ------------------------------------------------------------ MMA issuer of tile t
            const int t = warp - (4 * NT + 1);
            constexpr uint32_t idS = idesc_bf16(kBM, kBN, 0, 0);       // Q, K both K-major
            // P from TMEM, V MN-major with N = D: at D = 128 the two 64-column
            // atoms are 16 KB apart (the descriptor's leading byte offset)
            constexpr uint32_t idO = idesc_f16(kBM, D, 0, 1);  // P and V in f16
            const uint32_t tS = tmem + t * 128, tO = tmem + 256 + t * 64, tP = tmem + 384 + t * 64;
            // S_t = Q_t K^T from Q buffer qb and K stage st. K step kk reads atom
            // kk / 4 at byte offset 32 (kk % 4); both are added to the
            // descriptors' start-address field (16-byte units)
            const uint64_t dq0 = smem_desc_sw128(smem_u32(sm.q[0][t]), 16, 1024);
            const uint64_t dq1 = smem_desc_sw128(smem_u32(sm.q[kQBufs - 1][t]), 16, 1024);
            auto s_product = [&](int qb, int stage) {
                const uint64_t dq = qb == 0 ? dq0 : dq1;
                const uint64_t dk = smem_desc_sw128(smem_u32(sm.k[stage]), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk / 4) * kAtomBytes) >> 4) + 2 * (kk % 4);
                    mma_ss(tS, dq + off, dk + off, idS, kk > 0);
                }
            };
            int r0, kb_lo, nblk;
            tile_blocks(0, r0, kb_lo, nblk);
            bool ok = wait_phase(&sm.q_full[0], 0, flags, abort_word, P.wait_ns) &&
                      wait_phase(&sm.k_full[0], 0, flags, abort_word, P.wait_ns);
            if (ok) {
                tc_fence_after();
                s_product(0, 0);
                mma_commit(&sm.s_full[t]);
                if (nblk == 1) mma_commit(&sm.q_empty[0]);  // the tile's only S product
            }
            int g = 0;
            for (int k = 0; ok && k < ntile; ++k) {
                tile_blocks(k, r0, kb_lo, nblk);
                const int qb = k % kQBufs;
                for (int i = 0; i < nblk; ++i, ++g) {
                    const int st = g % kStages;
                    const int st1 = (g + 1) % kStages;
                    // S_t of the next block (of this tile, or the first of the next tile)
                    // as soon as S_t of this block has been read
                    const bool next_here = i + 1 < nblk;
                    if (next_here || k + 1 < ntile) {
                        if (!(ok = wait_phase(&sm.s_loaded[t], g & 1, flags, abort_word, P.wait_ns))) break;
                        int nqb = qb, last_of_tile = i + 2 == nblk;
                        if (!next_here) {
                            int nr0, nkb_lo, nnblk;
                            tile_blocks(k + 1, nr0, nkb_lo, nnblk);
                            nqb = (k + 1) % kQBufs;
                            last_of_tile = nnblk == 1;
                            if (!(ok = wait_phase(&sm.q_full[nqb], ((k + 1) / kQBufs) & 1, flags, abort_word, P.wait_ns)))
                                break;
                        }
                        if (!(ok = wait_phase(&sm.k_full[st1], ((g + 1) / kStages) & 1, flags, abort_word, P.wait_ns)))
                            break;
                        tc_fence_after();
                        s_product(nqb, st1);
                        mma_commit(&sm.s_full[t]);
                        // the last S product of a tile frees its Q buffer once it completes
                        if (last_of_tile) mma_commit(&sm.q_empty[nqb]);
                    }
                    // O_t += P_t(g) V(g); the first block of a tile overwrites O_t,
                    // which the softmax has read for the previous tile
                    if (!(ok = wait_phase(&sm.p_full[t], g & 1, flags, abort_word, P.wait_ns))) break;
                    if (!(ok = wait_phase(&sm.v_full[st], (g / kStages) & 1, flags, abort_word, P.wait_ns))) break;
                    if (i == 0 && k > 0 && !(ok = wait_phase(&sm.o_free[t], (k - 1) & 1, flags, abort_word, P.wait_ns)))
                        break;
                    tc_fence_after();
                    const uint64_t dv = smem_desc_sw128(smem_u32(sm.v[st]), kAtomBytes, 1024);
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        mma_ts(tO, tP + kk * 8, dv + (uint64_t)((kk * 16 * 128) >> 4), idO, (i > 0 || kk > 0));
                    mma_commit(&sm.o_done[t]);
                    // this tile's last reads of stage st (K(g) by S_t(g), V(g) by the product above)
                    mma_commit(&sm.kv_empty[st]);
                }
            }
            // every MMA issued above must finish before tensor memory is released
            mma_commit(&sm.drained[t]);
            drain_phase(&sm.drained[t], 0, P.wait_ns);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<512>(tmem);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

// [T, H, dim] bf16 viewed as a 3-D tensor (d, head, token); box = 64 columns
// (one 128-byte swizzle row) x 1 head x box_rows tokens.
bool make_head_tile_map(CUtensorMap* map, const void* base, int tokens, int heads, int box_rows,
                        int dim) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)dim * 2, (cuuint64_t)heads * dim * 2};
    cuuint32_t box[3] = {(cuuint32_t)kAtomCols, 1, (cuuint32_t)box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [T, H, 64] fp32 (the dQ accumulator) as (d, head, token) with 128-byte
// swizzle; box = box_rows tokens x 1 head x 32 floats (one 128-byte row).
bool make_f32_head_half_map(CUtensorMap* map, void* base, int tokens, int heads, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)heads, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {64 * 4, (cuuint64_t)heads * 64 * 4};
    cuuint32_t box[3] = {32, 1, (cuuint32_t)box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_fwd_supported(const Problem& P, bool bf16) {
    return bf16 && (P.head_dim == 64 || P.head_dim == 128) && encode_fn() != nullptr && P.total > 0;
}

// the f16 copy of V
size_t tc_fwd_workspace_bytes(const Problem& P, bool bf16) {
    return bf16 ? (size_t)P.total * P.h_kv * P.head_dim * 2 : 0;
}

// True if the compiled kernel uses exactly the register count its setmaxnreg
// split was sized for.
template <typename Kernel>
static bool launch_regs_ok(Kernel kernel) {
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, kernel) == cudaSuccess && fa.numRegs == kLaunchRegs;
}

template <int NT, int D>
static cudaError_t launch_fwd(const Problem& P, const CUtensorMap& mq, const CUtensorMap& mk,
                              const CUtensorMap& mv, const float* sinks, void* o, void* o_lo,
                              float* lse, uint32_t* flags, cudaStream_t st) {
    if (NT == 2) {
        // the register split above is only safe at exactly this launch value
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, fwd_tc_kernel<NT, D>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    }
    const size_t smem = sizeof(FwdSmem<NT, D>) + 1024;
    cudaError_t attr_err = cudaFuncSetAttribute(
        fwd_tc_kernel<NT, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (attr_err != cudaSuccess) return attr_err;
    dim3 grid((P.max_seqlen + kBM - 1) / kBM, P.h_q / NT, P.nseq);
    // right after the conversion of V (tc_fwd): may start while it finishes
    cudaError_t le = launch_after(fwd_tc_kernel<NT, D>, grid, dim3(fwd_threads<NT>()), smem, st, mq, mk, mv,
                                  P, sinks, (__nv_bfloat16*)o, (__nv_bfloat16*)o_lo, lse, flags);
    count_launches(1);
    return le != cudaSuccess ? le : cudaGetLastError();
}

// Row tiles per CTA of the multi-tile forward. Without a short window a tile
// has up to max_seqlen / 128 key blocks and two tiles per CTA measured best
// (four lengthened the causal 2 x 8192 forward by 5 %). With a window of at
// most 256 keys, more tiles spread a CTA's start-up over more work and fewer
// leave more, shorter CTAs to fill the last wave: the count minimises
// waves x (start-up + mean tiles per CTA) over 4, 8, 12 and 16, the start-up
// counted as one tile's time and every sequence taken at the mean length
// (cu_seqlens stays on the device); a tie goes to the larger count. A
// list-scheduling model of the launch ranks the counts the same way on the
// 4 x 8192 and the 48-sequence packed window layers, where the measured best
// were 8 and 16.
// Rows up to which a causal layer without a short window runs two tiles per
// CTA (measured: 2 x 8192 forward -1.1 %, 48 packed sequences of at most 8192
// -7.8 %, 1 x 32768 +1.5 %; the limit lies between the last two).
constexpr int kTwoTileMaxRows = 16384;

static int fwd_tiles_per_cta(const Problem& P, int nt) {
    if (P.window <= 0 || P.window > 2 * kBN) return 2;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        sms = 148;
    const long long mean_len = ((long long)P.total + P.nseq - 1) / P.nseq;
    const long long nrb = mean_len > 0 ? (mean_len + kBM - 1) / kBM : 1;
    const long long slices = (long long)(P.h_q / nt) * P.nseq;
    int best = 4;
    double best_est = 0.0;
    for (int t = 4; t <= 16; t += 4) {
        const long long per_seq = (nrb + t - 1) / t;
        const long long waves = (per_seq * slices + sms - 1) / sms;
        const double est = (double)waves * (1.0 + (double)nrb / (double)per_seq);
        if (t == 4 || est <= best_est) {
            best = t;
            best_est = est;
        }
    }
    return best;
}

template <int NT>
static cudaError_t launch_fwd_tiles(const Problem& P, const CUtensorMap& mq, const CUtensorMap& mk,
                                    const CUtensorMap& mv, const float* sinks, void* o, void* o_lo,
                                    float* lse, uint32_t* flags, cudaStream_t st) {
    if (NT == 2) {
        // the register split above is only safe at exactly this launch value
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, fwd_tc_tiles_kernel<NT>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    }
    const size_t smem = sizeof(FwdTilesSmem<NT>) + 1024;
    cudaError_t attr_err = cudaFuncSetAttribute(
        fwd_tc_tiles_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (attr_err != cudaSuccess) return attr_err;
    // the epilogue's store maps: [T, H_q, 64] O and o_lo, 128-row boxes
    CUtensorMap mo, mol;
    memset(&mo, 0, sizeof(mo));
    memset(&mol, 0, sizeof(mol));
    if (!make_head_tile_map(&mo, o, P.total, P.h_q, kBM) ||
        (o_lo && !make_head_tile_map(&mol, o_lo, P.total, P.h_q, kBM)))
        return cudaErrorInvalidValue;
    const int nrb = (P.max_seqlen + kBM - 1) / kBM;
    const int tiles = fwd_tiles_per_cta(P, NT);
    dim3 grid((nrb + tiles - 1) / tiles, P.h_q / NT, P.nseq);
    cudaError_t le = launch_after(fwd_tc_tiles_kernel<NT>, grid, dim3(fwd_threads<NT>()), smem, st, mq, mk,
                                  mv, mo, mol, P, sinks, (__nv_bfloat16*)o, (__nv_bfloat16*)o_lo, lse, flags,
                                  tiles);
    count_launches(1);
    return le != cudaSuccess ? le : cudaGetLastError();
}

cudaError_t tc_fwd(const Problem& P, const void* q, const void* k, const void* v,
                   const float* sinks, void* o, void* o_lo, float* lse, uint32_t* flags,
                   void* workspace, cudaStream_t st) {
    if (P.nseq == 0 || P.max_seqlen == 0) return cudaSuccess;
    // V in f16 for the P V product (the same 2-byte layout; TMA copies bytes)
    void* v16 = workspace;
    // (the conversion also zeroes the workspace's flag word for the forward)
    cudaError_t e = convert_bf16_to_f16(v, v16, (size_t)P.total * P.h_kv * P.head_dim, st, flags);
    if (e != cudaSuccess) return e;
    CUtensorMap mq, mk, mv;
    if (!make_head_tile_map(&mq, q, P.total, P.h_q, kBM, P.head_dim) ||
        !make_head_tile_map(&mk, k, P.total, P.h_kv, kBN, P.head_dim) ||
        !make_head_tile_map(&mv, v16, P.total, P.h_kv, kBN, P.head_dim))
        return cudaErrorInvalidValue;
    if (P.head_dim == 128) return launch_fwd<1, 128>(P, mq, mk, mv, sinks, o, o_lo, lse, flags, st);
    // The two-tile kernels split their registers (setmaxnreg) and run only if
    // the compiler gave them exactly kLaunchRegs; otherwise the one-tile kernel
    // of the same kind (no split) computes the same result.
    const bool pair = P.group % 2 == 0;
    if (P.causal && P.window > 0 && P.window <= 2 * kBN) {
        if (pair && launch_regs_ok(fwd_tc_tiles_kernel<2>))
            return launch_fwd_tiles<2>(P, mq, mk, mv, sinks, o, o_lo, lse, flags, st);
        return launch_fwd_tiles<1>(P, mq, mk, mv, sinks, o, o_lo, lse, flags, st);
    }
    // Causal rows of up to kTwoTileMaxRows: two row tiles per CTA in the
    // multi-tile kernel. Longer rows make a two-tile CTA long enough that the
    // launch's tail grows more than the shared start-up saves.
    if (P.causal && pair && P.max_seqlen <= kTwoTileMaxRows && launch_regs_ok(fwd_tc_tiles_kernel<2>))
        return launch_fwd_tiles<2>(P, mq, mk, mv, sinks, o, o_lo, lse, flags, st);
    if (pair && launch_regs_ok(fwd_tc_kernel<2, 64>))
        return launch_fwd<2, 64>(P, mq, mk, mv, sinks, o, o_lo, lse, flags, st);
    return launch_fwd<1, 64>(P, mq, mk, mv, sinks, o, o_lo, lse, flags, st);
}

}  // namespace sinkattn
