// tc_common.cuh - pieces shared by the tensor-core kernels: bounded mbarrier
// waits driven by the global nanosecond timer, and the TMA tensor-map builder
// for [T, H, 64] bf16 tensors. The wait limit is a kernel argument
// (Problem::wait_ns, 2 s unless a test lowers it).
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace sinkattn {
namespace tc {

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase; on timeout raises the timeout flag and
// the CTA abort word. Returns false if the wait did not complete (timeout, or
// another role of the CTA already gave up).
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, uint32_t* flags,
                                           volatile int* abort_word, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_word) return false;
        if (now_ns() - t0 > limit_ns) {
            atomicOr(flags, kFlagTimeout);
            *abort_word = 1;
            return false;
        }
    }
}

// Time-bounded wait that ignores the abort word: used only to let copies or
// MMAs that were already issued finish before shared or tensor memory is
// given up.
__device__ __forceinline__ void drain_phase(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = now_ns();
    while (!mbar_try_wait(bar, parity) && now_ns() - t0 < limit_ns) {
    }
}

}  // namespace tc

// [T, H, dim] bf16 viewed as a 3-D tensor (d, head, token) with 128-byte
// swizzle; box = box_rows tokens x 1 head x 64 columns (dim = 64 or 128; a
// 128-wide row is fetched as two boxes). Returns false if the driver's encoder
// is unavailable or rejects the tensor.
bool make_head_tile_map(CUtensorMap* map, const void* base, int tokens, int heads, int box_rows,
                        int dim = 64);

// [T, H, 64] fp32 viewed the same way, box = box_rows tokens x 1 head x 32
// floats (128 bytes, 128-byte swizzle): used to reduce-add dQ blocks.
bool make_f32_head_half_map(CUtensorMap* map, void* base, int tokens, int heads, int box_rows);

}  // namespace sinkattn
