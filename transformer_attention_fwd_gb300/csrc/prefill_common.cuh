// prefill_common.cuh -- pieces shared by the tensor-core prefill kernels
// (prefill_bf16.cu and prefill_d64.cu): tile sizes, the snake order of work
// items over a persistent grid, the QK^T and P.V MMA groups and the waits
// used by the MMA warp and while draining after an abort.
#pragma once

#include <cstdint>

#include "sm100.cuh"

namespace attn {
namespace prefill {

constexpr int BM = 128;                  // query rows per tile = TMEM lanes
constexpr int BN = 128;                  // keys per K/V tile
constexpr int kBoxCols = 64;             // 64 bf16 = one 128-byte swizzle row
constexpr int kBoxBytes = kBoxCols * BM * 2;

// The k-th item of this CTA: the longest-first list is dealt in passes of
// gridDim.x items, alternating direction (snake order), which balances the
// causal work across CTAs without any global counter.  -1 when this CTA has
// no item in the (last, partial) pass k.
__device__ __forceinline__ int snake_item(int k, int n_items) {
    const int g = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    const int idx = k * g + ((k & 1) ? (g - 1 - c) : c);
    return idx < n_items ? idx : -1;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    const uint32_t s = smem_u32(p);
    return p + ((1024u - (s & 1023u)) & 1023u);
}

// The low word of a shared-memory descriptor holds the start address >> 4 in
// its low 14 bits.  Shared memory ends below 256 KB, so adding a byte offset
// >> 4 to the low word moves the start address without carrying into the
// other fields; this keeps each K step of an MMA group at one integer add.
__device__ __forceinline__ uint64_t desc_advance(uint64_t d, uint32_t off16) {
    const uint32_t lo = static_cast<uint32_t>(d) + off16;
    return (d & 0xFFFFFFFF00000000ull) | lo;
}

// S[tmem cols] = Q_tile . K_tile^T : M = 128, N = 128, K = D in steps of 16.
// K step kk reads columns 16kk .. 16kk+15: 64-column box kk/4, 32 bytes
// (kk%4) into each 128-byte row.  qd/kd: descriptors of the tiles' first box.
template <int D, bool kF16 = false>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t qd, uint64_t kd,
                                         uint32_t leader) {
    constexpr uint32_t idesc = mma_idesc_bf16_f32(BM, BN, false, false, kF16);
    constexpr int kSteps = D / 16;
    uint64_t a[kSteps], b[kSteps];
#pragma unroll
    for (int kk = 0; kk < kSteps; ++kk) {
        const uint32_t off16 = static_cast<uint32_t>(((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4);
        a[kk] = desc_advance(qd, off16);
        b[kk] = desc_advance(kd, off16);
    }
    if constexpr (kSteps == 8)
        mma_bf16_ss_x8(d_tmem, a, b, idesc, 0u, leader);
    else
        mma_bf16_ss_x4(d_tmem, a, b, idesc, 0u, leader);
}

// O[tmem cols] (+)= P . V_tile : M = 128, N = D, K = 128 keys in steps of 16.
// P is read from tensor memory (8 columns per 16 keys); V is MN-major, K step
// kk starts 16 key rows (2 KB) further.  vd: descriptor of the V tile.
// kExtra > 0: N = D + kExtra, the extra columns read from the 64-column atom
// at vd's leading-dimension offset (the box of ones).
template <int D, bool kF16 = false, int kExtra = 0>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint64_t vd,
                                         bool accumulate, uint32_t leader) {
    constexpr uint32_t idesc = mma_idesc_bf16_f32(BM, D + kExtra, false, true, kF16);
    uint32_t a[BN / 16];
    uint64_t b[BN / 16];
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
        a[kk] = p_tmem + kk * 8;
        b[kk] = desc_advance(vd, kk * (16 * 128 >> 4));
    }
    mma_bf16_ts_x8(o_tmem, a, b, idesc, accumulate ? 1u : 0u, leader);
}

// Wait without recording a timeout (used only while draining after an abort).
__device__ __forceinline__ void wait_quiet(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return;
    }
}

constexpr uint64_t kDrainLimitNs = 200ull * 1000ull * 1000ull;

// A wait taken by every lane of the MMA warp.  All lanes poll the same
// barrier in the same instructions, so they leave together; no vote is taken
// because warp votes (like elect.sync) wait for the warp's queued MMAs to be
// taken by the tensor pipe, while __syncwarp does not.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitGuard& g,
                                          unsigned site) {
    const bool ok = mbar_wait(bar, parity, g, site);
    __syncwarp();
    return ok;
}

}  // namespace prefill
}  // namespace attn
