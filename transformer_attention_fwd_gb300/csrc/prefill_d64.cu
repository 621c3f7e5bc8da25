// prefill_d64.cu -- bf16 (or fp16) attention forward for head dim 64 on the
// 5th-generation tensor cores, two CTAs per SM, one 128-row query tile per
// work item.
//
// The method is the tiled attention with online softmax of
// "3.3 Self-Attention机制深入理解" §12.2/§12.3 (walk the key/value tiles of a
// query tile, fold each S = Q K^T tile into a running row maximum and row
// sum, accumulate P V), with the causal tile classes of "第 11 章 · Attention
// 入门" §11.8.3 (tiles above the diagonal are never visited, tiles across it
// are masked) and the GQA head map of §11.8.1 (query head hq reads K/V head
// hq / (Hq / Hkv)).  A runtime window > 0 keeps only each row's most recent
// keys (§11.8.4).
//
// Why a kernel of its own for D = 64: at D = 64 a key tile's two MMAs are
// shorter than its softmax, and short problems (GPT-2-small: 2.5 work items
// per SM of 1..8 key tiles each) spend much of their time in per-item costs:
// the first tile, the diagonal tile and the epilogue.  Here every SM runs two
// independent CTAs, so one CTA's per-item costs overlap the other's steady
// tiles, and within a CTA the next QK^T overlaps the current softmax:
//
// Tensor memory (256 of the SM's 512 columns per CTA): S (fp32, 128 columns)
// at 0, P (packed 16-bit pairs, 64 columns) at 128, O (fp32, 64 columns) at
// 192.  P does not alias S, so QK^T of key tile j+1 is issued as soon as the
// softmax has read S(j) into registers, and runs while the softmax computes
// the weights of tile j.  The order on the tensor pipe is
//     QK(j+1)  PV(j)  QK(j+2)  PV(j+1) ...
// and across items the next item's first QK^T precedes the last P.V of the
// current one.
//
// Warps (256 threads, __launch_bounds__(256, 2)):
//   warp 0      TMA producer for Q and K tiles        (one lane)
//   warp 3      TMA producer for V tiles              (one lane)
//   warp 1      MMA issuer (whole warp, converged; one stored leader lane)
//   warp 2      tensor-memory allocator
//   warps 4-7   softmax and epilogue: warp w owns TMEM lane quarter w % 4,
//               one query row per thread, all 128 keys of a tile in registers
// The producers pull the next item's first Q, K and V tiles into L2 while the
// current item runs.  The epilogue stages each warp's 32 rows of O in the
// item's Q buffer and writes them with one TMA store.
//
// Softmax per tile, per row (base 2, x = s * scale * log2 e): the row maximum
// of the tile's visible scores is taken every tile; the running reference m
// moves only when that maximum exceeds m by more than 8, so weights
// 2^(x - m) stay below 2^8 (finite in bf16 and fp16 alike) and O is rarely
// rescaled.  Keys are classified per 32-key chunk for the whole warp (all
// visible, none visible, or some): only chunks crossing a row's limit are
// masked element-wise, and chunks no row of the warp sees are weighted against
// an offset of -inf, which gives exact zeros.
#include <cuda.h>
#include <cuda_runtime.h>
#include <climits>
#include <cmath>
#include <cstdint>

#include "attn_internal.h"
#include "prefill_common.cuh"
#include "sm100.cuh"

namespace attn {
namespace {

using namespace prefill;

constexpr int D = 64;
constexpr int kThreads = 256;
constexpr int kTileBytes = kBoxBytes;  // 128 rows x 64 columns of 16-bit values
constexpr int kQStages = 2, kKStages = 2, kVStages = 2;
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kQStages * kTileBytes;
constexpr int kVOff = kKOff + kKStages * kTileBytes;
constexpr int kBarOff = kVOff + kVStages * kTileBytes;
constexpr int kBarBytes = 256;
constexpr int kSmemBytes = kBarOff + kBarBytes + 1024;  // + 1024-byte alignment slack
static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs must fit in one SM's shared memory");
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColP = 128, kColO = 192;
constexpr float kLn2 = 0.6931471805599453f;
// The running reference moves only when a tile's row maximum exceeds it by
// more than this many powers of two.
constexpr float kRescaleThreshold = 8.0f;

// Register split (setmaxnreg): two CTAs of 256 threads share the SM's 65536
// registers, 128 a thread at launch; the four control warps drop to 56 and the
// four softmax warps rise to 200: 128 x 56 + 128 x 200 = 32768 = 256 x 128.
constexpr int kCtrlRegs = 56;
constexpr int kSoftmaxRegs = 200;
static_assert(128 * kCtrlRegs + 128 * kSoftmaxRegs <= kThreads * 128, "register split too large");

// Wait sites reported in the status word when a wait times out (numbered
// after the other prefill kernel's).
enum : unsigned {
    SITE_Q_EMPTY = 32, SITE_K_EMPTY, SITE_V_EMPTY, SITE_Q_FULL, SITE_K_FULL, SITE_V_FULL,
    SITE_S_FULL, SITE_S_FREE, SITE_P_FULL, SITE_PV_DONE, SITE_O_FREE
};

struct Bars {
    uint64_t q_full[kQStages], q_empty[kQStages];
    uint64_t k_full[kKStages], k_empty[kKStages];
    uint64_t v_full[kVStages], v_empty[kVStages];
    uint64_t s_full;   // QK^T of the current tile is in S          (MMA commit)
    uint64_t s_free;   // the softmax has read S into registers     (4 warps)
    uint64_t p_full;   // P is written (and O rescaled if needed)   (4 warps)
    uint64_t pv_done;  // the last P.V has completed                (MMA commit)
    uint64_t o_free;   // the epilogue has read O out               (4 warps)
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= kBarBytes, "barrier block too large");

struct Params {
    uint16_t* o;
    float* lse;
    int Hq, Hkv, Tq, Tk, group, causal;
    int window;  // > 0: each row also drops keys more than window-1 before its own
    float scale_log2;
    int n_qtiles, n_bh, n_items;
    unsigned* status;
    unsigned long long limit_ns;
};

// A work item: query tile qt (128 rows) of head bh of the [B*Hq] planes; it
// reads K/V plane bkv and visits key tiles lo .. n-1.
struct Item {
    int bh, qt, bkv, lo, n;
};

// Items are numbered from the last query tile (the longest under the causal
// mask) to the first, heads fastest, so heads that share a K/V head are
// neighbours and the snake order deals the longest items first.
__device__ __forceinline__ Item decode_item(int idx, const Params& p) {
    Item it;
    const int qrev = idx / p.n_bh;
    it.bh = idx - qrev * p.n_bh;
    it.qt = p.n_qtiles - 1 - qrev;
    const int b = it.bh / p.Hq, hq = it.bh - b * p.Hq;
    it.bkv = b * p.Hkv + hq / p.group;
    const int r0 = it.qt * BM;
    const int off = p.Tk - p.Tq;
    it.lo = 0;
    if (p.window > 0) {
        const int first_key = r0 + off - p.window + 1;  // of row r0
        it.lo = first_key > 0 ? first_key / BN : 0;
    }
    if (p.causal) {
        const int rlast = min(r0 + BM - 1, p.Tq - 1);
        it.n = min(p.Tk - 1, rlast + off) / BN + 1;
    } else {
        it.n = (p.Tk + BN - 1) / BN;
    }
    return it;
}

// ----------------------------------------------------------------------------
// Roles
// ----------------------------------------------------------------------------
__device__ void producer_qk(const CUtensorMap* tmQ, const CUtensorMap* tmK, uint8_t* smem,
                            Bars* bars, const Params& p, const WaitGuard& g) {
    uint32_t q_it = 0, k_it = 0;
    for (int k = 0; k * static_cast<int>(gridDim.x) < p.n_items; ++k) {
        const int idx = snake_item(k, p.n_items);
        if (idx < 0) continue;
        const Item it = decode_item(idx, p);
        const int qs = q_it % kQStages;
        if (q_it >= (uint32_t)kQStages &&
            !mbar_wait(&bars->q_empty[qs], ((q_it / kQStages) & 1) ^ 1, g, SITE_Q_EMPTY))
            goto drain;
        mbar_arrive_expect_tx(&bars->q_full[qs], kTileBytes);
        tma_load_3d(smem + kQOff + qs * kTileBytes, tmQ, &bars->q_full[qs], 0, it.qt * BM, it.bh);
        ++q_it;
        // Pull the next item's Q and first K tile into L2 meanwhile.
        const int nx_idx = snake_item(k + 1, p.n_items);
        if (nx_idx >= 0) {
            const Item nx = decode_item(nx_idx, p);
            tma_prefetch_l2_3d(tmQ, 0, nx.qt * BM, nx.bh);
            tma_prefetch_l2_3d(tmK, 0, nx.lo * BN, nx.bkv);
        }
        for (int j = it.lo; j < it.n; ++j, ++k_it) {
            const int s = k_it % kKStages;
            if (k_it >= (uint32_t)kKStages &&
                !mbar_wait(&bars->k_empty[s], ((k_it / kKStages) & 1) ^ 1, g, SITE_K_EMPTY))
                goto drain;
            mbar_arrive_expect_tx(&bars->k_full[s], kTileBytes);
            tma_load_3d(smem + kKOff + s * kTileBytes, tmK, &bars->k_full[s], 0, j * BN, it.bkv);
        }
    }
    return;
drain:
    // Let copies already in flight land before the CTA leaves.
    for (uint32_t i = (q_it > (uint32_t)kQStages ? q_it - kQStages : 0); i < q_it; ++i)
        wait_quiet(&bars->q_full[i % kQStages], (i / kQStages) & 1, kDrainLimitNs);
    for (uint32_t i = (k_it > (uint32_t)kKStages ? k_it - kKStages : 0); i < k_it; ++i)
        wait_quiet(&bars->k_full[i % kKStages], (i / kKStages) & 1, kDrainLimitNs);
}

__device__ void producer_v(const CUtensorMap* tmV, uint8_t* smem, Bars* bars, const Params& p,
                           const WaitGuard& g) {
    uint32_t v_it = 0;
    for (int k = 0; k * static_cast<int>(gridDim.x) < p.n_items; ++k) {
        const int idx = snake_item(k, p.n_items);
        if (idx < 0) continue;
        const Item it = decode_item(idx, p);
        const int nx_idx = snake_item(k + 1, p.n_items);
        if (nx_idx >= 0) {  // the next item's first V tile into L2 meanwhile
            const Item nx = decode_item(nx_idx, p);
            tma_prefetch_l2_3d(tmV, 0, nx.lo * BN, nx.bkv);
        }
        for (int j = it.lo; j < it.n; ++j, ++v_it) {
            const int s = v_it % kVStages;
            if (v_it >= (uint32_t)kVStages &&
                !mbar_wait(&bars->v_empty[s], ((v_it / kVStages) & 1) ^ 1, g, SITE_V_EMPTY))
                goto drain;
            mbar_arrive_expect_tx(&bars->v_full[s], kTileBytes);
            tma_load_3d(smem + kVOff + s * kTileBytes, tmV, &bars->v_full[s], 0, j * BN, it.bkv);
        }
    }
    return;
drain:
    for (uint32_t i = (v_it > (uint32_t)kVStages ? v_it - kVStages : 0); i < v_it; ++i)
        wait_quiet(&bars->v_full[i % kVStages], (i / kVStages) & 1, kDrainLimitNs);
}

// The MMA warp walks the key tiles of all its items as one sequence.  For
// each tile it issues QK^T into S once the softmax has read the previous S,
// then the P.V of the previous tile once its P is written.
template <bool kF16>
__device__ void mma_issuer(uint8_t* smem, Bars* bars, uint32_t tmem, const Params& p,
                           const WaitGuard& g) {
    constexpr uint32_t kTile16 = kTileBytes >> 4;  // one tile in descriptor units
    const uint64_t q_desc0 = smem_desc_sw128(smem_u32(smem + kQOff), 16, 1024);
    const uint64_t k_desc0 = smem_desc_sw128(smem_u32(smem + kKOff), 16, 1024);
    const uint64_t v_desc0 = smem_desc_sw128(smem_u32(smem + kVOff), kBoxBytes, 1024);
    uint32_t q_it = 0, k_it = 0, v_it = 0, s_cnt = 0, p_cnt = 0, o_cnt = 0;
    // The P.V still to issue: the previous tile's (first / last tile of its item).
    bool pending = false, pend_first = false, pend_last = false;
    const uint32_t leader = elect_leader();

    auto issue_pending_pv = [&]() -> bool {
        if (!warp_wait(&bars->p_full, p_cnt & 1, g, SITE_P_FULL)) return false;
        ++p_cnt;
        const uint32_t vs = v_it % kVStages;
        if (!warp_wait(&bars->v_full[vs], (v_it / kVStages) & 1, g, SITE_V_FULL)) return false;
        // An item's first P.V overwrites O: the previous item's epilogue must
        // have read it out.
        if (pend_first && o_cnt > 0 && !warp_wait(&bars->o_free, (o_cnt - 1) & 1, g, SITE_O_FREE))
            return false;
        tc_fence_after_sync();
        issue_pv<D, kF16>(tmem + kColO, tmem + kColP, desc_advance(v_desc0, vs * kTile16),
                          !pend_first, leader);
        mma_commit(&bars->pv_done, leader);
        mma_commit(&bars->v_empty[vs], leader);
        ++v_it;
        if (pend_last) ++o_cnt;
        return true;
    };

    for (int k = 0; k * static_cast<int>(gridDim.x) < p.n_items; ++k) {
        const int idx = snake_item(k, p.n_items);
        if (idx < 0) continue;
        const Item it = decode_item(idx, p);
        const uint32_t qs = q_it % kQStages;
        if (!warp_wait(&bars->q_full[qs], (q_it / kQStages) & 1, g, SITE_Q_FULL)) goto drain;
        ++q_it;
        const uint64_t q_desc = desc_advance(q_desc0, qs * kTile16);
        for (int j = it.lo; j < it.n; ++j) {
            const uint32_t ks = k_it % kKStages;
            if (!warp_wait(&bars->k_full[ks], (k_it / kKStages) & 1, g, SITE_K_FULL)) goto drain;
            if (s_cnt > 0 && !warp_wait(&bars->s_free, (s_cnt - 1) & 1, g, SITE_S_FREE)) goto drain;
            tc_fence_after_sync();
            issue_qk<D, kF16>(tmem + kColS, q_desc, desc_advance(k_desc0, ks * kTile16), leader);
            mma_commit(&bars->s_full, leader);
            mma_commit(&bars->k_empty[ks], leader);
            ++k_it;
            ++s_cnt;
            if (pending && !issue_pending_pv()) goto drain;
            pending = true;
            pend_first = (j == it.lo);
            pend_last = (j == it.n - 1);
        }
    }
    if (pending) issue_pending_pv();
drain:
    // Wait for every MMA issued so far before tensor memory is released.
    mma_commit(&bars->drain, leader);
    wait_quiet(&bars->drain, 0, kDrainLimitNs);
}

// Row maximum of 32 scores (two interleaved 3-input max chains).
__device__ __forceinline__ float chunk_max(const uint32_t* s) {
    float a = fmaxf(__uint_as_float(s[0]), __uint_as_float(s[1]));
    float b = fmaxf(__uint_as_float(s[2]), __uint_as_float(s[3]));
#pragma unroll
    for (int i = 4; i < 32; i += 4) {
        a = fmax3(a, __uint_as_float(s[i]), __uint_as_float(s[i + 1]));
        b = fmax3(b, __uint_as_float(s[i + 2]), __uint_as_float(s[i + 3]));
    }
    return fmaxf(a, b);
}

// Weights of 32 scores against the reference: p receives 16 packed pairs
// (keys 2i, 2i+1 in pair i), acc_e the exact sums (two packed accumulators),
// acc_r the sums of the rounded weights.
template <bool kF16>
__device__ __forceinline__ void chunk_exp2(const uint32_t* s, uint64_t sc2, uint64_t nm2,
                                           uint32_t* p, uint64_t (&acc_e)[2],
                                           float (&acc_r)[4]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint64_t x2 =
            f2_fma(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), sc2, nm2);
        float x0, x1;
        f2_unpack(x2, x0, x1);
        const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
        const uint32_t pk = Elem16<kF16>::pack(e0, e1);
        acc_e[i & 1] = f2_add(acc_e[i & 1], f2_pack(e0, e1));
        Elem16<kF16>::add2(pk, acc_r[2 * (i & 1)], acc_r[2 * (i & 1) + 1]);
        p[i] = pk;
    }
}

// Softmax warps 4-7: one query row per thread.  Per key tile: read S, release
// it to the MMA warp, take the row maximum of the visible keys, move the
// reference if needed (rescaling O after the previous P.V has landed), write
// the weights P and release them to the MMA warp.  Per item: the epilogue
// O / sum -> 16-bit output and lse.
template <bool kF16>
__device__ void softmax_rows(uint8_t* smem, const CUtensorMap* tmO, Bars* bars, uint32_t tmem,
                             const Params& p, const WaitGuard& g) {
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int quarter = warp & 3;
    const uint32_t lanes = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
    const bool win = p.window > 0;
    const int off = p.Tk - p.Tq;
    uint32_t s_cnt = 0, pv_cnt = 0, q_it = 0;

    for (int k = 0; k * static_cast<int>(gridDim.x) < p.n_items; ++k) {
        const int idx = snake_item(k, p.n_items);
        if (idx < 0) continue;
        const Item it = decode_item(idx, p);
        const int wrow0 = it.qt * BM + 32 * quarter;  // first row of this warp
        const int row = wrow0 + lane;
        // Last visible key (causal limit or end of the keys) and first visible
        // key (window) of this row and of the warp's first and last rows.  Both
        // grow with the row, so the warp's extremes are those of its ends.
        auto lim_of = [&](int r) { return p.causal ? min(r + off, p.Tk - 1) : p.Tk - 1; };
        auto lft_of = [&](int r) { return win ? r + off - p.window + 1 : INT_MIN; };
        const int lim = lim_of(row), lim_lo = lim_of(wrow0), lim_hi = lim_of(wrow0 + 31);
        const int lft = lft_of(row), lft_lo = lft_of(wrow0), lft_hi = lft_of(wrow0 + 31);
        float m = -INFINITY, l = 0.0f, lr = 0.0f;

        for (int j = it.lo; j < it.n; ++j) {
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full, s_cnt & 1, g, SITE_S_FULL)))
                return;
            ++s_cnt;
            tc_fence_after_sync();
            uint32_t s[2][64];
            tmem_ld32x64(lanes + kColS, s[0]);
            tmem_ld32x64(lanes + kColS + 64, s[1]);
            tmem_wait_ld64(s[0]);
            reg_order64(s[1]);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->s_free);  // QK^T of the next tile may run

            // Chunk classes for the whole warp: 0 = no row sees a key of the
            // chunk, 2 = every row sees all of them, 1 = mask element-wise.
            // Only tiles that cross some row's limit (the diagonal, the end of
            // the keys, a window's start) are classified at all.
            const int key0 = j * BN;
            int cls[4] = {2, 2, 2, 2};
            float mx;
            if (!(key0 + BN - 1 <= lim_lo && key0 >= lft_hi)) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int kc = key0 + 32 * c;
                    const bool none = kc > lim_hi || kc + 31 < lft_lo;
                    const bool all = kc + 31 <= lim_lo && kc >= lft_hi;
                    cls[c] = none ? 0 : (all ? 2 : 1);
                }
                mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t* sc = &s[c >> 1][32 * (c & 1)];
                    if (cls[c] == 1) {
                        // Keep this a branch: executed on every tile as
                        // selects, the masking would cost every tile.
                        asm volatile("" ::: "memory");
                        const int kc = key0 + 32 * c;
                        const int dr = lim - kc;             // last visible offset in the chunk
                        const int dl = win ? lft - kc : -1;  // first visible offset
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (e > dr || e < dl) sc[e] = __float_as_uint(-INFINITY);
                    }
                    if (cls[c] != 0) mx = fmaxf(mx, chunk_max(sc));
                }
            } else {
                mx = fmaxf(fmaxf(chunk_max(&s[0][0]), chunk_max(&s[0][32])),
                           fmaxf(chunk_max(&s[1][0]), chunk_max(&s[1][32])));
            }

            // Reference: the first tile sets it to the row maximum; later tiles
            // move it only when their maximum exceeds it by more than the
            // threshold (then l, lr and O are scaled by alpha).
            const float mc = mx * p.scale_log2;  // -inf if this row sees no key here
            float alpha = 1.0f;
            bool rescale = false;
            if (j == it.lo) {
                m = mc;
            } else {
                const bool need = mc > m + kRescaleThreshold;
                if (need) {
                    alpha = (m == -INFINITY) ? 0.0f : ex2_approx(m - mc);
                    l *= alpha;
                    lr *= alpha;
                    m = mc;
                }
                rescale = __any_sync(0xffffffffu, need);
            }
            const float nm = (m == -INFINITY) ? 0.0f : -m;
            const uint64_t nm2 = f2_pack(nm, nm);

            // A chunk that no row of the warp sees is weighted against an
            // offset of -inf, which gives exact zeros without a branch (a
            // branch around the chunk here costs the softmax its registers).
            const uint64_t zero2 = f2_pack(-INFINITY, -INFINITY);
            uint32_t pk[64];
            uint64_t acc_e[2] = {0ull, 0ull};
            float acc_r[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int c = 0; c < 4; ++c)
                chunk_exp2<kF16>(&s[c >> 1][32 * (c & 1)], sc2, cls[c] == 0 ? zero2 : nm2,
                                 &pk[16 * c], acc_e, acc_r);

            // P and O belong to the previous tile's P.V until it completes.
            if (j > it.lo) {
                if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done, pv_cnt & 1, g, SITE_PV_DONE)))
                    return;
                ++pv_cnt;
                tc_fence_after_sync();
            }
            if (rescale) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t ov[32];
                    tmem_ld32(lanes + kColO + 32 * h, ov);
                    tmem_wait_ld(ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    tmem_st32(lanes + kColO + 32 * h, ov);
                }
            }
            tmem_st32x64(lanes + kColP, pk);
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_full);

            float e0, e1, e2, e3;
            f2_unpack(acc_e[0], e0, e1);
            f2_unpack(acc_e[1], e2, e3);
            l += (e0 + e1) + (e2 + e3);
            lr += (acc_r[0] + acc_r[1]) + (acc_r[2] + acc_r[3]);
        }

        // Epilogue: O = O_acc / lr -> 16-bit; lse = (m + log2 l) * ln 2.
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done, pv_cnt & 1, g, SITE_PV_DONE)))
            return;
        ++pv_cnt;
        tc_fence_after_sync();
        uint32_t ov[64];
        tmem_ld32x64(lanes + kColO, ov);
        tmem_wait_ld64(ov);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->o_free);  // the next item's P.V may overwrite O
        // The item's Q stage is free (its last QK^T completed before the last
        // P.V): this warp's 32 rows are staged there in the tensor map's
        // 128-byte-swizzled layout (16-byte chunk c of row r at c ^ (r % 8))
        // and written out by one TMA store, which leaves out rows past Tq.
        const int qs = q_it % kQStages;
        ++q_it;
        uint8_t* stage = smem + kQOff + qs * kTileBytes + 32 * quarter * 128;
        const float inv = 1.0f / lr;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint4 w;
            w.x = Elem16<kF16>::pack(__uint_as_float(ov[8 * c + 0]) * inv,
                                     __uint_as_float(ov[8 * c + 1]) * inv);
            w.y = Elem16<kF16>::pack(__uint_as_float(ov[8 * c + 2]) * inv,
                                     __uint_as_float(ov[8 * c + 3]) * inv);
            w.z = Elem16<kF16>::pack(__uint_as_float(ov[8 * c + 4]) * inv,
                                     __uint_as_float(ov[8 * c + 5]) * inv);
            w.w = Elem16<kF16>::pack(__uint_as_float(ov[8 * c + 6]) * inv,
                                     __uint_as_float(ov[8 * c + 7]) * inv);
            *reinterpret_cast<uint4*>(stage + lane * 128 + ((c ^ (lane & 7)) << 4)) = w;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (wrow0 < p.Tq) {
                tma_store_3d(tmO, stage, 0, wrow0, it.bh);
                bulk_commit_group();
                bulk_wait_group_read0();  // the stage may take the next Q once read out
            }
            mbar_arrive(&bars->q_empty[qs]);
        }
        if (row < p.Tq && p.lse != nullptr)
            p.lse[static_cast<int64_t>(it.bh) * p.Tq + row] = (m + __log2f(l)) * kLn2;
    }
    if (lane == 0) bulk_wait_group0();  // the last stores have landed
}

template <bool kF16>
__global__ void __launch_bounds__(kThreads, 2)
prefill_d64_kernel(const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmO, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(&bars->q_full[s], 1);
            mbar_init(&bars->q_empty[s], 4);  // the four softmax warps' O stores
        }
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
        }
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->s_free, 4);
        mbar_init(&bars->p_full, 4);
        mbar_init(&bars->pv_done, 1);
        mbar_init(&bars->o_free, 4);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
    }
    if (warp == 2) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    const WaitGuard g{p.status, &bars->abort, p.limit_ns};

    if (warp < 4) {
        regs_decrease<kCtrlRegs>();
        if (warp == 0) {
            if (lane == 0) producer_qk(&tmQ, &tmK, smem, bars, p, g);
        } else if (warp == 3) {
            if (lane == 0) producer_v(&tmV, smem, bars, p, g);
        } else if (warp == 1) {
            mma_issuer<kF16>(smem, bars, tmem, p, g);
        }
    } else {
        regs_increase<kSoftmaxRegs>();
        softmax_rows<kF16>(smem, &tmO, bars, tmem, p, g);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool kF16>
cudaError_t launch(const PrefillMaps& maps, const Params& prm, int grid, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_d64_kernel<kF16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        // Ask for the whole shared-memory carveout so that two CTAs fit.
        e = cudaFuncSetAttribute(prefill_d64_kernel<kF16>,
                                 cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    prefill_d64_kernel<kF16><<<grid, kThreads, kSmemBytes, stream>>>(maps.q, maps.k, maps.v, maps.o,
                                                                      prm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_d64(const PrefillMaps& maps, uint16_t* o, float* lse, const Shape& s,
                               const LaunchEnv& env, int* grid_out, int* items_out,
                               int* kernels_launched) {
    Params prm;
    prm.o = o;
    prm.lse = lse;
    prm.Hq = s.Hq;
    prm.Hkv = s.Hkv;
    prm.Tq = s.Tq;
    prm.Tk = s.Tk;
    prm.group = s.Hq / s.Hkv;
    prm.causal = s.causal;
    prm.window = s.causal ? s.window : 0;
    prm.scale_log2 = s.scale * 1.4426950408889634f;
    prm.n_qtiles = (s.Tq + BM - 1) / BM;
    prm.n_bh = s.B * s.Hq;
    const long long items = static_cast<long long>(prm.n_qtiles) * prm.n_bh;
    if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    prm.n_items = static_cast<int>(items);
    prm.status = env.status;
    prm.limit_ns = env.wait_limit_ns;
    const long long slots = 2LL * env.num_sms;
    const int grid = static_cast<int>(items < slots ? items : slots);
    if (grid_out) *grid_out = grid;
    if (items_out) *items_out = prm.n_items;
    if (kernels_launched) *kernels_launched = 1;
    return s.f16 ? launch<true>(maps, prm, grid, env.stream)
                 : launch<false>(maps, prm, grid, env.stream);
}

}  // namespace attn
