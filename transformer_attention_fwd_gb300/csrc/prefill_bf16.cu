// prefill_bf16.cu -- bf16 (or fp16) attention forward on the 5th-generation
// tensor cores (tcgen05), fp32 accumulation in tensor memory.
//
// The method is the tiled attention with online softmax of
// "3.3 Self-Attention机制深入理解" §12.2/§12.3: for every tile of query rows
// walk the key/value tiles, compute S = Q K^T, fold S into a running row
// maximum and row sum, and accumulate P V, so the score matrix never leaves
// the SM.  Causal tiles wholly above the diagonal are never visited and only
// tiles that straddle the diagonal (or the end of the keys) are masked element
// by element ("第 11 章 · Attention 入门" §11.8.3).  Query head hq reads K/V head
// hq / (Hq / Hkv) (§11.8.1).
//
// GB300 mapping (one persistent CTA per SM, 384 threads):
//   warp 0      TMA producer for Q and K tiles        (one elected lane)
//   warp 3      TMA producer for V tiles              (one elected lane)
//   warp 1      MMA issuer        (whole warp, converged; elect.sync issues)
//   warp 2      tensor-memory allocator
//   warps 4-11  softmax: warp w owns TMEM lanes 32(w%4) + 16((w-4)/4) .. +15,
//               i.e. 16 rows of each query tile, four threads per row
// A work item is 256 query rows (two 128-row tiles) of one (b, hq).  Tensor
// memory (512 columns x 128 lanes x 32 bit) holds S0, S1 (128 columns each),
// O0, O1 (D columns each).  P overwrites the first 64 columns of its S tile as
// packed bf16 and feeds the P.V MMA straight from tensor memory.  The MMA
// issue order per key tile j is
//     S0(j)  PV1(j-1)  S1(j)  PV0(j)
// so the softmax works on one tile while the tensor core runs the other
// tile's products; every tile is spread over two warps per SM sub-partition,
// which halves the latency of its softmax against one warp per row quarter.
// The softmax computes a row maximum only on a row's first tile and on the
// rare tile whose weights outgrow 2^64 (2^17 for fp16); every other tile is
// weighted against the running reference directly.
//
// Template arguments: head dim D, kPacked (sequences packed along the token
// axis of (T, H, D) tensors, one record per work item written by the
// scheduling kernels of varlen_sched.cu), kF16 (fp16 instead of bf16 I/O).
// A runtime window (> 0) limits each row to its most recent keys.
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

constexpr int NQT = 2;                   // query tiles per work item
constexpr int kItemRows = BM * NQT;
constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 256;  // warps 4-11
constexpr uint32_t kTmemCols = 512;
constexpr float kLn2 = 0.6931471805599453f;

// Wait sites reported in the status word when a wait times out.
enum : unsigned {
    SITE_Q_EMPTY = 1, SITE_K_EMPTY, SITE_V_EMPTY, SITE_Q_FULL, SITE_K_FULL, SITE_V_FULL,
    SITE_P_FULL, SITE_O_EMPTY, SITE_S_FULL, SITE_O_FULL, SITE_DIAG_LOAD, SITE_DIAG_MMA,
    SITE_DIAG_TIMEOUT
};

template <int D>
struct Cfg {
    static constexpr int kChunks = D / kBoxCols;
    static constexpr int kTileBytes = kChunks * kBoxBytes;  // 128 rows x D bf16
    static constexpr int kQStages = (D == 128) ? 1 : 2;    // Q buffers (2 query tiles each)
    static constexpr int kKStages = (D == 128) ? 3 : 4;
    static constexpr int kVStages = (D == 128) ? 2 : 4;
    // At D = 64 the P.V product also sums the rounded weights: its B operand
    // gets 16 more columns from a constant box of ones, so O carries
    // sum_k bf16(P[r, k]) in columns D .. D+15 and the softmax does not add
    // them up (tensor memory has room: 2 x (64 + 16) + 256 columns).
    static constexpr int kLrCols = (D == 64) ? 16 : 0;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kQStages * NQT * kTileBytes;
    static constexpr int kVOff = kKOff + kKStages * kTileBytes;
    static constexpr int kOnesOff = kVOff + kVStages * kTileBytes;  // 128 x 64 ones (kLrCols)
    static constexpr int kBarOff = kOnesOff + (kLrCols ? kBoxBytes : 0);
    static constexpr int kBarBytes = 256;
    static constexpr int kSmemBytes = kBarOff + kBarBytes + 1024;  // + 1024-byte alignment slack
    // Tensor-memory columns of the S/P and O accumulators of query tile t.
    __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
    __device__ static constexpr uint32_t col_o(int t) {
        return 256u + static_cast<uint32_t>(D + kLrCols) * t;
    }
};

// Register split (setmaxnreg): the CTA launches with 168 registers per thread
// (384 x 168 = 64512); the four control warps drop to 64 and the eight
// softmax warps rise to 216: 128 x 64 + 256 x 216 = 63488 <= 64512.
constexpr int kCtrlRegs = 64;
constexpr int kSoftmaxRegs = 216;
static_assert(128 * kCtrlRegs + 256 * kSoftmaxRegs <= kThreads * 168, "register split too large");

// Share of the exponentials of an unmasked tile evaluated by the polynomial
// (exp2_poly_x2) instead of the MUFU unit: pairs with
// (i % kPolyEvery) == kPolyEvery - 1, i.e. one pair in kPolyEvery (0: none).
// GB300's MUFU issues ex2 at twice the rate of earlier Blackwell parts and the
// softmax warps are bound by instruction issue, not by MUFU, so moving work
// to the FMA pipe does not pay: measured on the T=8192 causal workload with
// the current softmax layout, none (1387 TFLOP/s) beat one chunk in 8 (1329),
// in 4 (1188), in 3 (1204) and in 2 (1109).
#ifndef ATTN_PREFILL_POLY_EVERY
#define ATTN_PREFILL_POLY_EVERY 0
#endif
constexpr int kPolyEvery = ATTN_PREFILL_POLY_EVERY;

struct Bars {
    uint64_t q_full[2], q_empty[2];
    uint64_t k_full[4], k_empty[4];
    uint64_t v_full[4], v_empty[4];
    uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block too large");

struct PrefillParams {
    uint16_t* o;
    float* lse;
    int Hq, Hkv, Tq, Tk, group, causal;
    int window;  // > 0: each row also drops keys more than window-1 before its own
    float scale_log2;
    int n_qblocks, n_bh, n_items;
    // Packed mode ((T, H, D) tensors, sequences back to back along T): two
    // int4 per work item (see Record) and the device-side item count
    // (n_items is then an upper bound); total_q rows of q and o, lse
    // [Hq, total_q].
    const int4* items;
    const int* n_items_dev;
    int total_q;
    // Key splits (dense mode, non-causal, no window): item idx covers key
    // tiles [s * tiles_per_split, (s + 1) * tiles_per_split) of its head,
    // s = idx % splits, and writes its normalised partial output (fp32
    // [rows, splits, D]) and base-2 log-sum-exp ([rows, splits]) to ws_o and
    // ws_lse instead of O and lse; a combine kernel merges the splits.
    int splits, tiles_per_split;
    float* ws_o;
    float* ws_lse;
    unsigned* status;
    unsigned long long limit_ns;
};

// A work item: query block qb (two 128-row tiles) of one query head.
// Dense mode: head bh of the [B*Hq] planes, KV plane bkv, lengths p.Tq, p.Tk.
// Packed mode (kPacked): head bh of the sequence at query rows q0.. and key
// rows k0.. of the packed tensors, lengths Tq, Tk; bkv is the KV head.
struct Item {
    int bh, qb, bkv;
    int n[2];   // query tile t visits key tiles lo[t] .. n[t]-1 (n = 0: tile is past Tq)
    int lo[2];  // first key tile holding a key of the tile's first row's window
    int split;  // key split (0 without splits)
    int q0, k0, Tq, Tk;  // packed mode only
};

// One packed-mode work item, as the scheduling kernels write it:
// {q0, Tq, k0, Tk}, {query block, head, -, -}.
struct Record {
    int4 r[2];
};

// Work item idx -> head and query block.  Dense: query blocks are numbered
// from the last (longest under the causal mask) to the first.  Packed: the
// item's record is passed in (the scheduling kernels use the same order).
template <bool kPacked>
__device__ __forceinline__ Item decode_item(int idx, const PrefillParams& p, const Record& rec) {
    Item it;
    int Tq, Tk;
    it.split = 0;
    if constexpr (!kPacked) {
        if (p.splits > 1) {
            it.split = idx % p.splits;
            idx /= p.splits;
        }
        const int qrev = idx / p.n_bh;
        it.bh = idx - qrev * p.n_bh;
        it.qb = p.n_qblocks - 1 - qrev;
        const int b = it.bh / p.Hq, hq = it.bh - b * p.Hq;
        it.bkv = b * p.Hkv + hq / p.group;
        Tq = p.Tq;
        Tk = p.Tk;
    } else {
        it.q0 = rec.r[0].x;
        it.Tq = Tq = rec.r[0].y;
        it.k0 = rec.r[0].z;
        it.Tk = Tk = rec.r[0].w;
        it.qb = rec.r[1].x;
        it.bh = rec.r[1].y;
        it.bkv = it.bh / p.group;
    }
#pragma unroll
    for (int t = 0; t < NQT; ++t) {
        const int r0 = it.qb * kItemRows + t * BM;
        it.lo[t] = 0;
        if (p.window > 0 && r0 < Tq) {
            const int first_key = r0 + (Tk - Tq) - p.window + 1;  // of row r0
            it.lo[t] = first_key > 0 ? first_key / BN : 0;
        }
        if (r0 >= Tq) {
            it.n[t] = 0;
        } else if (p.causal) {
            const int rlast = min(r0 + BM - 1, Tq - 1);
            const int kmax = min(Tk - 1, rlast + (Tk - Tq));
            it.n[t] = kmax / BN + 1;
        } else {
            it.n[t] = (Tk + BN - 1) / BN;
        }
        if (!kPacked && p.splits > 1 && it.n[t] > 0) {  // this split's key tiles
            it.lo[t] = it.split * p.tiles_per_split;
            it.n[t] = min(it.n[t], it.lo[t] + p.tiles_per_split);
        }
    }
    return it;
}

// Packed mode: the record of item idx.  The next item's record is pulled
// into L1 at the same time, so the load that starts the next item hits L1
// instead of waiting on L2 (no registers are held across the item for it).
template <bool kPacked>
__device__ __forceinline__ Record fetch_record(const PrefillParams& p, int idx, int next_idx) {
    Record rec;
    if constexpr (kPacked) {
        if (next_idx >= 0)
            asm volatile("prefetch.global.L1 [%0];" ::"l"(p.items + 2 * static_cast<int64_t>(next_idx)));
        rec.r[0] = __ldg(p.items + 2 * static_cast<int64_t>(idx));
        rec.r[1] = __ldg(p.items + 2 * static_cast<int64_t>(idx) + 1);
    } else {
        rec.r[0] = rec.r[1] = make_int4(0, 0, 0, 0);
    }
    return rec;
}

// TMA coordinates (dims 1, 2) of query row r / key row r of an item.  Dense
// tensors are viewed as [B*H][T][D] (rows along dim 1), packed ones as
// [T][H][D] (rows along dim 2).
template <bool kPacked>
__device__ __forceinline__ int2 q_coord(const Item& it, int r) {
    return kPacked ? make_int2(it.bh, it.q0 + r) : make_int2(r, it.bh);
}
template <bool kPacked>
__device__ __forceinline__ int2 k_coord(const Item& it, int r) {
    return kPacked ? make_int2(it.bkv, it.k0 + r) : make_int2(r, it.bkv);
}

// ----------------------------------------------------------------------------
// Roles
// ----------------------------------------------------------------------------
template <int D, bool kPacked>
__device__ void producer_qk(const CUtensorMap* tmQ, const CUtensorMap* tmK, uint8_t* smem,
                            Bars* bars, const PrefillParams& p, int n_items, const WaitGuard& g) {
    using C = Cfg<D>;
    uint32_t kv_it = 0, q_it = 0;
    for (int k = 0; k * static_cast<int>(gridDim.x) < n_items; ++k) {
        const int idx = snake_item(k, n_items);
        if (idx < 0) continue;
        const Item it = decode_item<kPacked>(
            idx, p, fetch_record<kPacked>(p, idx, snake_item(k + 1, n_items)));
        const int nkv = max(it.n[0], it.n[1]);
        const int j0 = it.lo[0];  // tile 0's window starts first
        const int qs = q_it % C::kQStages;
        const uint32_t qph = (q_it / C::kQStages) & 1;
        if (q_it >= (uint32_t)C::kQStages &&
            !mbar_wait(&bars->q_empty[qs], qph ^ 1, g, SITE_Q_EMPTY))
            goto drain;
        mbar_arrive_expect_tx(&bars->q_full[qs],
                              ((it.n[0] > 0) + (it.n[1] > 0)) * C::kTileBytes);
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
            if (it.n[t] == 0) continue;
            const int2 xy = q_coord<kPacked>(it, it.qb * kItemRows + t * BM);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_3d(smem + C::kQOff + (qs * NQT + t) * C::kTileBytes + c * kBoxBytes,
                            tmQ, &bars->q_full[qs], c * kBoxCols, xy.x, xy.y);
        }
        ++q_it;
        for (int j = j0; j < nkv; ++j, ++kv_it) {
            const int s = kv_it % C::kKStages;
            const uint32_t ph = (kv_it / C::kKStages) & 1;
            if (kv_it >= C::kKStages && !mbar_wait(&bars->k_empty[s], ph ^ 1, g, SITE_K_EMPTY))
                goto drain;
            mbar_arrive_expect_tx(&bars->k_full[s], C::kTileBytes);
            const int2 xy = k_coord<kPacked>(it, j * BN);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_3d(smem + C::kKOff + s * C::kTileBytes + c * kBoxBytes, tmK,
                            &bars->k_full[s], c * kBoxCols, xy.x, xy.y);
        }
    }
    return;
drain:
    // Let copies already in flight land before the CTA leaves.
    for (uint32_t i = (q_it > (uint32_t)C::kQStages ? q_it - C::kQStages : 0); i < q_it; ++i)
        wait_quiet(&bars->q_full[i % C::kQStages], (i / C::kQStages) & 1, kDrainLimitNs);
    for (uint32_t i = (kv_it > (uint32_t)C::kKStages ? kv_it - C::kKStages : 0); i < kv_it; ++i)
        wait_quiet(&bars->k_full[i % C::kKStages], (i / C::kKStages) & 1, kDrainLimitNs);
}

template <int D, bool kPacked>
__device__ void producer_v(const CUtensorMap* tmV, uint8_t* smem, Bars* bars,
                           const PrefillParams& p, int n_items, const WaitGuard& g) {
    using C = Cfg<D>;
    uint32_t kv_it = 0;
    for (int k = 0; k * static_cast<int>(gridDim.x) < n_items; ++k) {
        const int idx = snake_item(k, n_items);
        if (idx < 0) continue;
        const Item it = decode_item<kPacked>(
            idx, p, fetch_record<kPacked>(p, idx, snake_item(k + 1, n_items)));
        const int nkv = max(it.n[0], it.n[1]);
        const int j0 = it.lo[0];  // tile 0's window starts first
        for (int j = j0; j < nkv; ++j, ++kv_it) {
            const int s = kv_it % C::kVStages;
            const uint32_t ph = (kv_it / C::kVStages) & 1;
            if (kv_it >= C::kVStages && !mbar_wait(&bars->v_empty[s], ph ^ 1, g, SITE_V_EMPTY))
                goto drain;
            mbar_arrive_expect_tx(&bars->v_full[s], C::kTileBytes);
            const int2 xy = k_coord<kPacked>(it, j * BN);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_3d(smem + C::kVOff + s * C::kTileBytes + c * kBoxBytes, tmV,
                            &bars->v_full[s], c * kBoxCols, xy.x, xy.y);
        }
    }
    return;
drain:
    for (uint32_t i = (kv_it > (uint32_t)C::kVStages ? kv_it - C::kVStages : 0); i < kv_it; ++i)
        wait_quiet(&bars->v_full[i % C::kVStages], (i / C::kVStages) & 1, kDrainLimitNs);
}

template <int D, bool kPacked, bool kF16>
__device__ void mma_issuer(uint8_t* smem, Bars* bars, uint32_t tmem, const PrefillParams& p,
                           int n_items, const WaitGuard& g) {
    using C = Cfg<D>;
    constexpr uint32_t kTile16 = C::kTileBytes >> 4;  // one tile in descriptor units
    // Descriptors of the first Q, K and V tiles; the others are kTile16 apart.
    const uint64_t q_desc0 = smem_desc_sw128(smem_u32(smem + C::kQOff), 16, 1024);
    const uint64_t k_desc0 = smem_desc_sw128(smem_u32(smem + C::kKOff), 16, 1024);
    const uint64_t v_desc0 = smem_desc_sw128(smem_u32(smem + C::kVOff), kBoxBytes, 1024);
    // With the rounded-weight columns (D = 64) a V stage's descriptor also
    // locates the box of ones: it follows the V ring, one leading-dimension
    // offset past the stage, so stage s has start +s tiles and offset -s
    // tiles (both fields stay in range: no carry between them).
    const uint64_t v_desc_lr0 =
        smem_desc_sw128(smem_u32(smem + C::kVOff), C::kOnesOff - C::kVOff, 1024);
    auto v_desc_of = [&](uint32_t stage) -> uint64_t {
        if constexpr (C::kLrCols > 0)
            return v_desc_lr0 + stage * kTile16 - (static_cast<uint64_t>(stage * kTile16) << 16);
        else
            return desc_advance(v_desc0, stage * kTile16);
    };
    // Rolling ring positions: stage and phase parity of the next K and V tile
    // and of the V tile of the previous key tile (read by PV1 one step late).
    uint32_t ks = 0, kph = 0, vs = 0, vph = 0, pvs = 0, pvph = 0;
    uint32_t q_it = 0;
    uint32_t p_cnt[2] = {0, 0}, o_cnt[2] = {0, 0};
    const uint32_t leader = elect_leader();

    for (int k = 0; k * static_cast<int>(gridDim.x) < n_items; ++k) {
        const int idx = snake_item(k, n_items);
        if (idx < 0) continue;
        const Item it = decode_item<kPacked>(
            idx, p, fetch_record<kPacked>(p, idx, snake_item(k + 1, n_items)));
        const int n0 = it.n[0], n1 = it.n[1];
        const int lo0 = it.lo[0], lo1 = it.lo[1];  // query tile t is active for lo_t <= j < n_t
        const int nkv = max(n0, n1);
        const uint32_t qs = q_it % C::kQStages;
        if (!warp_wait(&bars->q_full[qs], (q_it / C::kQStages) & 1, g, SITE_Q_FULL)) goto drain;
        ++q_it;
        tc_fence_after_sync();
        const uint64_t q_desc = desc_advance(q_desc0, qs * NQT * kTile16);
        for (int j = lo0; j <= nkv; ++j) {
            const uint64_t k_desc = desc_advance(k_desc0, ks * kTile16);
            const uint64_t v_desc = v_desc_of(vs);
            if (j < nkv) {
                if (!warp_wait(&bars->k_full[ks], kph, g, SITE_K_FULL)) goto drain;
                tc_fence_after_sync();
                if (j >= lo0 && j < n0) {
                    issue_qk<D, kF16>(tmem + C::col_s(0), q_desc, k_desc, leader);
                    mma_commit(&bars->s_full[0], leader);
                }
            }
            if (j - 1 >= lo1 && j - 1 < n1) {  // PV1(j-1)
                if (!warp_wait(&bars->p_full[1], p_cnt[1] & 1, g, SITE_P_FULL)) goto drain;
                ++p_cnt[1];
                if (!warp_wait(&bars->v_full[pvs], pvph, g, SITE_V_FULL)) goto drain;
                if (j - 1 == lo1 && o_cnt[1] > 0 &&
                    !warp_wait(&bars->o_empty[1], (o_cnt[1] - 1) & 1, g, SITE_O_EMPTY))
                    goto drain;
                tc_fence_after_sync();
                issue_pv<D, kF16, C::kLrCols>(tmem + C::col_o(1), tmem + C::col_s(1),
                                              v_desc_of(pvs), j - 1 > lo1, leader);
                if (j - 1 == n1 - 1) {
                    mma_commit(&bars->o_full[1], leader);
                    ++o_cnt[1];
                }
            }
            if (j > lo0) mma_commit(&bars->v_empty[pvs], leader);
            if (j < nkv) {
                if (j >= lo1 && j < n1) {
                    issue_qk<D, kF16>(tmem + C::col_s(1), desc_advance(q_desc, kTile16), k_desc,
                                leader);
                    mma_commit(&bars->s_full[1], leader);
                }
                mma_commit(&bars->k_empty[ks], leader);
                if (j == nkv - 1) mma_commit(&bars->q_empty[qs], leader);
                if (j >= lo0 && j < n0) {  // PV0(j)
                    if (!warp_wait(&bars->p_full[0], p_cnt[0] & 1, g, SITE_P_FULL)) goto drain;
                    ++p_cnt[0];
                    if (!warp_wait(&bars->v_full[vs], vph, g, SITE_V_FULL)) goto drain;
                    if (j == lo0 && o_cnt[0] > 0 &&
                        !warp_wait(&bars->o_empty[0], (o_cnt[0] - 1) & 1, g, SITE_O_EMPTY))
                        goto drain;
                    tc_fence_after_sync();
                    issue_pv<D, kF16, C::kLrCols>(tmem + C::col_o(0), tmem + C::col_s(0), v_desc,
                                                  j > lo0, leader);
                    if (j == n0 - 1) {
                        mma_commit(&bars->o_full[0], leader);
                        ++o_cnt[0];
                    }
                }
                // Advance the rings: this key tile's V becomes the previous one.
                pvs = vs;
                pvph = vph;
                if (++ks == static_cast<uint32_t>(C::kKStages)) { ks = 0; kph ^= 1u; }
                if (++vs == static_cast<uint32_t>(C::kVStages)) { vs = 0; vph ^= 1u; }
            }
        }
    }
drain:
    // Wait for every MMA issued so far before tensor memory is released.
    mma_commit(&bars->drain, leader);
    wait_quiet(&bars->drain, 0, kDrainLimitNs);
}

// Softmax work of one warp on one S tile: 16 rows (TMEM lanes L0 .. L0+15)
// x 128 keys.  Thread i holds rows a = L0 + i/4 and b = a + 8, and in each
// 8-key chunk n the keys 8n + 2(i%4) and 8n + 2(i%4) + 1 of both rows
// (registers 4n .. 4n+3 of the .16x256b load: a, a, b, b).  The four threads
// of a row hold its 128 keys between them.

// Exponentials 2^(s*scale - m) of one tile.  p receives the packed bf16 pairs
// in .16x128b order (p[2n] row a, p[2n+1] row b, both P column 4n + i%4, i.e.
// keys 8n + 2(i%4) and +1); se/sr receive this thread's exact and
// bf16-rounded partial row sums.
// kSumRounded: also sum the rounded weights (sr); false when the P.V
// product sums them in its extra columns.
template <bool kPoly, bool kF16, bool kSumRounded = true>
__device__ __forceinline__ void tile_exp2(const uint32_t (&s)[64], float scale_log2,
                                          float neg_ma, float neg_mb, uint32_t (&p)[32],
                                          float (&se)[2], float (&sr)[2]) {
    const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
    const uint64_t nm2[2] = {f2_pack(neg_ma, neg_ma), f2_pack(neg_mb, neg_mb)};
    uint64_t acc_e[2][2] = {{0, 0}, {0, 0}};
    float acc_r[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};
#pragma unroll
    for (int n = 0; n < 16; ++n) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(s[4 * n + 2 * r]),
                                               __uint_as_float(s[4 * n + 2 * r + 1])),
                                       sc2, nm2[r]);
            float e0, e1;
            if (kPoly && kPolyEvery > 0 &&
                (n % (kPolyEvery > 0 ? kPolyEvery : 1)) == kPolyEvery - 1) {
                exp2_poly_x2(x2, e0, e1);
            } else {
                float x0, x1;
                f2_unpack(x2, x0, x1);
                e0 = ex2_approx(x0);
                e1 = ex2_approx(x1);
            }
            const uint32_t pk = Elem16<kF16>::pack(e0, e1);
            acc_e[r][n & 1] = f2_add(acc_e[r][n & 1], f2_pack(e0, e1));
            if constexpr (kSumRounded) Elem16<kF16>::add2(pk, acc_r[r][0], acc_r[r][1]);
            p[2 * n + r] = pk;
        }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        float e0, e1, e2, e3;
        f2_unpack(acc_e[r][0], e0, e1);
        f2_unpack(acc_e[r][1], e2, e3);
        se[r] = (e0 + e1) + (e2 + e3);
        sr[r] = acc_r[r][0] + acc_r[r][1];
    }
}

// On a tile that straddles the diagonal or the end of the keys, keys past a
// row's last visible key become -inf.  A thread's element (n, k) holds key
// key0 + 8n + (k & 1); dr = last visible key - key0 of its rows a (k < 2) and
// b, so each test compares a compile-time offset with one register.
__device__ __forceinline__ void mask_right(uint32_t (&s)[64], int dr_a, int dr_b) {
#pragma unroll
    for (int n = 0; n < 16; ++n)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (8 * n + (k & 1) > ((k < 2) ? dr_a : dr_b)) s[4 * n + k] = __float_as_uint(-INFINITY);
}

// With a sliding window ("Attention 入门" §11.8.4, only the most recent W
// tokens), keys before a row's first visible key become -inf too (dl = first
// visible key - key0).
__device__ __forceinline__ void mask_left(uint32_t (&s)[64], int dl_a, int dl_b) {
#pragma unroll
    for (int n = 0; n < 16; ++n)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (8 * n + (k & 1) < ((k < 2) ? dl_a : dl_b)) s[4 * n + k] = __float_as_uint(-INFINITY);
}

// Per-thread softmax state of one query tile: running reference m (log2
// units, the same in the four threads of a row) and this thread's partial
// exact (l) and bf16-rounded (lr) row sums, for rows a and b.
struct RowState {
    float m[2], l[2], lr[2];
};

// One S tile through the softmax: S -> P (bf16, in place in tensor memory),
// sums and reference updated, O rescaled when the reference moves.
// mask_r / mask_l: the tile crosses some row's last / first visible key.
template <int D, bool kF16>
__device__ __forceinline__ void softmax_tile(RowState& st, uint32_t s_addr, uint32_t o_addr,
                                             bool mask_r, bool mask_l, int key0, int lim_a,
                                             int lim_b, int lft_a, int lft_b, bool first,
                                             float scale_log2) {
    constexpr int kLr = Cfg<D>::kLrCols;
    constexpr bool kSumR = kLr == 0;
    uint32_t s[64];
    tmem_ld_16x256b_x16(s_addr, s);
    tmem_wait_ld64(s);
    if (mask_r) mask_right(s, lim_a - key0, lim_b - key0);
    if (mask_l) mask_left(s, lft_a - key0, lft_b - key0);
    const bool masked = mask_r || mask_l;
    // Fast path: weights against the running reference without a row
    // maximum.  bf16 P and the fp32 sums and accumulators have fp32's
    // exponent range, so weights far above 1 lose no relative precision; a
    // partial sum above 2^62 (a row sum above 2^64) or one that is not finite
    // means m must move, and the warp redoes the tile on the exact path.  A
    // row's first tile always takes the exact path.
    uint32_t pk[32];
    float se[2], sr[2];
    bool exact = first;
    if (!first) {
        if (masked)
            tile_exp2<false, kF16, kSumR>(s, scale_log2, -st.m[0], -st.m[1], pk, se, sr);
        else
            tile_exp2<true, kF16, kSumR>(s, scale_log2, -st.m[0], -st.m[1], pk, se, sr);
        exact = !(se[0] <= Elem16<kF16>::kMaxPartial) || !(se[1] <= Elem16<kF16>::kMaxPartial);
    }
    if (__any_sync(0xffffffffu, exact)) {
        // Exact path: row maximum (this thread's 32 keys, then the four
        // threads of the row), move m and rescale l, lr and O.
        float mx[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float c0 = fmaxf(__uint_as_float(s[2 * r]), __uint_as_float(s[2 * r + 1]));
            float c1 = fmaxf(__uint_as_float(s[4 + 2 * r]), __uint_as_float(s[4 + 2 * r + 1]));
#pragma unroll
            for (int n = 2; n < 16; n += 2) {
                c0 = fmax3(c0, __uint_as_float(s[4 * n + 2 * r]), __uint_as_float(s[4 * n + 2 * r + 1]));
                c1 = fmax3(c1, __uint_as_float(s[4 * n + 4 + 2 * r]),
                           __uint_as_float(s[4 * n + 4 + 2 * r + 1]));
            }
            float v = fmaxf(c0, c1);
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
            mx[r] = v;
        }
        float alpha[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const float m_new = fmaxf(st.m[r], mx[r] * scale_log2);
            const float m_use = (m_new == -INFINITY) ? st.m[r] : m_new;
            alpha[r] = (st.m[r] == -INFINITY) ? 0.0f : ex2_approx(st.m[r] - m_use);
            st.l[r] *= alpha[r];
            st.lr[r] *= alpha[r];
            st.m[r] = m_use;
        }
        if (!first) {
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t ov[32];
                tmem_ld_16x256b_x8(o_addr + 64 * c, ov);
                tmem_wait_ld(ov);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha[(i >> 1) & 1]);
                tmem_st_16x256b_x8(o_addr + 64 * c, ov);
            }
            if constexpr (kLr > 0) {  // the rounded-weight columns move with O
                uint32_t lv[8];
                tmem_ld_16x256b_x2(o_addr + D, lv);
                tmem_wait_ld8(lv);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    lv[i] = __float_as_uint(__uint_as_float(lv[i]) * alpha[(i >> 1) & 1]);
                tmem_st_16x256b_x2(o_addr + D, lv);
            }
        }
        const float nma = (st.m[0] == -INFINITY) ? 0.0f : -st.m[0];
        const float nmb = (st.m[1] == -INFINITY) ? 0.0f : -st.m[1];
        if (masked)
            tile_exp2<false, kF16, kSumR>(s, scale_log2, nma, nmb, pk, se, sr);
        else
            tile_exp2<true, kF16, kSumR>(s, scale_log2, nma, nmb, pk, se, sr);
    }
    // P overwrites the first 64 columns of the tile (keys 2j, 2j+1 in column j).
    tmem_st_16x128b_x16(s_addr, pk);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        st.l[r] += se[r];
        st.lr[r] += sr[r];
    }
}

// Softmax warps 4-11: each 16-row slice of both query tiles belongs to one
// warp (lane quarter warp % 4, half (warp - 4) / 4), so every tile is worked
// on by two warps per SM sub-partition.  Per key tile the tiles are taken in
// the order the MMA warp produces them (S0 before S1).
template <int D, bool kPacked, bool kF16>
__device__ void softmax_group(Bars* bars, uint32_t tmem, const PrefillParams& p, int n_items,
                              const WaitGuard& g) {
    using C = Cfg<D>;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int l0 = 32 * (warp & 3) + 16 * ((warp - 4) >> 2);  // first TMEM lane of this warp
    const int ra = l0 + lane / 4;                              // rows a, a + 8 of a tile
    const int kq = 2 * (lane & 3);                             // key offset inside a chunk
    const uint32_t lanes = tmem + (static_cast<uint32_t>(l0) << 16);
    uint32_t s_cnt[2] = {0, 0}, o_cnt[2] = {0, 0};

    for (int k = 0; k * static_cast<int>(gridDim.x) < n_items; ++k) {
        const int idx = snake_item(k, n_items);
        if (idx < 0) continue;
        const Item it = decode_item<kPacked>(
            idx, p, fetch_record<kPacked>(p, idx, snake_item(k + 1, n_items)));
        const int nkv = max(it.n[0], it.n[1]);
        const int j0 = it.lo[0];  // tile 0's window starts first
        const int Tq = kPacked ? it.Tq : p.Tq, Tk = kPacked ? it.Tk : p.Tk;
        RowState st[2];
        int lim_a[2], lim_b[2], lim_first[2], lft_a[2], lft_b[2], lft_last[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int r0 = it.qb * kItemRows + t * BM;
            // Last visible key of rows a, b and of the tile's first row.
            const int off = Tk - Tq;
            lim_a[t] = p.causal ? min(r0 + ra + off, Tk - 1) : Tk - 1;
            lim_b[t] = p.causal ? min(r0 + ra + 8 + off, Tk - 1) : Tk - 1;
            lim_first[t] = p.causal ? min(r0 + off, Tk - 1) : Tk - 1;
            // First visible key of rows a, b and of the tile's last row inside
            // Tq (window; INT_MIN without one).  The sums stay below Tk + BM:
            // no overflow.
            const bool win = p.window > 0;
            const int wl = off - p.window + 1;
            lft_a[t] = win ? r0 + ra + wl : INT_MIN;
            lft_b[t] = win ? r0 + ra + 8 + wl : INT_MIN;
            lft_last[t] = win ? min(r0 + BM - 1, Tq - 1) + wl : INT_MIN;
            st[t].m[0] = st[t].m[1] = -INFINITY;
            st[t].l[0] = st[t].l[1] = st[t].lr[0] = st[t].lr[1] = 0.0f;
        }
        for (int j = j0; j < nkv; ++j) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (j < it.lo[t] || j >= it.n[t]) continue;
                if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[t], s_cnt[t] & 1, g, SITE_S_FULL)))
                    return;
                ++s_cnt[t];
                tc_fence_after_sync();
                const int kbase = j * BN;
                softmax_tile<D, kF16>(st[t], lanes + C::col_s(t), lanes + C::col_o(t),
                                      kbase + BN - 1 > lim_first[t], kbase < lft_last[t],
                                      kbase + kq, lim_a[t], lim_b[t], lft_a[t], lft_b[t],
                                      j == it.lo[t], p.scale_log2);
                tmem_wait_st();
                tc_fence_before_sync();
                mbar_arrive(&bars->p_full[t]);
            }
        }

        // Epilogue: O = O_acc / lr -> bf16; lse = (m + log2 l) * ln 2.
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (it.n[t] == 0) continue;
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_full[t], o_cnt[t] & 1, g, SITE_O_FULL)))
                return;
            ++o_cnt[t];
            tc_fence_after_sync();
            float l[2], lr[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                l[r] = st[t].l[r] + __shfl_xor_sync(0xffffffffu, st[t].l[r], 1);
                l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
                lr[r] = st[t].lr[r] + __shfl_xor_sync(0xffffffffu, st[t].lr[r], 1);
                lr[r] += __shfl_xor_sync(0xffffffffu, lr[r], 2);
            }
            if constexpr (C::kLrCols > 0) {
                // The P.V product summed the rounded weights in columns D..D+15.
                uint32_t lv[8];
                tmem_ld_16x256b_x2(lanes + C::col_o(t) + D, lv);
                tmem_wait_ld8(lv);
                lr[0] = __uint_as_float(lv[0]);
                lr[1] = __uint_as_float(lv[2]);
            }
            const float inv[2] = {1.0f / lr[0], 1.0f / lr[1]};
            const int r0 = it.qb * kItemRows + t * BM;
            const int row[2] = {r0 + ra, r0 + ra + 8};
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t ov[32];
                tmem_ld_16x256b_x8(lanes + C::col_o(t) + 64 * c, ov);
                tmem_wait_ld(ov);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (row[r] >= Tq) continue;
                    const int64_t orow =
                        kPacked ? static_cast<int64_t>(it.q0 + row[r]) * p.Hq + it.bh
                                : static_cast<int64_t>(it.bh) * p.Tq + row[r];
                    if (!kPacked && p.splits > 1) {  // this split's partial output, fp32
                        float2* wptr = reinterpret_cast<float2*>(
                            p.ws_o + (orow * p.splits + it.split) * D + 64 * c + kq);
#pragma unroll
                        for (int n = 0; n < 8; ++n)
                            wptr[4 * n] = make_float2(__uint_as_float(ov[4 * n + 2 * r]) * inv[r],
                                                      __uint_as_float(ov[4 * n + 2 * r + 1]) * inv[r]);
                        continue;
                    }
                    uint32_t* optr =
                        reinterpret_cast<uint32_t*>(p.o + orow * D + 64 * c + kq);
#pragma unroll
                    for (int n = 0; n < 8; ++n)
                        optr[4 * n] =
                            Elem16<kF16>::pack(__uint_as_float(ov[4 * n + 2 * r]) * inv[r],
                                               __uint_as_float(ov[4 * n + 2 * r + 1]) * inv[r]);
                }
            }
            if (!kPacked && p.splits > 1) {  // the split's base-2 log-sum-exp
                if ((lane & 3) == 0) {
#pragma unroll
                    for (int r = 0; r < 2; ++r)
                        if (row[r] < Tq)
                            p.ws_lse[(static_cast<int64_t>(it.bh) * p.Tq + row[r]) * p.splits +
                                     it.split] = st[t].m[r] + __log2f(l[r]);
                }
            } else if ((lane & 3) == 0 && p.lse != nullptr) {
#pragma unroll
                for (int r = 0; r < 2; ++r)
                    if (row[r] < Tq)
                        p.lse[kPacked ? static_cast<int64_t>(it.bh) * p.total_q + it.q0 + row[r]
                                      : static_cast<int64_t>(it.bh) * p.Tq + row[r]] =
                            (st[t].m[r] + __log2f(l[r])) * kLn2;
            }
            tc_fence_before_sync();
            mbar_arrive(&bars->o_empty[t]);
        }
    }
}

template <int D, bool kPacked, bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
prefill_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    Bars* bars = reinterpret_cast<Bars*>(smem + C::kBarOff);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->q_full[s], 1);
            mbar_init(&bars->q_empty[s], 1);
        }
        for (int s = 0; s < 4; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bars->s_full[t], 1);
            mbar_init(&bars->p_full[t], kSoftmaxThreads);
            mbar_init(&bars->o_full[t], 1);
            mbar_init(&bars->o_empty[t], kSoftmaxThreads);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 2) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if constexpr (C::kLrCols > 0) {
        // The box of ones (every column, so any swizzle reads 1.0), written
        // through the generic proxy and fenced for the tensor core's reads.
        const uint32_t one2 = kF16 ? 0x3C003C00u : 0x3F803F80u;
        uint32_t* ones = reinterpret_cast<uint32_t*>(smem + C::kOnesOff);
        for (int i = threadIdx.x; i < kBoxBytes / 4; i += kThreads) ones[i] = one2;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    const WaitGuard g{p.status, &bars->abort, p.limit_ns};
    // Packed sequences: the scheduling kernels counted the items; the host's
    // figure is an upper bound.
    const int n_items = kPacked ? min(__ldg(p.n_items_dev), p.n_items) : p.n_items;

    if (warp < 4) {
        regs_decrease<kCtrlRegs>();
        if (warp == 0) {
            if (lane == 0) producer_qk<D, kPacked>(&tmQ, &tmK, smem, bars, p, n_items, g);
        } else if (warp == 3) {
            if (lane == 0) producer_v<D, kPacked>(&tmV, smem, bars, p, n_items, g);
        } else if (warp == 1) {
            mma_issuer<D, kPacked, kF16>(smem, bars, tmem, p, n_items, g);
        }
    } else {
        regs_increase<kSoftmaxRegs>();
        softmax_group<D, kPacked, kF16>(bars, tmem, p, n_items, g);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ----------------------------------------------------------------------------
// Diagnostics: one tile through the same MMA code, and a wait that times out.
// ----------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128, 1)
diag_mma_tile_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmV, float* s_out, float* o_out,
                     unsigned* status, unsigned long long limit_ns) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* sa = smem;
    uint8_t* sb = smem + C::kTileBytes;
    uint8_t* sv = smem + 2 * C::kTileBytes;
    Bars* bars = reinterpret_cast<Bars*>(smem + 3 * C::kTileBytes);
    const int warp = threadIdx.x / 32;
    const int row = threadIdx.x;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full[0], 1);
        mbar_init(&bars->s_full[0], 1);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&bars->tmem_base, 256);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    const WaitGuard g{status, &bars->abort, limit_ns};
    const uint32_t lane_addr = tmem_lane_base(tmem, warp);
    bool ok = true;

    if (warp == 0) {
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&bars->q_full[0], 3 * C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_2d(sa + c * kBoxBytes, &tmA, &bars->q_full[0], c * kBoxCols, 0);
                tma_load_2d(sb + c * kBoxBytes, &tmB, &bars->q_full[0], c * kBoxCols, 0);
                tma_load_2d(sv + c * kBoxBytes, &tmV, &bars->q_full[0], c * kBoxCols, 0);
            }
        }
        __syncwarp();
        const uint32_t leader = elect_leader();
        if (warp_wait(&bars->q_full[0], 0, g, SITE_DIAG_LOAD)) {
            tc_fence_after_sync();
            issue_qk<D>(tmem, smem_desc_sw128(smem_u32(sa), 16, 1024),
                        smem_desc_sw128(smem_u32(sb), 16, 1024), leader);
            mma_commit(&bars->s_full[0], leader);
        }
    }
    ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[0], 0, g, SITE_DIAG_MMA));
    if (ok) {
        tc_fence_after_sync();
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(lane_addr + 32 * c, r[c]);
        tmem_wait_ld(r[0]);
        reg_order(r[1]);
        reg_order(r[2]);
        reg_order(r[3]);
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) s_out[row * 128 + 32 * c + i] = __uint_as_float(r[c][i]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                r[2 * h][i] = pack_bf16x2(__uint_as_float(r[2 * h][2 * i]),
                                          __uint_as_float(r[2 * h][2 * i + 1]));
#pragma unroll
            for (int i = 0; i < 16; ++i)
                r[2 * h][16 + i] = pack_bf16x2(__uint_as_float(r[2 * h + 1][2 * i]),
                                               __uint_as_float(r[2 * h + 1][2 * i + 1]));
        }
        tmem_st32(lane_addr, r[0]);
        tmem_st32(lane_addr + 32, r[2]);
        tmem_wait_st();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0 && __all_sync(0xffffffffu, ok && !bars->abort)) {
        const uint32_t leader = elect_leader();
        tc_fence_after_sync();
        issue_pv<D>(tmem + 128, tmem, smem_desc_sw128(smem_u32(sv), kBoxBytes, 1024), false,
                    leader);
        mma_commit(&bars->s_full[0], leader);
    }
    ok = ok && !bars->abort;
    if (__all_sync(0xffffffffu, ok && mbar_wait(&bars->s_full[0], 1, g, SITE_DIAG_MMA))) {
        tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(lane_addr + 128 + 32 * c, ov);
            tmem_wait_ld(ov);
#pragma unroll
            for (int i = 0; i < 32; ++i) o_out[row * D + 32 * c + i] = __uint_as_float(ov[i]);
        }
    }
    if (warp == 0) {
        mma_commit(&bars->drain, elect_leader());
        wait_quiet(&bars->drain, 0, kDrainLimitNs);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 256);
    }
}

__global__ void diag_wait_timeout_kernel(unsigned* status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitGuard g{status, &abort_flag, limit_ns};
    if (threadIdx.x == 0) mbar_wait(&bar, 0, g, SITE_DIAG_TIMEOUT);  // nobody arrives
    __syncthreads();
}

template <int D, bool kPacked, bool kF16 = false>
cudaError_t launch_prefill_d(const PrefillMaps& maps, const PrefillParams& prm, int grid,
                             cudaStream_t stream) {
    using C = Cfg<D>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_bf16_kernel<D, kPacked, kF16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    prefill_bf16_kernel<D, kPacked, kF16>
        <<<grid, kThreads, C::kSmemBytes, stream>>>(maps.q, maps.k, maps.v, prm);
    return cudaGetLastError();
}

}  // namespace

int prefill_block_rows() { return kItemRows; }
int prefill_box_rows() { return BM; }

cudaError_t launch_prefill_bf16(const PrefillMaps& maps, uint16_t* o, float* lse,
                                const Shape& s, const LaunchEnv& env, int* grid_out,
                                int* items_out, int* kernels_launched) {
    // Head dim 64 runs two CTAs per SM on one query tile each (prefill_d64.cu).
    if (s.D == 64) return launch_prefill_d64(maps, o, lse, s, env, grid_out, items_out, kernels_launched);
    PrefillParams prm;
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
    prm.n_qblocks = (s.Tq + kItemRows - 1) / kItemRows;
    prm.n_bh = s.B * s.Hq;
    // Key splits (non-causal, no window; the caller checks): every split gets
    // at least one key tile.
    prm.splits = 1;
    prm.tiles_per_split = 0;
    prm.ws_o = s.split_o;
    prm.ws_lse = s.split_lse;
    if (s.kv_splits > 1) {
        const int tiles = (s.Tk + BN - 1) / BN;
        prm.tiles_per_split = (tiles + s.kv_splits - 1) / s.kv_splits;
        prm.splits = (tiles + prm.tiles_per_split - 1) / prm.tiles_per_split;
    }
    const long long items = static_cast<long long>(prm.n_qblocks) * prm.n_bh * prm.splits;
    if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    prm.n_items = static_cast<int>(items);
    prm.items = nullptr;
    prm.n_items_dev = nullptr;
    prm.total_q = 0;
    prm.status = env.status;
    prm.limit_ns = env.wait_limit_ns;
    const int grid = static_cast<int>(items < env.num_sms ? items : env.num_sms);
    if (grid_out) *grid_out = grid;
    if (items_out) *items_out = prm.n_items;
    if (kernels_launched) *kernels_launched = 1;
    return s.f16 ? launch_prefill_d<128, false, true>(maps, prm, grid, env.stream)
                 : launch_prefill_d<128, false>(maps, prm, grid, env.stream);
}

cudaError_t launch_prefill_packed_bf16(const PrefillMaps& maps, uint16_t* o, float* lse,
                                       const VarlenShape& s, const VarlenSchedule& sched,
                                       const LaunchEnv& env, int* grid_out,
                                       int* kernels_launched) {
    PrefillParams prm;
    prm.o = o;
    prm.lse = lse;
    prm.Hq = s.Hq;
    prm.Hkv = s.Hkv;
    prm.Tq = 0;
    prm.Tk = 0;
    prm.group = s.Hq / s.Hkv;
    prm.causal = s.causal;
    prm.window = s.causal ? s.window : 0;
    prm.scale_log2 = s.scale * 1.4426950408889634f;
    prm.n_qblocks = 0;
    prm.n_bh = 0;
    prm.n_items = sched.item_bound;
    prm.items = sched.items;
    prm.n_items_dev = sched.n_items;
    prm.total_q = s.total_q;
    prm.splits = 1;
    prm.tiles_per_split = 0;
    prm.ws_o = nullptr;
    prm.ws_lse = nullptr;
    prm.status = env.status;
    prm.limit_ns = env.wait_limit_ns;
    const int grid = sched.item_bound < env.num_sms ? sched.item_bound : env.num_sms;
    if (grid_out) *grid_out = grid;
    if (grid < 1) {
        if (kernels_launched) *kernels_launched = 0;
        return cudaSuccess;
    }
    if (kernels_launched) *kernels_launched = 1;
    if (s.f16)
        return (s.D == 64) ? launch_prefill_d<64, true, true>(maps, prm, grid, env.stream)
                           : launch_prefill_d<128, true, true>(maps, prm, grid, env.stream);
    return (s.D == 64) ? launch_prefill_d<64, true>(maps, prm, grid, env.stream)
                       : launch_prefill_d<128, true>(maps, prm, grid, env.stream);
}

cudaError_t launch_diag_mma_tile(const CUtensorMap& a, const CUtensorMap& b,
                                 const CUtensorMap& v, float* s_out, float* o_out, int D,
                                 const LaunchEnv& env) {
    if (D == 64) {
        constexpr int smem = 3 * Cfg<64>::kTileBytes + 256 + 1024;
        cudaError_t e = cudaFuncSetAttribute(diag_mma_tile_kernel<64>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        diag_mma_tile_kernel<64><<<1, 128, smem, env.stream>>>(a, b, v, s_out, o_out, env.status,
                                                                env.wait_limit_ns);
    } else {
        constexpr int smem = 3 * Cfg<128>::kTileBytes + 256 + 1024;
        cudaError_t e = cudaFuncSetAttribute(diag_mma_tile_kernel<128>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        diag_mma_tile_kernel<128><<<1, 128, smem, env.stream>>>(a, b, v, s_out, o_out, env.status,
                                                                 env.wait_limit_ns);
    }
    return cudaGetLastError();
}

cudaError_t launch_diag_wait_timeout(const LaunchEnv& env, uint64_t limit_ns) {
    diag_wait_timeout_kernel<<<1, 32, 0, env.stream>>>(env.status, limit_ns);
    return cudaGetLastError();
}

}  // namespace attn
