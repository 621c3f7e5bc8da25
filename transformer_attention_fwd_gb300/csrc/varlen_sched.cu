// Work items of the packed variable-length prefill.
//
// Sequences are packed back to back along the token axis of (T, H, D)
// tensors ("第 11 章 · Attention 入门", 11.11, the (T, H, D) layout), with
// per-sequence offsets cu_q / cu_k held on the device.  A work item is one
// query block (two 128-row tiles) of one head of one sequence, as in the
// dense prefill.  The items are laid out longest first, as the dense
// prefill numbers them: level L holds query block L of every sequence that
// has more than L blocks, and levels run from the highest down, so the
// persistent grid's snake dealing balances the causal work.
//
// Two kernels, both on the caller's stream before the prefill kernel:
//   varlen_schedule_kernel (one block): validates the offsets, counts the
//     sequences by query-block count, sorts the sequences by that count
//     (descending; a counting sort) and writes the level offsets;
//   varlen_items_kernel (one block per SM): writes one 32-byte record per
//     item, so the prefill kernel reads an item with two loads instead of a
//     search, and gives query rows of sequences without keys O = 0 and
//     lse = -inf.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "attn_internal.h"
#include "sm100.cuh"

namespace attn {
namespace {

constexpr int kSchedThreads = 1024;  // the block scan below assumes exactly 32 warps
constexpr int kItemsThreads = 256;

// Byte offsets of the workspace arrays (host-computed, passed by value).
struct VarlenLayout {
    int cap;         // most query blocks one sequence can have
    int item_bound;  // most items the schedule can produce
    size_t hist, fill, start, level_off, meta, seqs, items, total;
};

size_t align16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

bool make_layout(const VarlenShape& s, int rows, VarlenLayout* L) {
    const long long cap = (static_cast<long long>(s.total_q) + rows - 1) / rows;
    // sum over sequences of ceil(Tq_b / rows) <= total_q / rows + (sequences with Tq_b > 0)
    const long long blocks = s.total_q / rows + (s.B < s.total_q ? s.B : s.total_q);
    const long long bound = blocks * s.Hq;
    if (bound > INT_MAX || cap > INT_MAX - 2) return false;
    L->cap = static_cast<int>(cap);
    L->item_bound = static_cast<int>(bound);
    size_t at = 0;
    const size_t ints = static_cast<size_t>(cap + 1) * sizeof(int);
    L->hist = at;      at = align16(at + ints);
    L->fill = at;      at = align16(at + ints);
    L->start = at;     at = align16(at + ints);
    L->level_off = at; at = align16(at + ints);
    L->meta = at;      at = align16(at + 4 * sizeof(int));
    L->seqs = at;      at = align16(at + static_cast<size_t>(s.B) * sizeof(int4));
    at = (at + 127) & ~static_cast<size_t>(127);  // 32-byte records never straddle a line
    L->items = at;     at = align16(at + static_cast<size_t>(bound) * 2 * sizeof(int4));
    L->total = at;
    return true;
}

// Sequence b's rows, checked against the tensors: {q0, Tq, k0, Tk}, or
// zeros with *valid = false.  Returns its query-block count, 0 when it has
// no queries, no keys or bad offsets.
__device__ __forceinline__ int read_sequence(const int* cu_q, const int* cu_k, int b,
                                             int total_q, int total_k, int causal, int rows,
                                             int4* sq, bool* valid) {
    const int q0 = cu_q[b], q1 = cu_q[b + 1], k0 = cu_k[b], k1 = cu_k[b + 1];
    bool ok = 0 <= q0 && q0 <= q1 && q1 <= total_q && 0 <= k0 && k0 <= k1 && k1 <= total_k;
    if (ok && causal && q1 - q0 > k1 - k0) ok = false;  // bottom-right causal needs Tq <= Tk
    *valid = ok;
    if (!ok) {
        *sq = make_int4(0, 0, 0, 0);
        return 0;
    }
    const int tq = q1 - q0, tk = k1 - k0;
    *sq = make_int4(q0, tq, k0, tk);
    if (tk == 0) return 0;
    return tq / rows + (tq % rows != 0);
}

// Exclusive scan of one int per thread over a block of exactly 32 warps;
// *total is the block's sum.  Every thread of the block must call it.
__device__ __forceinline__ int block_excl_scan(int v, int* warp_sum, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        warp_sum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int excl = incl - v + (warp > 0 ? warp_sum[warp - 1] : 0);
    *total = warp_sum[31];
    __syncthreads();  // warp_sum is reused by the next call
    return excl;
}

__global__ void __launch_bounds__(kSchedThreads)
varlen_schedule_kernel(const int* cu_q, const int* cu_k, int B, int total_q, int total_k,
                       int causal, int Hq, int rows, VarlenLayout L, uint8_t* ws,
                       unsigned* status) {
    int* hist = reinterpret_cast<int*>(ws + L.hist);    // sequences with c query blocks
    int* fill = reinterpret_cast<int*>(ws + L.fill);    // scatter counters
    int* start = reinterpret_cast<int*>(ws + L.start);  // sequences with more than c blocks
    int* off = reinterpret_cast<int*>(ws + L.level_off);
    int* meta = reinterpret_cast<int*>(ws + L.meta);
    int4* seqs = reinterpret_cast<int4*>(ws + L.seqs);
    __shared__ int warp_sum[32];
    __shared__ int s_levels, s_empty;
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_levels = 0;
        s_empty = 0;
    }
    for (int i = tid; i <= L.cap; i += kSchedThreads) {
        hist[i] = 0;
        fill[i] = 0;
    }
    __syncthreads();

    // Count the sequences by query-block count; flag bad offsets.
    for (int b = tid; b < B; b += kSchedThreads) {
        int4 sq;
        bool valid;
        const int c = read_sequence(cu_q, cu_k, b, total_q, total_k, causal, rows, &sq, &valid);
        if (!valid) atomicOr(status, ATTN_DEV_BAD_INPUT);
        if (c > 0) {
            atomicAdd(&hist[c], 1);
            atomicMax(&s_levels, c);
        } else if (valid && sq.y > 0) {
            atomicAdd(&s_empty, 1);  // queries without keys
        }
    }
    __syncthreads();

    // start[c] = number of sequences with more than c blocks (a suffix sum,
    // taken in chunks of the block from the top count down).
    int carry = 0;
    for (int base = 0; base <= L.cap; base += kSchedThreads) {
        const int c = L.cap - (base + tid);
        const int e = (c >= 0 && c < L.cap) ? hist[c + 1] : 0;
        int total;
        const int excl = block_excl_scan(e, warp_sum, &total);
        if (c >= 0) start[c] = carry + excl + e;
        carry += total;
    }
    __syncthreads();

    // Level lam (query block nl-1-lam) holds Hq items per sequence with more
    // than nl-1-lam blocks: the first start[nl-1-lam] sequences once sorted.
    const int nl = s_levels;
    carry = 0;
    for (int base = 0; base <= nl; base += kSchedThreads) {
        const int lam = base + tid;
        const int g = lam < nl ? start[nl - 1 - lam] : 0;
        int total;
        const int excl = block_excl_scan(g, warp_sum, &total);
        if (lam <= nl) off[lam] = (carry + excl) * Hq;
        carry += total;
    }
    if (tid == 0) {
        meta[0] = carry * Hq;
        meta[1] = nl;
        meta[2] = s_empty;
    }

    // Counting sort: the sequences with c blocks go to positions start[c] ..
    // start[c] + hist[c] - 1 (in no particular order among themselves).
    for (int b = tid; b < B; b += kSchedThreads) {
        int4 sq;
        bool valid;
        const int c = read_sequence(cu_q, cu_k, b, total_q, total_k, causal, rows, &sq, &valid);
        if (c > 0) seqs[start[c] + atomicAdd(&fill[c], 1)] = sq;
    }
}

__global__ void __launch_bounds__(kItemsThreads)
varlen_items_kernel(const int* cu_q, const int* cu_k, int B, int total_q, int total_k,
                    int causal, int Hq, int D, int rows, VarlenLayout L, uint8_t* ws,
                    uint16_t* o, float* lse) {
    const int* off = reinterpret_cast<const int*>(ws + L.level_off);
    const int* meta = reinterpret_cast<const int*>(ws + L.meta);
    const int4* seqs = reinterpret_cast<const int4*>(ws + L.seqs);
    int4* items = reinterpret_cast<int4*>(ws + L.items);
    const int n = min(meta[0], L.item_bound), nl = meta[1];
    const int stride = gridDim.x * blockDim.x;
    for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += stride) {
        int lo = 0, hi = nl;  // off[lo] <= idx < off[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (off[mid] <= idx) lo = mid;
            else hi = mid;
        }
        const int r = idx - off[lo];
        const int bi = r / Hq, h = r - bi * Hq;
        items[2 * static_cast<int64_t>(idx)] = seqs[bi];
        items[2 * static_cast<int64_t>(idx) + 1] = make_int4(nl - 1 - lo, h, 0, 0);
    }
    if (meta[2] == 0) return;
    // Query rows of sequences without keys: their softmax is over an empty set.
    for (int row = blockIdx.x * blockDim.x + threadIdx.x; row < total_q; row += stride) {
        int lo = 0, hi = B;  // the last sequence starting at or before row
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cu_q[mid] <= row) lo = mid;
            else hi = mid;
        }
        int4 sq;
        bool valid;
        read_sequence(cu_q, cu_k, lo, total_q, total_k, causal, rows, &sq, &valid);
        if (!valid || sq.w != 0 || row < sq.x || row >= sq.x + sq.y) continue;
        uint4* orow = reinterpret_cast<uint4*>(o + static_cast<int64_t>(row) * Hq * D);
        for (int i = 0; i < Hq * D / 8; ++i) orow[i] = make_uint4(0, 0, 0, 0);
        if (lse != nullptr)
            for (int h = 0; h < Hq; ++h) lse[static_cast<int64_t>(h) * total_q + row] = -INFINITY;
    }
}

}  // namespace

size_t varlen_workspace_bytes(const VarlenShape& s) {
    VarlenLayout L;
    return make_layout(s, prefill_block_rows(), &L) ? L.total : 0;
}

cudaError_t launch_varlen_schedule(const int* cu_q, const int* cu_k, const VarlenShape& s,
                                   void* ws, uint16_t* o, float* lse, const LaunchEnv& env,
                                   VarlenSchedule* out, int* kernels_launched) {
    const int rows = prefill_block_rows();
    VarlenLayout L;
    if (!make_layout(s, rows, &L)) return cudaErrorInvalidConfiguration;
    uint8_t* w = static_cast<uint8_t*>(ws);
    varlen_schedule_kernel<<<1, kSchedThreads, 0, env.stream>>>(
        cu_q, cu_k, s.B, s.total_q, s.total_k, s.causal, s.Hq, rows, L, w, env.status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    varlen_items_kernel<<<env.num_sms, kItemsThreads, 0, env.stream>>>(
        cu_q, cu_k, s.B, s.total_q, s.total_k, s.causal, s.Hq, s.D, rows, L, w, o, lse);
    e = cudaGetLastError();
    out->items = reinterpret_cast<const int4*>(w + L.items);
    out->n_items = reinterpret_cast<const int*>(w + L.meta);
    out->item_bound = L.item_bound;
    if (kernels_launched) *kernels_launched = 2;
    return e;
}

}  // namespace attn
