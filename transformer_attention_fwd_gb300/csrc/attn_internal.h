// attn_internal.h -- host-side interface between the C-ABI layer (attn_api.cu)
// and the per-kernel launchers.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/attn.h"

namespace attn {

// Everything a launcher needs besides the tensors.
struct LaunchEnv {
    cudaStream_t stream;
    unsigned* status;      // device status word (see sm100.cuh)
    uint64_t wait_limit_ns;
    int num_sms;
    int device;
};

struct Shape {
    int B, Hq, Hkv, Tq, Tk, D;
    int causal;
    float scale;
    int window = 0;  // > 0: sliding window of that many keys (causal, prefill kernel)
    int f16 = 0;     // 16-bit I/O is fp16 instead of bf16 (prefill and stream-K decode)
    // D = 128 prefill kernel only, non-causal without window: > 1 cuts every
    // head's keys into that many ranges; each writes its normalised partial
    // output to split_o [B*Hq*Tq, splits, D] and its base-2 log-sum-exp to
    // split_lse [B*Hq*Tq, splits] instead of O and lse (the split count is
    // lowered so that no range is empty; the launcher reports it in items).
    int kv_splits = 1;
    float* split_o = nullptr;
    float* split_lse = nullptr;
};

// Each launcher returns cudaSuccess or the CUDA error of its launch; argument
// validation has been done by the caller.
cudaError_t launch_simt_f32(const float* q, const float* k, const float* v, float* o,
                            float* lse, const Shape& s, const LaunchEnv& env,
                            int* kernels_launched);

// Prefill on tensor cores.  Tensor maps are built by the caller.
struct PrefillMaps {
    CUtensorMap q, k, v;
    CUtensorMap o;  // head dim 64 only: O as [B*Hq][Tq][D], box 64 x 32 rows (one warp's rows)
};
cudaError_t launch_prefill_bf16(const PrefillMaps& maps, uint16_t* o, float* lse,
                                const Shape& s, const LaunchEnv& env, int* grid_out,
                                int* items_out, int* kernels_launched);
int prefill_block_rows();  // query rows per CTA work item
// Dense prefill at head dim 64 (two CTAs per SM, one 128-row query tile per
// work item); launch_prefill_bf16 routes D = 64 here.
cudaError_t launch_prefill_d64(const PrefillMaps& maps, uint16_t* o, float* lse, const Shape& s,
                               const LaunchEnv& env, int* grid_out, int* items_out,
                               int* kernels_launched);

// Packed variable-length prefill: q [total_q, Hq, D], k and v [total_k, Hkv,
// D], sequence b at rows cu_q[b] .. cu_q[b+1]-1 of q and cu_k[b] ..
// cu_k[b+1]-1 of k and v; o like q, lse [Hq, total_q].
struct VarlenShape {
    int B, Hq, Hkv, total_q, total_k, D;
    int causal;
    int window;  // > 0: sliding window (causal only)
    float scale;
    int f16 = 0;  // fp16 q, k, v and o instead of bf16
};
// One work item of the packed prefill: {q0, Tq, k0, Tk}, {query block, head, 0, 0}.
struct VarlenSchedule {
    const int4* items;     // 2 int4 per item, longest query blocks first
    const int* n_items;    // device: number of items written
    int item_bound;        // host: upper bound on the item count
};
// Workspace for the scheduling kernels (bytes); 0 if the item count could
// overflow an int.
size_t varlen_workspace_bytes(const VarlenShape& s);
// Validates the offsets on the device (bad ones set ATTN_DEV_BAD_INPUT and
// drop the sequence), writes O = 0 and lse = -inf for query rows whose
// sequence has no keys, and lays out the work items in `ws`.
cudaError_t launch_varlen_schedule(const int* cu_q, const int* cu_k, const VarlenShape& s,
                                   void* ws, uint16_t* o, float* lse, const LaunchEnv& env,
                                   VarlenSchedule* out, int* kernels_launched);
// Tensor maps over the packed tensors (rows along dim 2) are built by the caller.
cudaError_t launch_prefill_packed_bf16(const PrefillMaps& maps, uint16_t* o, float* lse,
                                       const VarlenShape& s, const VarlenSchedule& sched,
                                       const LaunchEnv& env, int* grid_out,
                                       int* kernels_launched);
int prefill_box_rows();    // rows of one TMA box (Q, K and V tiles)

// Split-KV decode.  ws_o: [B*Hq, splits, D] fp32, ws_lse: [B*Hq, splits] fp32
// (log2 domain); unused (may be null) when splits == 1.
cudaError_t launch_decode_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               uint16_t* o, float* lse, float* ws_o, float* ws_lse,
                               const Shape& s, int splits, const LaunchEnv& env,
                               int* kernels_launched);
// The merge of split partials alone (ws_o [rows, splits, D], ws_lse [rows,
// splits] base 2) into bf16 (f16: fp16) O and lse (may be null).
cudaError_t launch_decode_combine(const float* ws_o, const float* ws_lse, uint16_t* o, float* lse,
                                  int rows, int D, int splits, bool f16, const LaunchEnv& env);
int decode_choose_splits(const Shape& s, int num_sms);

// Stream-K decode: one persistent CTA per SM over equal slices of all keys;
// ws holds the fragments of units that slice boundaries cut.
size_t decode_stream_workspace_bytes(const Shape& s, int num_sms);
cudaError_t launch_decode_stream_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                      uint16_t* o, float* lse, float* ws, const Shape& s,
                                      const LaunchEnv& env, int* grid_out, int* kernels_launched);
size_t decode_workspace_bytes(const Shape& s, int splits);

// Decode over a paged KV cache: kv [num_blocks, 2, Hkv, page, D], block_table
// [B, max_pages], seq_lens [B] (device).  The workspace holds the length
// prefix, the slice geometry and the fragment slots.
struct PagedShape {
    int B, Hq, Hkv, D;
    int page, max_pages, num_blocks;
    float scale;
    int f16 = 0;  // fp16 q, cache and o instead of bf16
};
size_t decode_paged_workspace_bytes(const PagedShape& s, int num_sms);
cudaError_t launch_decode_paged_bf16(const uint16_t* q, const uint16_t* kv,
                                     const int32_t* block_table, const int32_t* seq_lens,
                                     uint16_t* o, float* lse, void* ws, const PagedShape& s,
                                     const LaunchEnv& env, int* grid_out, int* kernels_launched);

// Diagnostics.
cudaError_t launch_diag_mma_tile(const CUtensorMap& a, const CUtensorMap& b,
                                 const CUtensorMap& v, float* s_out, float* o_out, int D,
                                 const LaunchEnv& env);
cudaError_t launch_diag_wait_timeout(const LaunchEnv& env, uint64_t limit_ns);

}  // namespace attn
