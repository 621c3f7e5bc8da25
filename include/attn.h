/*
 * attn.h -- C ABI of libattn.so: scaled dot-product attention forward on one
 * NVIDIA GB300 (sm_103a).
 *
 * The operation ("第 11 章 · Attention 入门" §11.1; "3.3 Self-Attention机制深入理解"
 * §3.6, complete formula):
 *
 *     O = softmax(Q K^T * scale + mask) V
 *
 * evaluated per (batch b, query head hq) with key/value head
 * hkv = hq / (Hq / Hkv) ("Attention 入门" §11.8.1 MHA/MQA/GQA; "Self-Attention
 * 机制深入理解" §9.3).  With causal != 0, query row i sees key j iff
 * j <= i + (Tk - Tq): the lower-triangular mask of "Self-Attention机制深入理解"
 * §10.2 when Tq == Tk, aligned so the last query sees the last key otherwise.
 * The score matrix is never written to memory: the kernels tile Q and K/V and
 * keep a running row max and sum ("Self-Attention机制深入理解" §7.3, §12.2,
 * §12.3).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory: q, k, v, o and lse are DEVICE pointers owned by the caller; the
 *   library keeps none of them after the call returns.
 * Layout: q and o are [B, Hq, Tq, D], k and v are [B, Hkv, Tk, D], row-major
 *   and contiguous, D innermost.  lse is float32 [B, Hq, Tq], or NULL when not
 *   wanted.  q, k, v, o must be 16-byte aligned; lse 4-byte aligned.
 * Element type: q, k, v and o share one type (attn_dtype); accumulation is
 *   always float32 ("Attention 入门" §11.8.5: 16-bit I/O, fp32 accumulation).
 * lse: natural-log log-sum-exp of the row's scaled, masked scores,
 *   lse_i = ln sum_j exp(scale * q_i . k_j).
 * Supported: B, Hq, Hkv, Tq, Tk >= 1; D in {64, 128}; Hq % Hkv == 0;
 *   causal requires Tq <= Tk; scale finite.  Element counts must fit in
 *   64-bit, Tq and Tk below 2^31.
 * Streams: every call is asynchronous on `stream` (0 = legacy default
 *   stream).  Argument errors are returned synchronously before anything is
 *   launched.  A launch failure returns ATTN_ERR_CUDA.  Errors raised while
 *   the kernel runs (a pipeline wait that ran out of time) are recorded in a
 *   device status word that attn_get_device_status reads.
 * Threads: entry points may be called from several host threads; the
 *   message of attn_last_error is per thread.
 */
#ifndef ATTN_H
#define ATTN_H

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* bad pointer, shape, alignment or scale */
    ATTN_ERR_UNSUPPORTED = 2, /* valid request this build cannot run (e.g. D) */
    ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
    ATTN_ERR_NO_MEMORY = 4,   /* workspace allocation failed */
    ATTN_ERR_TIMEOUT = 5,     /* a kernel pipeline wait ran out of time */
    ATTN_ERR_BAD_INPUT = 6    /* a kernel found a device-side index out of range */
} attn_status;

typedef enum { ATTN_F32 = 0, ATTN_BF16 = 1, ATTN_F16 = 2 } attn_dtype;

/*
 * attn_fwd -- attention forward, dispatching on dtype and Tq.
 *   ATTN_BF16, Tq == 1 -> split-KV decode (attn_fwd_decode, automatic split
 *                         count; "Attention 入门" §11.8.2: decode streams
 *                         K/V from the cache with a 1 x N query).
 *   ATTN_BF16, Tq >= 2 -> tensor-core prefill (attn_fwd_prefill).
 *   ATTN_F16           -> the same two paths with fp16 q, k, v and o (the
 *                         16-bit I/O of "Attention 入门" §11.8.5, fp32
 *                         accumulation): P is rounded to fp16 for the P.V
 *                         product, and the decode is the automatic mode.
 *   ATTN_F32           -> float32 tiled kernel on the CUDA cores.
 * scale multiplies the raw dot products; callers normally pass 1/sqrt(D)
 * ("Attention 入门" §11.1; "Self-Attention机制深入理解" §3.3, §6).
 */
attn_status attn_fwd(const void* q, const void* k, const void* v, void* o,
                     float* lse, int B, int Hq, int Hkv, int Tq, int Tk, int D,
                     int causal, float scale, attn_dtype dtype,
                     cudaStream_t stream);

/*
 * attn_fwd_host -- attn_fwd on HOST buffers: q, k, v are read from host
 * memory and o, lse are written back to host memory; the call enqueues the
 * copies and the compute on `stream` and returns (the outputs are in place
 * once `stream` has completed the call).  Arguments, layouts and errors are
 * those of attn_fwd, with host pointers (16-byte aligned; page-locked memory,
 * cudaMallocHost or cudaHostRegister, lets the copies overlap the compute,
 * pageable memory works but serialises them).
 * The (b, hkv) pairs are cut into up to five contiguous chunks (the first and
 * last smaller than the others); each chunk is
 * copied in on one copy stream, computed on `stream` (as attn_fwd with B =
 * its pairs, Hq = Hq / Hkv, Hkv = 1) and copied out on another, so the copies
 * of one chunk overlap the compute of its neighbours.  Device buffers for the
 * five tensors are allocated and freed stream-ordered on `stream`
 * (ATTN_ERR_NO_MEMORY if that fails).  The two copy streams are shared by all
 * calls on one device.
 */
attn_status attn_fwd_host(const void* q, const void* k, const void* v,
                          void* o, float* lse, int B, int Hq, int Hkv, int Tq,
                          int Tk, int D, int causal, float scale,
                          attn_dtype dtype, cudaStream_t stream);

/*
 * attn_fwd_prefill -- bf16 tiled attention on the 5th-generation tensor cores
 * ("Self-Attention机制深入理解" §12.2 tiling with §12.3 online softmax; causal
 * tiles wholly above the diagonal are skipped and the diagonal tile is masked
 * element-wise, "Attention 入门" §11.8.3).  Any Tq >= 1.  q, k, v, o are
 * bf16 (uint16 storage).  Same arguments and errors as attn_fwd.
 */
attn_status attn_fwd_prefill(const void* q, const void* k, const void* v,
                             void* o, float* lse, int B, int Hq, int Hkv,
                             int Tq, int Tk, int D, int causal, float scale,
                             cudaStream_t stream);

/*
 * attn_fwd_decode -- one query row per (b, hq) against a contiguous KV cache
 * (Tq == 1, so the causal mask keeps every key).  q, o: [B, Hq, 1, D] bf16;
 * k, v: [B, Hkv, Tk, D] bf16.  The keys of each (b, hkv) are cut into
 * num_splits contiguous ranges processed in parallel; each range yields a
 * normalised partial output and its log-sum-exp, merged afterwards with the
 * block-merge rule of "Self-Attention机制深入理解" §12.3.
 * num_splits: 0 = automatic: all keys of all (b, hkv) are laid end to end
 * and cut into one equal slice per SM, each slice streamed by one persistent
 * CTA (a (b, hkv) cut by a slice boundary is merged the same way); for MHA
 * (Hq == Hkv) instead the split ranges below, their count chosen to fill the
 * last wave of CTAs (measured faster there).  With 8 or more query heads per
 * KV head, automatic mode instead runs the tensor-core prefill kernel: the
 * query heads that share a KV head are the rows of a non-causal prefill
 * against its keys (q viewed as [B, Hkv, Hq/Hkv, D]), P rounded to bf16 for
 * the tensor cores as in attn_fwd_prefill.  At D = 128, when the B*Hkv
 * pairs fill at most half the SMs, each pair's keys are cut into
 * ranges of at least two 128-key tiles, one work item each, whose partials
 * are merged like the split ranges below (the range count is reported as
 * attn_last_launch_info's items); otherwise one work item per pair, with no
 * workspace, from B*Hq >= 512 query rows on.
 * 1..256 = that many equal ranges per (b, hkv) (clamped to the number of
 * keys).  The result does not depend on the split choice beyond float32
 * rounding.  Partial results live in a workspace the library allocates and
 * frees on `stream` (stream-ordered); a failed allocation returns
 * ATTN_ERR_NO_MEMORY.
 */
attn_status attn_fwd_decode(const void* q, const void* k, const void* v,
                            void* o, float* lse, int B, int Hq, int Hkv,
                            int Tk, int D, float scale, int num_splits,
                            cudaStream_t stream);

/*
 * attn_fwd_decode_noalloc -- attn_fwd_decode that allocates no device memory.
 * The pages have no counterpart to this entry point: it is an interface
 * variant of the decode call, not part of the method.
 *
 * Some callers cannot let a library allocate device memory during a call:
 * serving engines and frameworks that reserve all of HBM for their own
 * allocator up front (a driver allocation in the middle of a decode step could
 * then fail with out-of-memory), or that keep allocation, and the
 * synchronisation it may bring, out of a latency-critical decode step.  This
 * call takes the arguments of attn_fwd_decode and computes the same
 * attention, but writes the split partials into a fixed workspace that is
 * part of the library's device image: an 8 MiB array that every GPU loading
 * libattn.so holds until the process exits.  It calls no cudaMalloc, cudaFree
 * or other allocating routine.  Its results are bit-identical to
 * attn_fwd_decode's while the kernels are the same ones (automatic mode while
 * the stream-K fragments fit, and explicit split counts whose partials fit);
 * where it has to take the split kernel instead (larger shapes, below) they
 * agree within the split path's float32 rounding.  Beyond attn_fwd_decode's
 * errors it returns ATTN_ERR_UNSUPPORTED for an explicit num_splits whose
 * partials do not fit the array.
 *
 * Automatic mode (num_splits = 0) runs the kernels attn_fwd_decode picks.
 * With 8 or more query heads per KV head that is the prefill kernel, per
 * (b, hkv) with no workspace, or over key ranges with their partials in the
 * array (B*Hq*ranges*(D+1)*4 bytes; when that does not fit, the CUDA-core
 * kernels below run instead).  For MHA (Hq == Hkv) it is the split kernel
 * (next paragraph); otherwise the stream-K kernels, whenever their fragment
 * workspace fits in the 8 MiB:
 * B*Hq*nseg*(D+1)*4 bytes (plus 256), where nseg = ceil(Tk / slice) + 1 and
 * slice = ceil(B*Hkv*(Hq/Hkv/hc)*Tk / SMs) keys, hc being the heads one CTA
 * serves (8, 4, 2 or 1, the largest that divides Hq/Hkv).  That holds for
 * every shape with B*Hq <= 8128 query rows at D = 128 (16131 at D = 64).
 * Above that the call uses the split kernel instead, with the automatic
 * split count lowered until its partials, B*Hq*splits*(D+1)*4 bytes, fit (one
 * split needs no workspace at all).  An explicit num_splits uses the split
 * kernel; if its partials do not fit the call returns ATTN_ERR_UNSUPPORTED
 * with the sizes in attn_last_error().
 *
 * Sharing: every call uses the same array and overwrites the part it reads
 * before reading it, so nothing has to start at zero; but calls whose kernels
 * can run at the same time on the GPU (e.g. on two streams with no ordering
 * between them) race on the array and give undefined results.  Order such
 * calls, e.g. issue them on one stream.  After attn_get_device_status reports
 * ATTN_ERR_TIMEOUT for a call, its outputs may also hold data that earlier
 * calls left in the array (a kernel that gave up early leaves some partial
 * slots unwritten, and the combine step reads them).
 *
 * Set-up: the first call on each device looks up the array's device address
 * once (cudaGetSymbolAddress, with that device current).  Make that first call
 * before any stream capture.
 */
attn_status attn_fwd_decode_noalloc(const void* q, const void* k, const void* v,
                                    void* o, float* lse, int B, int Hq, int Hkv,
                                    int Tk, int D, float scale, int num_splits,
                                    cudaStream_t stream);

/*
 * attn_fwd_window -- causal attention with a sliding window ("第 11 章 ·
 * Attention 入门" §11.8.4, Sliding Window Attention: each query attends only
 * to the most recent `window` tokens).  Query row i, at position
 * i + (Tk - Tq) of the key sequence, sees keys i + (Tk - Tq) - window + 1 ..
 * i + (Tk - Tq) (clamped at 0): its own position and the window - 1 before
 * it.  Key tiles wholly outside every row's window are never visited.
 * bf16 or fp16 (ATTN_F32 returns ATTN_ERR_UNSUPPORTED); any Tq >= 1 runs on
 * the tensor-core prefill kernel.  window >= 1 (window >= Tk is plain causal
 * attention).  Otherwise the arguments, layouts and errors of attn_fwd with
 * causal = 1.
 */
attn_status attn_fwd_window(const void* q, const void* k, const void* v,
                            void* o, float* lse, int B, int Hq, int Hkv,
                            int Tq, int Tk, int D, int window, float scale,
                            attn_dtype dtype, cudaStream_t stream);

/*
 * attn_fwd_varlen -- attention over variable-length sequences packed
 * back to back along the token axis, in the (T, H, D) layout of "第 11 章 ·
 * Attention 入门", 11.11.  Each sequence is its own attention problem: with
 * causal = 1 its query rows are aligned to the end of its keys (a chunk of
 * new tokens against a longer history, §11.8.2), and window > 0 adds the
 * sliding window of attn_fwd_window (§11.8.4).
 *   q, o:   [total_q, Hq, D] bf16 or fp16 (dtype ATTN_BF16 / ATTN_F16; ATTN_F32
 *           returns ATTN_ERR_UNSUPPORTED), 16-byte aligned.
 *   k, v:   [total_k, Hkv, D] in the same type, 16-byte aligned.
 *   cu_seqlens_q, cu_seqlens_k: [B + 1] int32, device.  Sequence b owns
 *           query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key rows
 *           cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1.
 *   lse:    [Hq, total_q] float32 or NULL (natural-log log-sum-exp).
 *   D 64 or 128; Hq a multiple of Hkv (GQA); window >= 0 (0: none; > 0 needs
 *   causal); scale > 0.
 * A sequence with queries but no keys gets O = 0 and lse = -inf.  Rows of o
 * (and lse) outside every sequence are not written.  Key and value rows past
 * a sequence's end share a tile with it and are multiplied by an exact zero
 * weight, so every row of k and v up to total_k must hold finite values.
 * Device-side checks: offsets outside 0 .. total, decreasing offsets, or a
 * causal sequence with more queries than keys drop that sequence (its rows
 * are not written) and set a flag that attn_get_device_status reports as
 * ATTN_ERR_BAD_INPUT.  Workspace (the work-item schedule) is allocated and
 * freed on `stream`; a failed allocation returns ATTN_ERR_NO_MEMORY.
 * Host-side argument errors as for attn_fwd (ATTN_ERR_INVALID_ARG /
 * ATTN_ERR_UNSUPPORTED), before anything is launched.  total_q = 0 launches
 * nothing.
 */
attn_status attn_fwd_varlen(const void* q, const void* k, const void* v,
                            void* o, float* lse, const int* cu_seqlens_q,
                            const int* cu_seqlens_k, int B, int Hq, int Hkv,
                            int total_q, int total_k, int D, int causal,
                            int window, float scale, attn_dtype dtype,
                            cudaStream_t stream);

/*
 * attn_fwd_decode_paged -- decode (one query row per (b, hq)) against a paged
 * KV cache ("第 11 章 · Attention 入门", 11.11, the KV-cache / VMM passage: the
 * cache is a pool of physical blocks of `page_size` tokens, each holding the K
 * and the V rows of its tokens for every KV head, and block_table[req][t / 16]
 * names the block of token t of request req; 16 is that passage's page size,
 * any page_size >= 1 is accepted here).
 *   q, o:        [B, Hq, 1, D] bf16 or fp16 (dtype ATTN_BF16 / ATTN_F16;
 *                ATTN_F32 returns ATTN_ERR_UNSUPPORTED), 16-byte aligned.
 *   kv_cache:    [num_blocks, 2, Hkv, page_size, D] in the same type (index 0
 *                of the second dimension = K, 1 = V), 16-byte aligned.
 *   block_table: [B, max_pages_per_seq] int32, device; entry [b][p] is the
 *                block holding tokens p*page_size .. p*page_size+page_size-1 of
 *                request b.  Entries past a request's last page are not read.
 *   seq_lens:    [B] int32, device; keys of each request, 0 .. max_pages_per_seq
 *                * page_size.  The query sees all of its request's keys (no
 *                mask).  A request with 0 keys gets O = 0 and lse = -inf.
 *   lse:         [B, Hq] float32 or NULL.
 * The arithmetic is that of attn_fwd_decode's automatic mode: all keys of all
 * (request, KV head) units are laid end to end and cut into one equal slice
 * per SM; cut units are merged with the block-merge rule.  Workspace (length
 * prefix, slice geometry, per-SM partials) is allocated and freed on `stream`
 * (stream-ordered); a failed allocation returns ATTN_ERR_NO_MEMORY.
 * Device-side checks: a block id outside 0 .. num_blocks-1 or a length outside
 * 0 .. max_pages_per_seq*page_size is never used to address memory (block 0
 * is read, the length clamped); it sets a flag that attn_get_device_status
 * reports as ATTN_ERR_BAD_INPUT, and the outputs of that call are undefined.
 * Host-side argument errors as for attn_fwd (ATTN_ERR_INVALID_ARG /
 * ATTN_ERR_UNSUPPORTED), before anything is launched.
 */
attn_status attn_fwd_decode_paged(const void* q, const void* kv_cache,
                                  const int* block_table, const int* seq_lens,
                                  void* o, float* lse, int B, int Hq, int Hkv,
                                  int D, int page_size, int max_pages_per_seq,
                                  int num_blocks, float scale, attn_dtype dtype,
                                  cudaStream_t stream);

/*
 * attn_get_device_status -- synchronise `stream`, then read and clear the
 * device status word of the current device.  Returns ATTN_ERR_TIMEOUT when a
 * kernel gave up on a pipeline wait since the last call (its outputs are
 * then undefined), ATTN_ERR_BAD_INPUT when a kernel met a device-side index
 * outside its declared range (attn_fwd_decode_paged), ATTN_ERR_CUDA when
 * synchronising failed, else ATTN_OK.
 */
attn_status attn_get_device_status(cudaStream_t stream);

/* Message describing the last error returned on this host thread ("" if none).
 * The pointer stays valid until the next call on the same thread. */
const char* attn_last_error(void);

/* Number of work items (CTAs' worth of tiles) the last prefill call on this
 * thread scheduled and the grid it used; for tests and the bench. */
void attn_last_launch_info(int* grid, int* items, int* kernels_launched);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H */
