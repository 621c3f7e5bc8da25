// attn_api.cu -- the C ABI of libattn.so (declared in include/attn.h and
// include/attn_diag.h): argument validation, dispatch, TMA tensor maps, the
// decode workspace and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/attn.h"
#include "../../include/attn_diag.h"
#include "attn_internal.h"

namespace attn {

// Device status word: kernels OR error bits into it (see sm100.cuh).
__device__ unsigned g_attn_status;

namespace {

thread_local std::string t_last_error;
thread_local int t_last_grid = 0, t_last_items = 0, t_last_kernels = 0;

attn_status fail(attn_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

attn_status ok() {
    t_last_error.clear();
    return ATTN_OK;
}

attn_status cuda_fail(cudaError_t e, const char* what) {
    return fail(ATTN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Per-device facts gathered once.
struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    unsigned* status = nullptr;
    cudaStream_t h2d = nullptr, d2h = nullptr;  // attn_fwd_host's copy streams
};
std::mutex g_dev_mutex;
DeviceState g_dev[64];

constexpr uint64_t kWaitLimitNs = 2ull * 1000ull * 1000ull * 1000ull;  // 2 s per wait

attn_status device_env(cudaStream_t stream, LaunchEnv* env) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(ATTN_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    {
        std::lock_guard<std::mutex> lock(g_dev_mutex);
        DeviceState& d = g_dev[dev];
        if (!d.ready) {
            cudaDeviceProp prop;
            e = cudaGetDeviceProperties(&prop, dev);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
            d.num_sms = prop.multiProcessorCount;
            d.cc_major = prop.major;
            d.cc_minor = prop.minor;
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_attn_status);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
            d.status = static_cast<unsigned*>(p);
            d.ready = true;
        }
        if (!(d.cc_major == 10 && d.cc_minor == 3))
            return fail(ATTN_ERR_UNSUPPORTED,
                        "libattn.so is built for sm_103a; device %d has compute capability %d.%d",
                        dev, d.cc_major, d.cc_minor);
        env->num_sms = d.num_sms;
        env->status = d.status;
    }
    env->device = dev;
    env->stream = stream;
    env->wait_limit_ns = kWaitLimitNs;
    return ATTN_OK;
}

// ---------------------------------------------------------------------------
// Validation
// ---------------------------------------------------------------------------
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

attn_status validate(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     int B, int Hq, int Hkv, int Tq, int Tk, int D, int causal, float scale) {
    if (!q || !k || !v || !o) return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be non-null");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
        return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
    if (lse && !aligned(lse, 4)) return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
    if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Tk < 1 || D < 1)
        return fail(ATTN_ERR_INVALID_ARG,
                    "B, Hq, Hkv, Tq, Tk, D must be >= 1 (got %d, %d, %d, %d, %d, %d)", B, Hq, Hkv,
                    Tq, Tk, D);
    if (D != 64 && D != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim D=%d not supported (64 or 128)", D);
    if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
    if (causal && Tq > Tk)
        return fail(ATTN_ERR_INVALID_ARG, "causal attention needs Tq <= Tk (got Tq=%d, Tk=%d)", Tq, Tk);
    if (!std::isfinite(scale) || !(scale > 0.0f))
        return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and positive (got %g)", (double)scale);
    const long long bh = static_cast<long long>(B) * Hq, bkv = static_cast<long long>(B) * Hkv;
    if (bh > 0x7fffffffLL || bkv > 0x7fffffffLL)
        return fail(ATTN_ERR_INVALID_ARG, "B*Hq and B*Hkv must fit in 31 bits");
    if (Tq > 0x7fffffffLL - 1024 || Tk > 0x7fffffffLL - 1024)
        return fail(ATTN_ERR_INVALID_ARG, "Tq and Tk must be below 2^31 - 1024");
    return ATTN_OK;
}

// ---------------------------------------------------------------------------
// TMA tensor maps ([rows][D] bf16 slabs stacked over batch*heads), cached.
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

struct MapKey {
    const void* ptr;
    long long rows, slabs;
    int D, box_rows, rank, packed, f16;
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && rows == o.rows && slabs == o.slabs && D == o.D &&
               box_rows == o.box_rows && rank == o.rank && packed == o.packed && f16 == o.f16;
    }
};
struct MapEntry {
    MapKey key;
    CUtensorMap map;
};
std::mutex g_map_mutex;
std::vector<MapEntry> g_maps;  // most recently used last
constexpr size_t kMapCacheSize = 64;

// Tiled map over a [slabs][rows][D] bf16 (f16: fp16) tensor; box = 64
// columns x box_rows rows x 1 slab, 128-byte swizzle, zero fill outside the
// tensor.  packed: the tensor is [rows][slabs][D] instead (dims D, slabs,
// rows; box 64 x 1 x box_rows), which lands in shared memory in the same
// layout.
attn_status make_map(const void* ptr, long long rows, long long slabs, int D, int box_rows,
                     int rank, CUtensorMap* out, bool packed = false, bool f16 = false) {
    const MapKey key{ptr, rows, slabs, D, box_rows, rank, packed ? 1 : 0, f16 ? 1 : 0};
    {
        std::lock_guard<std::mutex> lock(g_map_mutex);
        for (size_t i = g_maps.size(); i-- > 0;) {
            if (g_maps[i].key == key) {
                *out = g_maps[i].map;
                if (i + 1 != g_maps.size()) {
                    MapEntry e = g_maps[i];
                    g_maps.erase(g_maps.begin() + static_cast<long>(i));
                    g_maps.push_back(e);
                }
                return ATTN_OK;
            }
        }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(slabs)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                             static_cast<cuuint64_t>(D) * 2 * static_cast<cuuint64_t>(rows)};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    if (packed) {
        dims[1] = static_cast<cuuint64_t>(slabs);
        dims[2] = static_cast<cuuint64_t>(rows);
        strides[1] = static_cast<cuuint64_t>(D) * 2 * static_cast<cuuint64_t>(slabs);
        box[1] = 1;
        box[2] = static_cast<cuuint32_t>(box_rows);
    }
    cuuint32_t estr[3] = {1, 1, 1};
    CUtensorMap m;
    CUresult r = fn(&m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    static_cast<cuuint32_t>(rank),
                    const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    {
        std::lock_guard<std::mutex> lock(g_map_mutex);
        if (g_maps.size() >= kMapCacheSize) g_maps.erase(g_maps.begin());
        g_maps.push_back(MapEntry{key, m});
    }
    *out = m;
    return ATTN_OK;
}

void record_launch(int grid, int items, int kernels) {
    t_last_grid = grid;
    t_last_items = items;
    t_last_kernels = kernels;
}

attn_status run_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                        const Shape& s, const LaunchEnv& env) {
    PrefillMaps maps;
    const int box = prefill_box_rows();
    const bool f16 = s.f16 != 0;
    attn_status st = make_map(q, s.Tq, static_cast<long long>(s.B) * s.Hq, s.D, box, 3, &maps.q,
                              false, f16);
    if (st != ATTN_OK) return st;
    st = make_map(k, s.Tk, static_cast<long long>(s.B) * s.Hkv, s.D, box, 3, &maps.k, false, f16);
    if (st != ATTN_OK) return st;
    st = make_map(v, s.Tk, static_cast<long long>(s.B) * s.Hkv, s.D, box, 3, &maps.v, false, f16);
    if (st != ATTN_OK) return st;
    if (s.D == 64) {  // the head-dim-64 kernel stores O through TMA, 32 rows per warp
        st = make_map(o, s.Tq, static_cast<long long>(s.B) * s.Hq, s.D, 32, 3, &maps.o, false, f16);
        if (st != ATTN_OK) return st;
    }
    int grid = 0, items = 0, kernels = 0;
    cudaError_t e = launch_prefill_bf16(maps, static_cast<uint16_t*>(o), lse, s, env, &grid,
                                        &items, &kernels);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    record_launch(grid, items, kernels);
    return ok();
}

// Automatic mode: the stream-K kernel (equal key slices per SM); its
// workspace holds the fragments of the units that slice boundaries cut.
attn_status run_decode_stream(const void* q, const void* k, const void* v, void* o, float* lse,
                              const Shape& s, const LaunchEnv& env) {
    const size_t bytes = decode_stream_workspace_bytes(s, env.num_sms);
    void* ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, bytes, env.stream);
    if (e != cudaSuccess || ws == nullptr) {
        cudaGetLastError();
        return fail(ATTN_ERR_NO_MEMORY, "decode workspace of %zu bytes: %s", bytes,
                    cudaGetErrorString(e));
    }
    int grid = 0, kernels = 0;
    e = launch_decode_stream_bf16(static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k),
                                  static_cast<const uint16_t*>(v), static_cast<uint16_t*>(o), lse,
                                  static_cast<float*>(ws), s, env, &grid, &kernels);
    cudaError_t f = cudaFreeAsync(ws, env.stream);
    if (e == cudaSuccess && f != cudaSuccess) e = f;
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    record_launch(grid, 0, kernels);
    return ok();
}

// Automatic decode for bf16 MHA (one query head per KV head) takes the split
// kernel rather than stream-K: its CTAs are small (64 registers a thread, four
// per SM), and in a same-process A/B over nine MHA shapes (D = 64 and 128, B
// = 1 to 128, Tk = 1024 to 32768) it streamed K/V 3 to 15 % faster.  From two
// query heads per KV head on, stream-K is ahead.  (fp16 has only stream-K.)
bool decode_prefers_split_kernel(const Shape& s) { return s.Hq == s.Hkv && !s.f16; }

// Automatic decode with many query heads per KV head runs on the tensor-core
// prefill kernel: the group of query heads that share K/V head (b, hkv) is a
// block of Tq = group query rows against Tk keys, non-causal, so with Q
// viewed as [B, Hkv, group, D] (the same memory) the decode is a prefill of
// B*Hkv heads.  The CUDA-core kernels spend 2*group*D multiply-adds per K/V
// row and are bound by instruction issue from group 8 on (about 3 TB/s at 8,
// 1.2 TB/s at 16), while the prefill streams one (b, hkv) per SM at about
// 42 GB/s each.  Same-process A/B, GB/s, CUDA-core -> prefill kernel (Hkv 8,
// Tk 4096, D 128): group 8 at B = 4, 8, 16, 32: 1490 -> 1361, 2083 -> 2724,
// 2651 -> 4375, 2985 -> 4873; group 4 at B = 64: 5879 -> 5409.  Hence: from
// 8 heads per KV head on, once B * Hq >= 512 query rows.
bool decode_prefers_prefill_kernel(const Shape& s, int /*num_sms*/) {
    const int group = s.Hq / s.Hkv;
    return group >= 8 && static_cast<long long>(s.B) * s.Hq >= 512;
}

attn_status run_decode_as_prefill(const void* q, const void* k, const void* v, void* o,
                                  float* lse, const Shape& s, const LaunchEnv& env) {
    Shape p{s.B, s.Hkv, s.Hkv, s.Hq / s.Hkv, s.Tk, s.D, 0, s.scale};
    p.f16 = s.f16;
    return run_prefill(q, k, v, o, lse, p, env);
}

// With few (b, hkv) the same prefill leaves SMs idle, so its keys are cut
// into ranges: each (b, hkv, range) is one work item writing a normalised
// partial output and its log-sum-exp, and the split decode's combine kernel
// merges the ranges ("3.3 Self-Attention机制深入理解" §12.3).  Taken at D = 128
// (bf16 or fp16) with 8 or more query heads per KV head when the (b, hkv)
// pairs fill at most half the SMs and each range still holds two key tiles;
// returns the range count (every range non-empty), or 1 when not taken.
int decode_group_splits(const Shape& s, int num_sms) {
    if (s.D != 128 || s.Hq / s.Hkv < 8) return 1;
    const long long pairs = static_cast<long long>(s.B) * s.Hkv;
    if (2 * pairs > num_sms) return 1;
    const int tiles = (s.Tk + 127) / 128;
    int splits = static_cast<int>(num_sms / pairs);
    if (splits > tiles / 2) splits = tiles / 2;
    if (splits < 2) return 1;
    const int per = (tiles + splits - 1) / splits;
    return (tiles + per - 1) / per;
}

size_t group_split_workspace_bytes(const Shape& s, int splits) {
    return static_cast<size_t>(s.B) * s.Hq * splits * (s.D + 1) * sizeof(float);
}

// ws: group_split_workspace_bytes(s, splits) bytes of device memory.
attn_status run_decode_as_split_prefill(const void* q, const void* k, const void* v, void* o,
                                        float* lse, const Shape& s, int splits, void* ws,
                                        const LaunchEnv& env) {
    Shape p{s.B, s.Hkv, s.Hkv, s.Hq / s.Hkv, s.Tk, s.D, 0, s.scale};
    const size_t rows = static_cast<size_t>(s.B) * s.Hq;
    p.f16 = s.f16;
    p.kv_splits = splits;
    p.split_o = static_cast<float*>(ws);
    p.split_lse = p.split_o + rows * splits * s.D;
    attn_status st = run_prefill(q, k, v, o, lse, p, env);
    if (st != ATTN_OK) return st;
    const int grid = t_last_grid;
    cudaError_t e = launch_decode_combine(p.split_o, p.split_lse, static_cast<uint16_t*>(o), lse,
                                          static_cast<int>(rows), s.D, splits, s.f16 != 0, env);
    if (e != cudaSuccess) return cuda_fail(e, "decode combine launch");
    record_launch(grid, splits, 2);
    return ok();
}

attn_status run_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                       const Shape& s, int num_splits, const LaunchEnv& env) {
    if (num_splits == 0) {
        const int ks = decode_group_splits(s, env.num_sms);
        if (ks > 1) {
            const size_t bytes = group_split_workspace_bytes(s, ks);
            void* ws = nullptr;
            cudaError_t e = cudaMallocAsync(&ws, bytes, env.stream);
            if (e != cudaSuccess || ws == nullptr) {
                cudaGetLastError();
                return fail(ATTN_ERR_NO_MEMORY, "decode workspace of %zu bytes: %s", bytes,
                            cudaGetErrorString(e));
            }
            attn_status st = run_decode_as_split_prefill(q, k, v, o, lse, s, ks, ws, env);
            e = cudaFreeAsync(ws, env.stream);
            if (st == ATTN_OK && e != cudaSuccess) return cuda_fail(e, "freeing the decode workspace");
            return st;
        }
        if (decode_prefers_prefill_kernel(s, env.num_sms))
            return run_decode_as_prefill(q, k, v, o, lse, s, env);
        if (!decode_prefers_split_kernel(s)) return run_decode_stream(q, k, v, o, lse, s, env);
        num_splits = decode_choose_splits(s, env.num_sms);
    }
    int splits = num_splits;
    if (splits > 256) splits = 256;
    if (splits > s.Tk) splits = s.Tk;
    // Recompute so that no split is empty.
    const int per = (s.Tk + splits - 1) / splits;
    splits = (s.Tk + per - 1) / per;

    float* ws_o = nullptr;
    float* ws_lse = nullptr;
    void* ws = nullptr;
    if (splits > 1) {
        const size_t bytes = decode_workspace_bytes(s, splits);
        cudaError_t e = cudaMallocAsync(&ws, bytes, env.stream);
        if (e != cudaSuccess || ws == nullptr) {
            cudaGetLastError();
            return fail(ATTN_ERR_NO_MEMORY, "decode workspace of %zu bytes: %s", bytes,
                        cudaGetErrorString(e));
        }
        ws_o = static_cast<float*>(ws);
        const size_t rows = static_cast<size_t>(s.B) * s.Hq;
        ws_lse = ws_o + rows * splits * s.D;
    }
    int kernels = 0;
    cudaError_t e = launch_decode_bf16(static_cast<const uint16_t*>(q),
                                       static_cast<const uint16_t*>(k),
                                       static_cast<const uint16_t*>(v), static_cast<uint16_t*>(o),
                                       lse, ws_o, ws_lse, s, splits, env, &kernels);
    if (ws) {
        cudaError_t f = cudaFreeAsync(ws, env.stream);
        if (e == cudaSuccess && f != cudaSuccess) e = f;
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    record_launch(s.B * s.Hkv, splits, kernels);
    return ok();
}

// attn_fwd's dispatch after validation: fp32 -> CUDA-core kernel; 16-bit
// Tq = 1 -> decode (stream-K, or the split kernel for bf16 MHA); otherwise the
// tensor-core prefill.
attn_status dispatch(const void* q, const void* k, const void* v, void* o, float* lse,
                     const Shape& s, attn_dtype dtype, const LaunchEnv& env) {
    if (dtype == ATTN_F32) {
        int kernels = 0;
        cudaError_t e = launch_simt_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                                        static_cast<const float*>(v), static_cast<float*>(o), lse,
                                        s, env, &kernels);
        if (e == cudaErrorInvalidConfiguration)
            return fail(ATTN_ERR_UNSUPPORTED, "Tq=%d too long for the fp32 kernel's grid", s.Tq);
        if (e != cudaSuccess) return cuda_fail(e, "fp32 launch");
        record_launch(s.B * s.Hq, (s.Tq + 15) / 16, kernels);
        return ok();
    }
    if (s.Tq == 1) return run_decode(q, k, v, o, lse, s, 0, env);
    return run_prefill(q, k, v, o, lse, s, env);
}

// attn_fwd_host's pipeline: the problem is cut into at most kHostChunks
// chunks of (b, hkv) units, the first and the last holding about
// 1/(kHostEdge * kHostChunks) of the units each (measured on the Llama-3-8B
// T = 8192 step: 5 chunks of 1, 2, 2, 2, 1 pairs 0.78 ms; 4 equal chunks
// 0.80 ms; 4 of 1, 3, 3, 1 pairs 0.82 ms; 2 or 8 equal chunks 0.90 / 0.94 ms).
constexpr int kHostChunks = 5;
constexpr int kHostEdge = 2;

// Unit boundaries of attn_fwd_host's chunks: bound[0] = 0 < ... <
// bound[chunks] = units.  The first and last chunks hold units / (kHostEdge
// * chunks) units (at least one) and the middle ones share the rest equally,
// which shortens the copy-in before the first compute and the compute and
// copy-out after the last copy-in.
int host_chunk_bounds(int units, int (&bound)[kHostChunks + 1]) {
    const int chunks = units < kHostChunks ? units : kHostChunks;
    bound[0] = 0;
    if (chunks < 3) {
        for (int c = 1; c <= chunks; ++c)
            bound[c] = static_cast<int>(static_cast<long long>(c) * units / chunks);
        return chunks;
    }
    int edge = units / (kHostEdge * chunks);
    if (edge < 1) edge = 1;
    const int mid = units - 2 * edge, nm = chunks - 2;
    bound[1] = edge;
    for (int c = 1; c <= nm; ++c) bound[c + 1] = edge + static_cast<int>(static_cast<long long>(c) * mid / nm);
    bound[chunks] = units;
    return chunks;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

attn_status attn_fwd_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int Hq, int Hkv, int Tq, int Tk, int D, int causal,
                             float scale, cudaStream_t stream) {
    attn_status st = validate(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, D, causal, scale);
    if (st != ATTN_OK) return st;
    LaunchEnv env;
    st = device_env(stream, &env);
    if (st != ATTN_OK) return st;
    const Shape s{B, Hq, Hkv, Tq, Tk, D, causal ? 1 : 0, scale};
    return run_prefill(q, k, v, o, lse, s, env);
}

attn_status attn_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int Tk, int D, float scale, int num_splits,
                            cudaStream_t stream) {
    attn_status st = validate(q, k, v, o, lse, B, Hq, Hkv, 1, Tk, D, 0, scale);
    if (st != ATTN_OK) return st;
    if (num_splits < 0 || num_splits > 256)
        return fail(ATTN_ERR_INVALID_ARG, "num_splits must be in 0..256 (got %d)", num_splits);
    LaunchEnv env;
    st = device_env(stream, &env);
    if (st != ATTN_OK) return st;
    const Shape s{B, Hq, Hkv, 1, Tk, D, 0, scale};
    return run_decode(q, k, v, o, lse, s, num_splits, env);
}

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Hq, int Hkv, int Tq, int Tk, int D, int causal, float scale,
                     attn_dtype dtype, cudaStream_t stream) {
    if (dtype != ATTN_F32 && dtype != ATTN_BF16 && dtype != ATTN_F16)
        return fail(ATTN_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dtype));
    attn_status st = validate(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, D, causal, scale);
    if (st != ATTN_OK) return st;
    LaunchEnv env;
    st = device_env(stream, &env);
    if (st != ATTN_OK) return st;
    Shape s{B, Hq, Hkv, Tq, Tk, D, causal ? 1 : 0, scale};
    s.f16 = dtype == ATTN_F16 ? 1 : 0;
    return dispatch(q, k, v, o, lse, s, dtype, env);
}

attn_status attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int Hq, int Hkv, int Tq, int Tk, int D, int causal, float scale,
                          attn_dtype dtype, cudaStream_t stream) {
    if (dtype != ATTN_F32 && dtype != ATTN_BF16 && dtype != ATTN_F16)
        return fail(ATTN_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dtype));
    attn_status st = validate(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, D, causal, scale);
    if (st != ATTN_OK) return st;
    LaunchEnv env;
    st = device_env(stream, &env);
    if (st != ATTN_OK) return st;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_dev_mutex);
        DeviceState& d = g_dev[env.device];
        if (d.h2d == nullptr) {
            cudaError_t e = cudaStreamCreateWithFlags(&d.h2d, cudaStreamNonBlocking);
            if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&d.d2h, cudaStreamNonBlocking);
            if (e != cudaSuccess) {
                d.h2d = d.d2h = nullptr;
                return cuda_fail(e, "creating the copy streams");
            }
        }
        h2d = d.h2d;
        d2h = d.d2h;
    }
    // Device copies of the five tensors in one stream-ordered allocation.
    const size_t el = dtype == ATTN_F32 ? 4 : 2;
    const size_t q_bytes = static_cast<size_t>(B) * Hq * Tq * D * el;
    const size_t kv_bytes = static_cast<size_t>(B) * Hkv * Tk * D * el;
    const size_t l_bytes = lse ? static_cast<size_t>(B) * Hq * Tq * sizeof(float) : 0;
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t off_k = up(q_bytes), off_v = off_k + up(kv_bytes), off_o = off_v + up(kv_bytes);
    const size_t off_l = off_o + up(q_bytes), total = off_l + up(l_bytes);
    uint8_t* ws = nullptr;
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&ws), total, env.stream);
    if (e != cudaSuccess || ws == nullptr) {
        cudaGetLastError();
        return fail(ATTN_ERR_NO_MEMORY, "device buffers of %zu bytes: %s", total,
                    cudaGetErrorString(e));
    }
    // Units: (b, hkv) pairs.  A contiguous range of units is a contiguous byte
    // range of every tensor and is itself a problem of shape [units, g, T, D]
    // against [units, 1, T, D]: the chunks are copied in, computed and copied
    // out on three streams, so that chunk c's compute overlaps chunk c+1's
    // inputs and chunk c-1's outputs.
    const int units = B * Hkv, g = Hq / Hkv;
    int bound[kHostChunks + 1];
    const int chunks = host_chunk_bounds(units, bound);
    const size_t uq = q_bytes / units, ukv = kv_bytes / units, ul = l_bytes / units;
    cudaEvent_t ev[2 * kHostChunks + 2];
    int n_ev = 0;
    for (; n_ev < 2 * chunks + 2; ++n_ev) {
        e = cudaEventCreateWithFlags(&ev[n_ev], cudaEventDisableTiming);
        if (e != cudaSuccess) break;
    }
    const char* what = "creating events";
    int kernels = 0, grid = 0;
    if (e == cudaSuccess) {
        cudaEvent_t ev_start = ev[0], ev_end = ev[1];
        cudaEvent_t* ev_in = ev + 2;
        cudaEvent_t* ev_out = ev + 2 + chunks;
        const uint8_t* qh = static_cast<const uint8_t*>(q);
        const uint8_t* kh = static_cast<const uint8_t*>(k);
        const uint8_t* vh = static_cast<const uint8_t*>(v);
        uint8_t* oh = static_cast<uint8_t*>(o);
        uint8_t* lh = reinterpret_cast<uint8_t*>(lse);
        what = "ordering the copy streams";
        e = cudaEventRecord(ev_start, env.stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h2d, ev_start, 0);
        for (int c = 0; c < chunks && e == cudaSuccess; ++c) {
            const size_t u0 = bound[c], u1 = bound[c + 1];
            what = "host-to-device copy";
            e = cudaMemcpyAsync(ws + u0 * uq, qh + u0 * uq, (u1 - u0) * uq, cudaMemcpyHostToDevice, h2d);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(ws + off_k + u0 * ukv, kh + u0 * ukv, (u1 - u0) * ukv,
                                    cudaMemcpyHostToDevice, h2d);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(ws + off_v + u0 * ukv, vh + u0 * ukv, (u1 - u0) * ukv,
                                    cudaMemcpyHostToDevice, h2d);
            if (e == cudaSuccess) e = cudaEventRecord(ev_in[c], h2d);
        }
        for (int c = 0; c < chunks && e == cudaSuccess; ++c) {
            const size_t u0 = bound[c], u1 = bound[c + 1];
            what = "ordering the compute stream";
            e = cudaStreamWaitEvent(env.stream, ev_in[c], 0);
            if (e != cudaSuccess) break;
            Shape s{static_cast<int>(u1 - u0), g, 1, Tq, Tk, D, causal ? 1 : 0, scale};
            s.f16 = dtype == ATTN_F16 ? 1 : 0;
            st = dispatch(ws + u0 * uq, ws + off_k + u0 * ukv, ws + off_v + u0 * ukv,
                          ws + off_o + u0 * uq,
                          lse ? reinterpret_cast<float*>(ws + off_l + u0 * ul) : nullptr, s, dtype,
                          env);
            if (st != ATTN_OK) break;
            kernels += t_last_kernels;
            grid = t_last_grid > grid ? t_last_grid : grid;
            e = cudaEventRecord(ev_out[c], env.stream);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(d2h, ev_out[c], 0);
            what = "device-to-host copy";
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(oh + u0 * uq, ws + off_o + u0 * uq, (u1 - u0) * uq,
                                    cudaMemcpyDeviceToHost, d2h);
            if (e == cudaSuccess && lse)
                e = cudaMemcpyAsync(lh + u0 * ul, ws + off_l + u0 * ul, (u1 - u0) * ul,
                                    cudaMemcpyDeviceToHost, d2h);
        }
        if (e == cudaSuccess && st == ATTN_OK) {
            what = "joining the copy streams";
            e = cudaEventRecord(ev_end, d2h);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(env.stream, ev_end, 0);
        }
    }
    cudaError_t f = cudaFreeAsync(ws, env.stream);
    for (int i = 0; i < n_ev; ++i) cudaEventDestroy(ev[i]);
    if (st != ATTN_OK) return st;
    if (e == cudaSuccess) e = f;
    if (e != cudaSuccess) return cuda_fail(e, what);
    record_launch(grid, chunks, kernels);
    return ok();
}

attn_status attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int Tq, int Tk, int D, int window,
                            float scale, attn_dtype dtype, cudaStream_t stream) {
    if (dtype == ATTN_F32)
        return fail(ATTN_ERR_UNSUPPORTED, "the sliding window is implemented for 16-bit I/O only");
    if (dtype != ATTN_BF16 && dtype != ATTN_F16)
        return fail(ATTN_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dtype));
    attn_status st = validate(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, D, 1, scale);
    if (st != ATTN_OK) return st;
    if (window < 1) return fail(ATTN_ERR_INVALID_ARG, "window must be >= 1 (got %d)", window);
    LaunchEnv env;
    st = device_env(stream, &env);
    if (st != ATTN_OK) return st;
    Shape s{B, Hq, Hkv, Tq, Tk, D, 1, scale};
    s.window = window;
    s.f16 = dtype == ATTN_F16 ? 1 : 0;
    return run_prefill(q, k, v, o, lse, s, env);
}

attn_status attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq,
                            int Hkv, int total_q, int total_k, int D, int causal, int window,
                            float scale, attn_dtype dtype, cudaStream_t stream) {
    if (dtype == ATTN_F32)
        return fail(ATTN_ERR_UNSUPPORTED, "packed sequences are implemented for 16-bit I/O only");
    if (dtype != ATTN_BF16 && dtype != ATTN_F16)
        return fail(ATTN_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dtype));
    if (B < 1 || Hq < 1 || Hkv < 1 || D < 1 || total_q < 0 || total_k < 0)
        return fail(ATTN_ERR_INVALID_ARG,
                    "B, Hq, Hkv, D must be >= 1 and total_q, total_k >= 0 (got %d, %d, %d, %d, %d, %d)",
                    B, Hq, Hkv, D, total_q, total_k);
    if (D != 64 && D != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim D=%d not supported (64 or 128)", D);
    if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
    if (!std::isfinite(scale) || !(scale > 0.0f))
        return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and positive (got %g)", (double)scale);
    if (window < 0) return fail(ATTN_ERR_INVALID_ARG, "window must be >= 0 (got %d)", window);
    if (window > 0 && !causal)
        return fail(ATTN_ERR_INVALID_ARG, "a sliding window needs the causal mask");
    if (total_q > 0x7fffffff - 1024 || total_k > 0x7fffffff - 1024 || B == 0x7fffffff)
        return fail(ATTN_ERR_INVALID_ARG, "total_q and total_k must be below 2^31 - 1024");
    if (total_q == 0) {  // nothing to compute (empty tensors may have null pointers)
        record_launch(0, 0, 0);
        return ok();
    }
    if (!q || !o || !cu_seqlens_q || !cu_seqlens_k || (total_k > 0 && (!k || !v)))
        return fail(ATTN_ERR_INVALID_ARG, "q, k, v, o, cu_seqlens_q and cu_seqlens_k must be non-null");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
        return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
    if (!aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4) || (lse && !aligned(lse, 4)))
        return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens_q, cu_seqlens_k and lse must be 4-byte aligned");
    VarlenShape s{B, Hq, Hkv, total_q, total_k, D, causal ? 1 : 0, window, scale};
    s.f16 = dtype == ATTN_F16 ? 1 : 0;
    const size_t bytes = varlen_workspace_bytes(s);
    if (bytes == 0)
        return fail(ATTN_ERR_INVALID_ARG, "too many work items (Hq * query blocks must fit in 31 bits)");
    LaunchEnv env;
    attn_status st = device_env(stream, &env);
    if (st != ATTN_OK) return st;
    PrefillMaps maps;
    const int box = prefill_box_rows();
    if (total_k > 0) {
        const bool f16 = s.f16 != 0;
        if ((st = make_map(q, total_q, Hq, D, box, 3, &maps.q, true, f16)) != ATTN_OK) return st;
        if ((st = make_map(k, total_k, Hkv, D, box, 3, &maps.k, true, f16)) != ATTN_OK) return st;
        if ((st = make_map(v, total_k, Hkv, D, box, 3, &maps.v, true, f16)) != ATTN_OK) return st;
    }
    void* ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, bytes, env.stream);
    if (e != cudaSuccess || ws == nullptr) {
        cudaGetLastError();
        return fail(ATTN_ERR_NO_MEMORY, "varlen workspace of %zu bytes: %s", bytes,
                    cudaGetErrorString(e));
    }
    VarlenSchedule sched{};
    int kernels = 0, grid = 0, k2 = 0;
    e = launch_varlen_schedule(cu_seqlens_q, cu_seqlens_k, s, ws, static_cast<uint16_t*>(o), lse,
                               env, &sched, &kernels);
    if (e == cudaSuccess && total_k > 0) {
        e = launch_prefill_packed_bf16(maps, static_cast<uint16_t*>(o), lse, s, sched, env, &grid,
                                       &k2);
        kernels += k2;
    }
    cudaError_t f = cudaFreeAsync(ws, env.stream);
    if (e == cudaSuccess && f != cudaSuccess) e = f;
    if (e != cudaSuccess) return cuda_fail(e, "varlen prefill launch");
    record_launch(grid, sched.item_bound, kernels);
    return ok();
}

attn_status attn_fwd_decode_paged(const void* q, const void* kv_cache, const int* block_table,
                                  const int* seq_lens, void* o, float* lse, int B, int Hq, int Hkv,
                                  int D, int page_size, int max_pages_per_seq, int num_blocks,
                                  float scale, attn_dtype dtype, cudaStream_t stream) {
    if (dtype == ATTN_F32)
        return fail(ATTN_ERR_UNSUPPORTED, "the paged decode is implemented for 16-bit I/O only");
    if (dtype != ATTN_BF16 && dtype != ATTN_F16)
        return fail(ATTN_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dtype));
    if (!q || !kv_cache || !block_table || !seq_lens || !o)
        return fail(ATTN_ERR_INVALID_ARG, "q, kv_cache, block_table, seq_lens and o must be non-null");
    if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(o, 16))
        return fail(ATTN_ERR_INVALID_ARG, "q, kv_cache and o must be 16-byte aligned");
    if (!aligned(block_table, 4) || !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)))
        return fail(ATTN_ERR_INVALID_ARG, "block_table, seq_lens and lse must be 4-byte aligned");
    if (B < 1 || Hq < 1 || Hkv < 1 || D < 1 || page_size < 1 || max_pages_per_seq < 1 ||
        num_blocks < 1)
        return fail(ATTN_ERR_INVALID_ARG,
                    "B, Hq, Hkv, D, page_size, max_pages_per_seq and num_blocks must be >= 1");
    if (D != 64 && D != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim D=%d not supported (64 or 128)", D);
    if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
    if (!std::isfinite(scale) || !(scale > 0.0f))
        return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and positive (got %g)", (double)scale);
    if (static_cast<long long>(B) * Hq > 0x7fffffffLL ||
        static_cast<long long>(B) * max_pages_per_seq > 0x7fffffffLL)
        return fail(ATTN_ERR_INVALID_ARG, "B*Hq and B*max_pages_per_seq must fit in 31 bits");
    if (static_cast<long long>(max_pages_per_seq) * page_size > 0x7fffffffLL - 1024)
        return fail(ATTN_ERR_INVALID_ARG, "max_pages_per_seq*page_size must be below 2^31 - 1024");
    LaunchEnv env;
    attn_status st = device_env(stream, &env);
    if (st != ATTN_OK) return st;
    PagedShape s{B, Hq, Hkv, D, page_size, max_pages_per_seq, num_blocks, scale};
    s.f16 = dtype == ATTN_F16 ? 1 : 0;
    const size_t bytes = decode_paged_workspace_bytes(s, env.num_sms);
    void* ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, bytes, env.stream);
    if (e != cudaSuccess || ws == nullptr) {
        cudaGetLastError();
        return fail(ATTN_ERR_NO_MEMORY, "paged decode workspace of %zu bytes: %s", bytes,
                    cudaGetErrorString(e));
    }
    int grid = 0, kernels = 0;
    e = launch_decode_paged_bf16(static_cast<const uint16_t*>(q),
                                 static_cast<const uint16_t*>(kv_cache),
                                 reinterpret_cast<const int32_t*>(block_table),
                                 reinterpret_cast<const int32_t*>(seq_lens),
                                 static_cast<uint16_t*>(o), lse, ws, s, env, &grid, &kernels);
    cudaError_t f = cudaFreeAsync(ws, env.stream);
    if (e == cudaSuccess && f != cudaSuccess) e = f;
    if (e != cudaSuccess) return cuda_fail(e, "paged decode launch");
    record_launch(grid, 0, kernels);
    return ok();
}

attn_status attn_get_device_status(cudaStream_t stream) {
    LaunchEnv env;
    attn_status st = device_env(stream, &env);
    if (st != ATTN_OK) return st;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned word = 0;
    e = cudaMemcpy(&word, env.status, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
    if (word != 0) {
        const unsigned zero = 0;
        e = cudaMemcpy(env.status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
    }
    constexpr unsigned kTimeoutBit = 1u, kBadInputBit = 2u;  // as the kernels set them (sm100.cuh)
    if (word & kTimeoutBit)
        return fail(ATTN_ERR_TIMEOUT, "a kernel pipeline wait timed out (site %u); outputs undefined",
                    (word >> 8) & 0xffu);
    if (word & kBadInputBit)
        return fail(ATTN_ERR_BAD_INPUT,
                    "a block id, sequence length or sequence offset was out of range (a safe "
                    "substitute was used, or the sequence was skipped); outputs undefined");
    return ok();
}

const char* attn_last_error(void) { return t_last_error.c_str(); }

void attn_last_launch_info(int* grid, int* items, int* kernels_launched) {
    if (grid) *grid = t_last_grid;
    if (items) *items = t_last_items;
    if (kernels_launched) *kernels_launched = t_last_kernels;
}

attn_status attn_diag_mma_tile(const void* a, const void* b, const void* v, float* s_out,
                               float* o_out, int D, cudaStream_t stream) {
    if (!a || !b || !v || !s_out || !o_out)
        return fail(ATTN_ERR_INVALID_ARG, "all pointers must be non-null");
    if (!aligned(a, 16) || !aligned(b, 16) || !aligned(v, 16))
        return fail(ATTN_ERR_INVALID_ARG, "a, b, v must be 16-byte aligned");
    if (D != 64 && D != 128) return fail(ATTN_ERR_UNSUPPORTED, "D must be 64 or 128");
    LaunchEnv env;
    attn_status st = device_env(stream, &env);
    if (st != ATTN_OK) return st;
    CUtensorMap ma, mb, mv;
    if ((st = make_map(a, 128, 1, D, 128, 2, &ma)) != ATTN_OK) return st;
    if ((st = make_map(b, 128, 1, D, 128, 2, &mb)) != ATTN_OK) return st;
    if ((st = make_map(v, 128, 1, D, 128, 2, &mv)) != ATTN_OK) return st;
    cudaError_t e = launch_diag_mma_tile(ma, mb, mv, s_out, o_out, D, env);
    if (e != cudaSuccess) return cuda_fail(e, "diag mma tile launch");
    record_launch(1, 1, 1);
    return ok();
}

attn_status attn_diag_wait_timeout(long long timeout_ns, cudaStream_t stream) {
    if (timeout_ns < 1000 || timeout_ns > 10LL * 1000 * 1000 * 1000)
        return fail(ATTN_ERR_INVALID_ARG, "timeout_ns must be in [1e3, 1e10]");
    LaunchEnv env;
    attn_status st = device_env(stream, &env);
    if (st != ATTN_OK) return st;
    cudaError_t e = launch_diag_wait_timeout(env, static_cast<uint64_t>(timeout_ns));
    if (e != cudaSuccess) return cuda_fail(e, "diag wait launch");
    record_launch(1, 1, 1);
    return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free decode (attn_fwd_decode_noalloc).
// ---------------------------------------------------------------------------
namespace attn {
namespace {

// Workspace of attn_fwd_decode_noalloc: a fixed array in the library's device
// image instead of memory allocated per call.  Every GPU that loads the
// library holds it until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64] = {};

// Device address of g_noalloc_scratch on the current device.  The host-side
// name of the array is only a stand-in, never a device address, so the
// address is looked up once per device (the first call on that device) with
// that device current.
attn_status noalloc_scratch(int dev, void** out) {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return ATTN_OK;
}

size_t noalloc_bytes(const Shape& s, int splits) {
    if (splits <= 1) return 0;
    return static_cast<size_t>(s.B) * s.Hq * splits * (s.D + 1) * sizeof(float);
}

int nonempty_splits(int splits, int Tk) {
    if (splits > 256) splits = 256;
    if (splits > Tk) splits = Tk;
    if (splits < 1) splits = 1;
    const int per = (Tk + splits - 1) / splits;
    return (Tk + per - 1) / per;
}

}  // namespace
}  // namespace attn

extern "C" attn_status attn_fwd_decode_noalloc(const void* q, const void* k, const void* v,
                                               void* o, float* lse, int B, int Hq, int Hkv,
                                               int Tk, int D, float scale, int num_splits,
                                               cudaStream_t stream) {
    using namespace attn;
    attn_status st = validate(q, k, v, o, lse, B, Hq, Hkv, 1, Tk, D, 0, scale);
    if (st != ATTN_OK) return st;
    if (num_splits < 0 || num_splits > 256)
        return fail(ATTN_ERR_INVALID_ARG, "num_splits must be in 0..256 (got %d)", num_splits);
    LaunchEnv env;
    st = device_env(stream, &env);
    if (st != ATTN_OK) return st;
    const Shape s{B, Hq, Hkv, 1, Tk, D, 0, scale};
    if (num_splits == 0) {
        const int ks = decode_group_splits(s, env.num_sms);
        if (ks > 1 && group_split_workspace_bytes(s, ks) <= kNoAllocScratchBytes) {
            void* ws = nullptr;
            st = noalloc_scratch(env.device, &ws);
            if (st != ATTN_OK) return st;
            return run_decode_as_split_prefill(q, k, v, o, lse, s, ks, ws, env);
        }
        if (ks == 1 && decode_prefers_prefill_kernel(s, env.num_sms))
            return run_decode_as_prefill(q, k, v, o, lse, s, env);  // no workspace at all
    }
    if (num_splits == 0 && !decode_prefers_split_kernel(s) &&
        decode_stream_workspace_bytes(s, env.num_sms) <= kNoAllocScratchBytes) {
        // Automatic mode: the stream-K kernels of attn_fwd_decode, their
        // fragments in the static array.
        void* ws = nullptr;
        st = noalloc_scratch(env.device, &ws);
        if (st != ATTN_OK) return st;
        int grid = 0, kernels = 0;
        cudaError_t e = launch_decode_stream_bf16(
            static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k),
            static_cast<const uint16_t*>(v), static_cast<uint16_t*>(o), lse,
            static_cast<float*>(ws), s, env, &grid, &kernels);
        if (e != cudaSuccess) return cuda_fail(e, "decode launch");
        record_launch(grid, 0, kernels);
        return ok();
    }
    // Explicit split counts, MHA, and automatic mode when the stream-K
    // fragments would not fit: the split kernel.
    int splits = nonempty_splits(num_splits > 0 ? num_splits : decode_choose_splits(s, env.num_sms), Tk);
    if (num_splits == 0)  // automatic count: lower it until the partials fit
        while (splits > 1 && noalloc_bytes(s, splits) > kNoAllocScratchBytes)
            splits = nonempty_splits(splits - 1, Tk);
    if (noalloc_bytes(s, splits) > kNoAllocScratchBytes)
        return fail(ATTN_ERR_UNSUPPORTED,
                    "decode with %d splits needs %zu bytes of scratch; the static workspace holds "
                    "%zu bytes (B*Hq*splits*(D+1)*4 must fit; pass fewer splits)",
                    splits, noalloc_bytes(s, splits), kNoAllocScratchBytes);
    float* ws_o = nullptr;
    float* ws_lse = nullptr;
    if (splits > 1) {
        void* ws = nullptr;
        st = noalloc_scratch(env.device, &ws);
        if (st != ATTN_OK) return st;
        ws_o = static_cast<float*>(ws);
        ws_lse = ws_o + static_cast<size_t>(B) * Hq * splits * D;
    }
    int kernels = 0;
    cudaError_t e = launch_decode_bf16(static_cast<const uint16_t*>(q),
                                       static_cast<const uint16_t*>(k),
                                       static_cast<const uint16_t*>(v), static_cast<uint16_t*>(o),
                                       lse, ws_o, ws_lse, s, splits, env, &kernels);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    record_launch(B * Hkv, splits, kernels);
    return ok();
}
