// decode_bf16.cu -- split-KV decode (one query row per (b, hq)) and the
// log-sum-exp combine.
//
// Decode is HBM bound: every K and V element is read once and serves all the
// query heads that share its KV head ("Attention 入门" §11.8.1 GQA,
// §11.8.2: decode is a 1 x N query against the cache;
// "Self-Attention机制深入理解" §11.2: decode attention is memory bound).  So
// this is CUDA-core code shaped for the memory system, not a GEMM:
//
//  * CTA = (b, hkv, chunk of HC query heads, split s); the split covers a
//    contiguous range of keys.  8 warps walk that range in blocks of KW keys.
//  * A key row (D bf16 = 128 or 256 bytes) is read by LPK = D/8 lanes with one
//    16-byte load each, so a warp load instruction covers 32*16 contiguous
//    bytes.  Each lane keeps the matching 8 query elements of every head.
//  * Partial dot products are finished with a butterfly reduce-scatter over
//    the LPK lanes: after log2(LPK) exchange steps each lane owns complete
//    scores for distinct (key, head) pairs, so the whole reduction costs
//    about one shuffle per score instead of one per lane.
//  * Online softmax in base 2 with a lazily updated running maximum: the
//    maximum is only moved (and the partial output rescaled) when a score
//    exceeds it by more than 2^8 ("Self-Attention机制深入理解" §7.3 and §12.3:
//    any common reference value gives the same normalised result).
//  * Each split writes its normalised partial output and its log-sum-exp;
//    the combine kernel merges the splits with the block-merge rule of §12.3.
//
// The default (automatic) mode is the stream-K kernel further down: the keys
// of all (b, hkv, head chunk) units are laid end to end and cut into one
// equal slice per SM; a producer warp bulk-copies each chunk of K and V rows
// into a shared-memory ring and eight consumer warps apply the arithmetic
// above (with the query columns and output accumulators as packed fp32
// pairs, two columns per f32x2 instruction).  Units cut by a slice boundary
// leave fragments that a combine kernel merges (one block per slice
// boundary, launched so that it is scheduled while the stream kernel runs).
// The same kernel reads a paged cache (kPaged: per-request lengths summed by
// every CTA, block-table indirection, two producer warps on alternate chunks
// whose lanes issue a chunk's per-block copies together) and fp16 instead of
// bf16 elements (kF16).
#include <cuda_runtime.h>
#include <cmath>
#include <cstdint>

#include "attn_internal.h"
#include "sm100.cuh"

namespace attn {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kNK = 4;  // keys per lane group per iteration
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint4 ld_stream_v4(const uint16_t* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(reinterpret_cast<uint64_t>(p)));
    return r;
}

// Eight 16-bit elements (bf16, or fp16 with kF16) -> fp32 (exact).
template <bool kF16 = false>
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    using E = Elem16<kF16>;
    f[0] = E::lo(u.x); f[1] = E::hi(u.x);
    f[2] = E::lo(u.y); f[3] = E::hi(u.y);
    f[4] = E::lo(u.z); f[5] = E::hi(u.z);
    f[6] = E::lo(u.w); f[7] = E::hi(u.w);
}

__device__ __forceinline__ float warp_allmax(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, m));
    return x;
}
__device__ __forceinline__ float warp_allsum(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

// Reduce-scatter of V values over the LPK lanes of a lane group (xor masks
// LPK/2 .. 1).  On return vals[0..NV) hold complete sums; see own_index().
template <int V, int LPK>
__device__ __forceinline__ void group_reduce_scatter(float (&vals)[V], int lane) {
    int cur = V;
#pragma unroll
    for (int m = LPK / 2; m >= 1; m >>= 1) {
        if (cur > 1) {
            const int half = cur / 2;
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                if (i < half) {
                    const float send = upper ? vals[i] : vals[i + half];
                    const float keep = upper ? vals[i + half] : vals[i];
                    vals[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                }
            }
            cur = half;
        } else {
            vals[0] += __shfl_xor_sync(0xffffffffu, vals[0], m);
        }
    }
}

// Index (key slot * HC + head) of the r-th complete value a lane owns after
// group_reduce_scatter, and whether this lane is the canonical owner (for
// V < LPK several lanes hold the same value).
template <int V, int LPK>
__device__ __forceinline__ int own_index(int sub, int r) {
    if constexpr (V >= LPK) return sub * (V / LPK) + r;
    else return sub / (LPK / V);
}
template <int V, int LPK>
__device__ __forceinline__ bool own_canonical(int sub) {
    if constexpr (V >= LPK) return true;
    else return (sub % (LPK / V)) == 0;
}

struct DecodeParams {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    uint16_t* o;
    float* lse;
    float* ws_o;
    float* ws_lse;
    int Hq, Hkv, Tk, splits, keys_per_split;
    float scale_log2;
};

template <int D, int HC>
__global__ void __launch_bounds__(kThreads)
decode_split_kernel(const DecodeParams p) {
    constexpr int LPK = D / 8;          // lanes per key row
    constexpr int KPL = 32 / LPK;       // keys per warp load instruction
    constexpr int KW = KPL * kNK;       // keys per warp iteration
    constexpr int NV0 = kNK * HC;       // partial values per lane before reduction
    constexpr int NV = NV0 >= LPK ? NV0 / LPK : 1;

    __shared__ __align__(16) float s_p[kWarps][KPL][NV0];
    __shared__ float s_m[kWarps][HC];
    __shared__ float s_l[kWarps][HC];
    __shared__ __align__(16) float s_acc[kWarps][HC][D];

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int grp = lane / LPK, sub = lane % LPK;
    const int pair = blockIdx.x;  // b * Hkv + hkv
    const int chunk = blockIdx.y;
    const int split = blockIdx.z;
    const int group = p.Hq / p.Hkv;
    const int b = pair / p.Hkv, hkv = pair % p.Hkv;
    const int hq0 = hkv * group + chunk * HC;

    const int kbeg = split * p.keys_per_split;
    const int kend = min(p.Tk, kbeg + p.keys_per_split);

    // This lane's 8 query elements of each head, pre-scaled so scores come
    // out in log2 units.
    float qf[HC][8];
#pragma unroll
    for (int h = 0; h < HC; ++h) {
        const uint16_t* qp = p.q + (static_cast<int64_t>(b) * p.Hq + hq0 + h) * D + sub * 8;
        const uint4 u = *reinterpret_cast<const uint4*>(qp);
        unpack8(u, qf[h]);
#pragma unroll
        for (int e = 0; e < 8; ++e) qf[h][e] *= p.scale_log2;
    }

    const uint16_t* kbase = p.k + static_cast<int64_t>(pair) * p.Tk * D + sub * 8;
    const uint16_t* vbase = p.v + static_cast<int64_t>(pair) * p.Tk * D + sub * 8;

    float m[HC];        // running maximum per head (warp-uniform)
    float acc[HC][8];   // partial output, this lane's 8 columns
    float lsum[NV];     // running sums of the values this lane owns
#pragma unroll
    for (int h = 0; h < HC; ++h) {
        m[h] = -INFINITY;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] = 0.0f;
    }
#pragma unroll
    for (int r = 0; r < NV; ++r) lsum[r] = 0.0f;

    for (int kb = kbeg + warp * KW; kb < kend; kb += kWarps * KW) {
        uint4 kr[kNK], vr[kNK];
#pragma unroll
        for (int n = 0; n < kNK; ++n) {
            const int key = kb + n * KPL + grp;
            if (key < kend) {
                kr[n] = ld_stream_v4(kbase + static_cast<int64_t>(key) * D);
                vr[n] = ld_stream_v4(vbase + static_cast<int64_t>(key) * D);
            } else {
                kr[n] = make_uint4(0, 0, 0, 0);
                vr[n] = make_uint4(0, 0, 0, 0);
            }
        }
        // Partial dot products over this lane's 8 columns.
        float part[NV0];
#pragma unroll
        for (int n = 0; n < kNK; ++n) {
            float kf[8];
            unpack8(kr[n], kf);
#pragma unroll
            for (int h = 0; h < HC; ++h) {
                float s = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e) s = fmaf(qf[h][e], kf[e], s);
                part[n * HC + h] = s;
            }
        }
        group_reduce_scatter<NV0, LPK>(part, lane);

        // Scores this lane owns; mask keys past the end of the split.
        float x[NV];
        int hown[NV];
        bool need = false;
#pragma unroll
        for (int r = 0; r < NV; ++r) {
            const int idx = own_index<NV0, LPK>(sub, r);
            const int n = idx / HC;
            hown[r] = idx % HC;
            const int key = kb + n * KPL + grp;
            x[r] = key < kend ? part[r] : -INFINITY;
            float mh = m[0];
#pragma unroll
            for (int h = 1; h < HC; ++h) mh = (hown[r] == h) ? m[h] : mh;
            need |= x[r] > mh + kRescaleThreshold;
        }
        if (__any_sync(0xffffffffu, need)) {
            // Move each head's maximum to the exact running maximum.
#pragma unroll
            for (int h = 0; h < HC; ++h) {
                float cm = -INFINITY;
#pragma unroll
                for (int r = 0; r < NV; ++r) cm = (hown[r] == h) ? fmaxf(cm, x[r]) : cm;
                cm = warp_allmax(cm);
                const float mnew = fmaxf(m[h], cm);
                const float alpha = (m[h] == -INFINITY) ? 0.0f : ex2_approx(m[h] - mnew);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[h][e] *= alpha;
#pragma unroll
                for (int r = 0; r < NV; ++r) lsum[r] = (hown[r] == h) ? lsum[r] * alpha : lsum[r];
                m[h] = mnew;
            }
        }
        // Weights; publish them to the lane group through shared memory.
#pragma unroll
        for (int r = 0; r < NV; ++r) {
            float mh = m[0];
#pragma unroll
            for (int h = 1; h < HC; ++h) mh = (hown[r] == h) ? m[h] : mh;
            const float pr = (x[r] == -INFINITY) ? 0.0f : ex2_approx(x[r] - mh);
            lsum[r] += pr;
            if (own_canonical<NV0, LPK>(sub)) s_p[warp][grp][own_index<NV0, LPK>(sub, r)] = pr;
        }
        __syncwarp();
        float pall[NV0];
#pragma unroll
        for (int i = 0; i < NV0; i += 4) {
            const float4 t = *reinterpret_cast<const float4*>(&s_p[warp][grp][i]);
            pall[i] = t.x; pall[i + 1] = t.y; pall[i + 2] = t.z; pall[i + 3] = t.w;
        }
        __syncwarp();
        // acc += P V over this lane's 8 columns.
#pragma unroll
        for (int n = 0; n < kNK; ++n) {
            float vf[8];
            unpack8(vr[n], vf);
#pragma unroll
            for (int h = 0; h < HC; ++h) {
                const float pw = pall[n * HC + h];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(pw, vf[e], acc[h][e]);
            }
        }
    }

    // Merge the lane groups of this warp (they share the warp-uniform max).
#pragma unroll
    for (int mask = LPK; mask < 32; mask <<= 1) {
#pragma unroll
        for (int h = 0; h < HC; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], mask);
    }
    float lw[HC];
#pragma unroll
    for (int h = 0; h < HC; ++h) {
        float t = 0.0f;
        if (own_canonical<NV0, LPK>(sub)) {
#pragma unroll
            for (int r = 0; r < NV; ++r) t += ((own_index<NV0, LPK>(sub, r) % HC) == h) ? lsum[r] : 0.0f;
        }
        lw[h] = warp_allsum(t);
    }
    if (lane < LPK) {
#pragma unroll
        for (int h = 0; h < HC; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) s_acc[warp][h][sub * 8 + e] = acc[h][e];
    }
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < HC; ++h) {
            s_m[warp][h] = m[h];
            s_l[warp][h] = lw[h];
        }
    }
    __syncthreads();

    // Merge the warps (block-merge rule) and write this split's result.
    for (int idx = threadIdx.x; idx < HC * D; idx += kThreads) {
        const int h = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][h]);
        float L = 0.0f, O = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float wt = (s_m[w][h] == -INFINITY) ? 0.0f : ex2_approx(s_m[w][h] - M);
            L = fmaf(s_l[w][h], wt, L);
            O = fmaf(s_acc[w][h][d], wt, O);
        }
        const int64_t row = static_cast<int64_t>(b) * p.Hq + hq0 + h;  // (b, hq)
        const float out = O / L;
        const float lse2 = M + __log2f(L);
        if (p.splits == 1) {
            const uint32_t pk = pack_bf16x2(out, 0.0f);
            p.o[row * D + d] = static_cast<uint16_t>(pk & 0xffffu);
            if (d == 0 && p.lse != nullptr) p.lse[row] = lse2 * kLn2;
        } else {
            p.ws_o[(row * p.splits + split) * D + d] = out;
            if (d == 0) p.ws_lse[row * p.splits + split] = lse2;
        }
    }
}

// Merge the splits of one (b, hq): lse = log sum_s e^{lse_s},
// O = sum_s e^{lse_s - lse} O_s (all in base 2 internally).
template <int D, bool kF16 = false>
__global__ void __launch_bounds__(D)
decode_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                      uint16_t* __restrict__ o, float* __restrict__ lse, int splits) {
    extern __shared__ float s_w[];
    const int64_t row = blockIdx.x;
    const int d = threadIdx.x;
    const float* l2 = ws_lse + row * splits;
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, l2[s]);
    float L = 0.0f;
    for (int s = d; s < splits; s += D) s_w[s] = ex2_approx(l2[s] - M);
    __syncthreads();
    for (int s = 0; s < splits; ++s) L += s_w[s];
    float acc = 0.0f;
    const float* op = ws_o + row * splits * D + d;
    for (int s = 0; s < splits; ++s) acc = fmaf(s_w[s], op[static_cast<int64_t>(s) * D], acc);
    const uint32_t pk = Elem16<kF16>::pack(acc / L, 0.0f);
    o[row * D + d] = static_cast<uint16_t>(pk & 0xffffu);
    if (d == 0 && lse != nullptr) lse[row] = (M + __log2f(L)) * kLn2;
}

template <int D, int HC>
cudaError_t launch_split(const DecodeParams& p, int pairs, int chunks, cudaStream_t st) {
    dim3 grid(pairs, chunks, p.splits);
    decode_split_kernel<D, HC><<<grid, kThreads, 0, st>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_split_d(const DecodeParams& p, int hc, int pairs, int chunks,
                           cudaStream_t st) {
    switch (hc) {
        case 8: return launch_split<D, 8>(p, pairs, chunks, st);
        case 4: return launch_split<D, 4>(p, pairs, chunks, st);
        case 2: return launch_split<D, 2>(p, pairs, chunks, st);
        default: return launch_split<D, 1>(p, pairs, chunks, st);
    }
}

int heads_per_cta(int group) {
    for (int hc : {8, 4, 2, 1})
        if (group % hc == 0) return hc;
    return 1;
}

// Resident CTAs per SM of the split kernel used for this shape.
int split_kernel_occupancy(int D, int hc) {
    int n = 0;
    cudaError_t e = cudaSuccess;
#define ATTN_OCC(DD, HH) \
    if (D == DD && hc == HH) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_split_kernel<DD, HH>, kThreads, 0);
    ATTN_OCC(64, 1) ATTN_OCC(64, 2) ATTN_OCC(64, 4) ATTN_OCC(64, 8)
    ATTN_OCC(128, 1) ATTN_OCC(128, 2) ATTN_OCC(128, 4) ATTN_OCC(128, 8)
#undef ATTN_OCC
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return n > 0 ? n : 1;
}

}  // namespace

// Split count: maximise the fill of the last wave of CTAs (waves / ceil(waves)
// over the SM slots the kernel can occupy), minus a small charge per split for
// the partial results each split writes and the combine reads; at least 256
// keys per split.
int decode_choose_splits(const Shape& s, int num_sms) {
    const int group = s.Hq / s.Hkv;
    const int hc = heads_per_cta(group);
    const int chunks = group / hc;
    const double ctas = static_cast<double>(s.B) * s.Hkv * chunks;
    const double slots = static_cast<double>(num_sms) * split_kernel_occupancy(s.D, hc);
    int max_s = (s.Tk + 255) / 256;
    if (max_s > 16) max_s = 16;
    if (max_s < 1) max_s = 1;
    int best = 1;
    double best_score = -1.0;
    for (int sp = 1; sp <= max_s; ++sp) {
        const double waves = ctas * sp / slots;
        const double fill = waves / std::ceil(waves);
        const double score = fill - 0.01 * sp;
        if (score > best_score + 1e-9) {
            best_score = score;
            best = sp;
        }
    }
    return best;
}

size_t decode_workspace_bytes(const Shape& s, int splits) {
    if (splits <= 1) return 0;
    const size_t rows = static_cast<size_t>(s.B) * s.Hq;
    return rows * splits * s.D * sizeof(float) + rows * splits * sizeof(float) + 256;
}

cudaError_t launch_decode_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               uint16_t* o, float* lse, float* ws_o, float* ws_lse,
                               const Shape& s, int splits, const LaunchEnv& env,
                               int* kernels_launched) {
    const int group = s.Hq / s.Hkv;
    const int hc = heads_per_cta(group);
    const int chunks = group / hc;
    const int pairs = s.B * s.Hkv;
    if (chunks > 65535) return cudaErrorInvalidConfiguration;
    DecodeParams p;
    p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse; p.ws_o = ws_o; p.ws_lse = ws_lse;
    p.Hq = s.Hq; p.Hkv = s.Hkv; p.Tk = s.Tk; p.splits = splits;
    p.keys_per_split = (s.Tk + splits - 1) / splits;
    p.scale_log2 = s.scale * 1.4426950408889634f;
    cudaError_t e = (s.D == 64) ? launch_split_d<64>(p, hc, pairs, chunks, env.stream)
                                : launch_split_d<128>(p, hc, pairs, chunks, env.stream);
    int launched = 1;
    if (e == cudaSuccess && splits > 1) {
        const int rows = s.B * s.Hq;
        const size_t sh = static_cast<size_t>(splits) * sizeof(float);
        if (s.D == 64)
            decode_combine_kernel<64><<<rows, 64, sh, env.stream>>>(ws_o, ws_lse, o, lse, splits);
        else
            decode_combine_kernel<128><<<rows, 128, sh, env.stream>>>(ws_o, ws_lse, o, lse, splits);
        e = cudaGetLastError();
        launched = 2;
    }
    if (kernels_launched) *kernels_launched = launched;
    return e;
}

cudaError_t launch_decode_combine(const float* ws_o, const float* ws_lse, uint16_t* o, float* lse,
                                  int rows, int D, int splits, bool f16, const LaunchEnv& env) {
    const size_t sh = static_cast<size_t>(splits) * sizeof(float);
    if (f16) {
        if (D == 64)
            decode_combine_kernel<64, true><<<rows, 64, sh, env.stream>>>(ws_o, ws_lse, o, lse, splits);
        else
            decode_combine_kernel<128, true><<<rows, 128, sh, env.stream>>>(ws_o, ws_lse, o, lse, splits);
    } else if (D == 64) {
        decode_combine_kernel<64><<<rows, 64, sh, env.stream>>>(ws_o, ws_lse, o, lse, splits);
    } else {
        decode_combine_kernel<128><<<rows, 128, sh, env.stream>>>(ws_o, ws_lse, o, lse, splits);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Stream-K decode (automatic mode).
//
// One persistent CTA per SM.  The keys of all (b, hkv, head chunk) units are
// laid end to end and cut into one equal contiguous slice per CTA, so every
// CTA streams the same number of bytes whatever B, Hkv and Tk are.  A slice
// covers whole units and at most two unit fragments; a unit cut by slice
// boundaries is merged by the combine kernel (block-merge rule,
// "Self-Attention机制深入理解" §12.3).  A producer warp copies each chunk of K
// and V rows (contiguous in the cache) into a shared-memory ring with bulk
// copies (paged cache: two producer warps, alternate chunks); eight compute
// warps consume the ring with the same arithmetic as the split kernel above.
// ---------------------------------------------------------------------------
namespace {

constexpr int kStreamWarps = 8;
// Producer warps: the dense cache needs one lane of one; the paged cache's
// per-block copies take all of them, on alternate chunks.
constexpr int kProducerWarps = 2;
constexpr int kStreamThreads = (kStreamWarps + kProducerWarps) * 32;
constexpr int kStageBytes = 32 * 1024;                   // K half + V half
constexpr int kStreamStages = 5;
// Paged mode: up to this many requests, every CTA computes the prefix of the
// request lengths itself, in shared memory; more run a prefix kernel first.
constexpr int kMaxPrefixB = 1024;

// Programmatic dependent launch: a grid launched with programmatic stream
// serialisation may start while the grid before it in the stream is still
// running.  It must wait for that grid (and its memory operations) before
// reading what the grid wrote; in a grid launched without the attribute the
// wait returns at once.  The earlier grid signals that its dependants may be
// scheduled once all its CTAs are resident.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

enum : unsigned { SITE_DEC_FULL = 40, SITE_DEC_EMPTY, SITE_DEC_SEG };

// Paged cache ("第 11 章 · Attention 入门", 11.11, the KV-cache / VMM passage:
// physical blocks of `page` tokens hold the K and V rows of those tokens for
// every KV head; block_table[req][t / page] names the block of token t).
struct PagedParams {
    const uint16_t* kv;          // [num_blocks, 2, Hkv, page, D], 0 = K, 1 = V
    const int32_t* block_table;  // [B, max_pages]
    const int32_t* seq_lens;     // [B] keys of each request
    // [B + 1] keys of requests 0..b-1 and [2] total virtual keys, keys per
    // CTA: written by the prefix kernel (in_kernel == 0) or, when every CTA
    // computes them itself (in_kernel == 1), by CTA 0 for the combine kernel.
    long long* cum;
    long long* geom;
    // [grid] for CTA c >= 1: the unit its slice starts in, {b, hkv * chunks +
    // chunk, offset of the slice start in the unit, unit length} (combine).
    int4* first_unit;
    int B, page, max_pages, num_blocks;
    int in_kernel;
};

struct StreamParams {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    uint16_t* o;
    float* lse;
    float* ws_o;
    float* ws_lse;
    int Hq, Hkv, Tk, group, chunks, nseg_max;
    long long total, per_cta;
    float scale_log2;
    unsigned* status;
    unsigned long long limit_ns;
    PagedParams pg;
};

struct StreamBars {
    uint64_t full[kStreamStages], empty[kStreamStages];
    uint64_t seg_in, seg_out;
    long long scan[32];  // paged mode: per-warp totals of the length prefix
    int abort;
};

template <int D, int HC, bool kPaged = false>
struct StreamLayout {
    static constexpr int LPK = D / 8;
    static constexpr int KPL = 32 / LPK;
    static constexpr int KW = KPL * kNK;
    static constexpr int NV0 = kNK * HC;
    static constexpr int CK = kStageBytes / (2 * D * 2);  // keys per chunk
    static_assert(CK == kStreamWarps * KW, "one warp iteration per warp per chunk");
    static constexpr int kRingOff = 0;
    static constexpr int kAccOff = kRingOff + kStreamStages * kStageBytes;
    static constexpr int kPOff = kAccOff + kStreamWarps * HC * D * 4;
    static constexpr int kMOff = kPOff + kStreamWarps * KPL * NV0 * 4;
    static constexpr int kLOff = kMOff + kStreamWarps * HC * 4;
    static constexpr int kBarOff = (kLOff + kStreamWarps * HC * 4 + 15) / 16 * 16;
    static constexpr int kCumOff = (kBarOff + static_cast<int>(sizeof(StreamBars)) + 15) / 16 * 16;
    static constexpr int kBytes = kCumOff + (kPaged ? (kMaxPrefixB + 1) * 8 : 0) + 128;
};

// One unit (request b, KV head hkv, head chunk) fragment [k0, k1) of its L
// keys; u numbers the units in (b, hkv, chunk) order.
struct Segment {
    long long u;
    int b, hkv, chunk;
    int k0, k1, L;
};

// Next fragment inside the virtual key range [v, v1): every unit has Tk keys.
__device__ __forceinline__ bool next_segment(long long& v, long long v1, const StreamParams& p,
                                             Segment& sg) {
    if (v >= v1) return false;
    const int Tk = p.Tk;
    sg.u = v / Tk;
    sg.L = Tk;
    sg.k0 = static_cast<int>(v - sg.u * Tk);
    const long long rem = v1 - v;
    sg.k1 = static_cast<int>(rem < Tk - sg.k0 ? sg.k0 + rem : Tk);
    const long long pair = sg.u / p.chunks;
    sg.chunk = static_cast<int>(sg.u - pair * p.chunks);
    sg.b = static_cast<int>(pair / p.Hkv);
    sg.hkv = static_cast<int>(pair % p.Hkv);
    v += sg.k1 - sg.k0;
    return true;
}

// The same with per-request lengths: request b's units start at
// cum[b] * (Hkv * chunks), each L_b = cum[b + 1] - cum[b] keys long.
__device__ __forceinline__ bool next_segment_paged(long long& v, long long v1,
                                                   const StreamParams& p, const long long* cum,
                                                   Segment& sg) {
    if (v >= v1) return false;
    const long long U = static_cast<long long>(p.Hkv) * p.chunks;
    int lo = 0, hi = p.pg.B - 1;  // last request whose first unit starts at or before v
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cum[mid] * U <= v) lo = mid; else hi = mid - 1;
    }
    const long long L = cum[lo + 1] - cum[lo];  // > 0: v lies inside request lo
    const long long r = v - cum[lo] * U;
    const long long w = r / L;
    sg.b = lo;
    sg.hkv = static_cast<int>(w / p.chunks);
    sg.chunk = static_cast<int>(w - static_cast<long long>(sg.hkv) * p.chunks);
    sg.u = static_cast<long long>(lo) * U + w;
    sg.L = static_cast<int>(L);
    sg.k0 = static_cast<int>(r - w * L);
    const long long rem = v1 - v;
    sg.k1 = static_cast<int>(rem < L - sg.k0 ? sg.k0 + rem : L);
    v += sg.k1 - sg.k0;
    return true;
}

// Block id of page `page` of request b, checked against the pool: an id
// outside it is reported in the status word and block 0 is used instead, so
// the copy stays inside the pool and the stage still receives the bytes its
// barrier expects.
__device__ __forceinline__ int paged_block_id_load(const StreamParams& p, int b, int page) {
    return p.pg.block_table[static_cast<int64_t>(b) * p.pg.max_pages + page];
}
__device__ __forceinline__ int paged_block_id_check(const StreamParams& p, int blk) {
    if (blk < 0 || blk >= p.pg.num_blocks) {
        atomicOr(p.status, ATTN_DEV_BAD_INPUT);
        blk = 0;
    }
    return blk;
}
__device__ __forceinline__ int paged_block_id(const StreamParams& p, int b, int page) {
    return paged_block_id_check(p, paged_block_id_load(p, b, page));
}

// Paged mode, every CTA: cum[b] = keys of requests 0..b-1 in shared memory
// (B <= kMaxPrefixB), with each length clamped into 0 .. max_pages * page
// (CTA 0 reports a length outside it in the status word).  Every thread of
// the CTA takes part.
__device__ void block_length_prefix(const StreamParams& p, long long* cum, long long* warp_tot) {
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int B = p.pg.B, max_keys = p.pg.max_pages * p.pg.page;
    const int per = (B + nt - 1) / nt;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    long long mine = 0;
    for (int b = b0; b < b1; ++b) {
        int L = p.pg.seq_lens[b];
        if (L < 0 || L > max_keys) {
            if (blockIdx.x == 0) atomicOr(p.status, ATTN_DEV_BAD_INPUT);
            L = L < 0 ? 0 : max_keys;
        }
        mine += L;
    }
    // Exclusive scan of the per-thread sums: within warps, then across warps.
    long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        long long w = lane < nt / 32 ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    long long run = incl - mine + (warp > 0 ? warp_tot[warp - 1] : 0);
    for (int b = b0; b < b1; ++b) {
        cum[b] = run;
        const int L = p.pg.seq_lens[b];
        run += L < 0 ? 0 : (L > max_keys ? max_keys : L);
    }
    if (tid == nt - 1) cum[B] = run;  // the last thread's range ends at B (or is empty)
    __syncthreads();
}

// Ten warps put three on two SM sub-partitions, whose 16K registers cap a
// thread at 168 (HC = 8 spills a little; splitting the heads would re-read K/V).
// kPaged: keys come from the paged cache, per-request lengths, and cut units
// leave their fragments in per-CTA slots (first segment of the CTA: slot 0,
// last: slot 1).
template <int D, int HC, bool kPaged, bool kF16 = false>
__global__ void __launch_bounds__(kStreamThreads, 1)
decode_stream_kernel(const StreamParams p) {
    using L = StreamLayout<D, HC, kPaged>;
    constexpr int LPK = L::LPK, KPL = L::KPL, KW = L::KW, NV0 = L::NV0, CK = L::CK;
    constexpr int NV = NV0 >= LPK ? NV0 / LPK : 1;
    constexpr int kHalf = kStageBytes / 2;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    float (*s_acc)[HC][D] = reinterpret_cast<float (*)[HC][D]>(smem + L::kAccOff);
    float (*s_p)[KPL][NV0] = reinterpret_cast<float (*)[KPL][NV0]>(smem + L::kPOff);
    float (*s_m)[HC] = reinterpret_cast<float (*)[HC]>(smem + L::kMOff);
    float (*s_l)[HC] = reinterpret_cast<float (*)[HC]>(smem + L::kLOff);
    StreamBars* bars = reinterpret_cast<StreamBars*>(smem + L::kBarOff);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStreamStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], kStreamWarps);
        }
        mbar_init(&bars->seg_in, kStreamWarps);
        mbar_init(&bars->seg_out, kStreamWarps);
        bars->abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitGuard g{p.status, &bars->abort, p.limit_ns};
    long long total = p.total, per_cta = p.per_cta;
    const long long* cum = nullptr;
    if constexpr (kPaged) {
        const long long units_per_req = static_cast<long long>(p.Hkv) * p.chunks;
        if (p.pg.in_kernel) {
            long long* s_cum = reinterpret_cast<long long*>(smem + L::kCumOff);
            block_length_prefix(p, s_cum, bars->scan);
            cum = s_cum;
            total = s_cum[p.pg.B] * units_per_req;
            per_cta = total > 0 ? (total + gridDim.x - 1) / gridDim.x : 1;
            if (blockIdx.x == 0) {  // for the combine kernel
                for (int i = threadIdx.x; i <= p.pg.B; i += blockDim.x) p.pg.cum[i] = s_cum[i];
                if (threadIdx.x == 0) {
                    p.pg.geom[0] = total;
                    p.pg.geom[1] = per_cta;
                }
            }
        } else {
            cum = p.pg.cum;
            total = p.pg.geom[0];
            per_cta = p.pg.geom[1];
        }
        // Requests without keys: O = 0 and lse = -inf (no slice covers them).
        for (int b = blockIdx.x; b < p.pg.B; b += gridDim.x) {
            if (cum[b + 1] != cum[b]) continue;
            for (int i = threadIdx.x; i < p.Hq * D; i += blockDim.x)
                p.o[static_cast<int64_t>(b) * p.Hq * D + i] = 0;
            if (p.lse != nullptr)
                for (int i = threadIdx.x; i < p.Hq; i += blockDim.x)
                    p.lse[static_cast<int64_t>(b) * p.Hq + i] = -INFINITY;
        }
    }
    grid_launch_dependents();
    const long long v_begin = static_cast<long long>(blockIdx.x) * per_cta;
    const long long v_end = v_begin + per_cta < total ? v_begin + per_cta : total;
    auto next = [&](long long& vv, Segment& sg) {
        return kPaged ? next_segment_paged(vv, v_end, p, cum, sg) : next_segment(vv, v_end, p, sg);
    };
    if constexpr (kPaged) {
        if (threadIdx.x == 0 && blockIdx.x > 0) {
            long long vv = v_begin;
            Segment sg0;
            if (next(vv, sg0))
                p.pg.first_unit[blockIdx.x] =
                    make_int4(sg0.b, sg0.hkv * p.chunks + sg0.chunk, sg0.k0, sg0.L);
        }
    }

    if (warp >= kStreamWarps && kPaged) {
        // Producers (paged): the producer warps take alternate chunks, and
        // the lanes of a warp issue a chunk's copies together.  Lane 2i
        // copies the K rows of the chunk's page i and lane 2i+1 its V rows;
        // each lane loads and checks its own block id, so the ids, the
        // address arithmetic and the copies of up to 8 pages take one pass
        // instead of a serial chain in one lane.  Pages beyond the first 8
        // (blocks of fewer than 8 keys) repeat the pass.  (Loading the next
        // chunk's ids while this chunk is issued measured slower: a lane's
        // outstanding loads delay its copy issue.)  Every lane runs the same
        // loop and waits on the stage barrier by itself: no warp-wide vote or
        // shuffle, which would wait for the issued copies to be taken by the
        // copy engine.  Page arithmetic uses shifts for power-of-two pages.
        const uint32_t pw = static_cast<uint32_t>(warp - kStreamWarps);
        const int P = p.pg.page;
        const int pshift = (P & (P - 1)) == 0 ? __ffs(P) - 1 : -1;
        const int pi = lane >> 1;
        const bool is_v = (lane & 1) != 0;
        const int64_t head_rows = static_cast<int64_t>(P) * D;
        const int64_t block_elems = 2 * static_cast<int64_t>(p.Hkv) * head_rows;
        uint32_t it = 0;
        long long v = v_begin;
        Segment sg;
        bool ok = true;
        while (ok && next(v, sg)) {
            const uint16_t* seg_base = p.pg.kv + static_cast<int64_t>(sg.hkv) * head_rows +
                                       (is_v ? static_cast<int64_t>(p.Hkv) * head_rows : 0);
            for (int kc = sg.k0; kc < sg.k1; kc += CK, ++it) {
                if (it % kProducerWarps != pw) continue;
                const int n = min(CK, sg.k1 - kc);
                const int s = it % kStreamStages;
                const int pg0 = pshift >= 0 ? kc >> pshift : kc / P;
                const int np = (pshift >= 0 ? (kc + n - 1) >> pshift : (kc + n - 1) / P) - pg0 + 1;
                // The block id is loaded before the stage wait and checked
                // after it, so that the load's latency overlaps the wait.
                int id = (lane < 16 && pi < np) ? paged_block_id_load(p, sg.b, pg0 + pi) : 0;
                if (it >= (uint32_t)kStreamStages &&
                    !mbar_wait(&bars->empty[s], ((it / kStreamStages) & 1) ^ 1, g, SITE_DEC_EMPTY)) {
                    ok = false;
                    break;
                }
                if (lane < 16 && pi < np) id = paged_block_id_check(p, id);
                uint8_t* stage = smem + L::kRingOff + s * kStageBytes;
                if (lane == 0)
                    mbar_arrive_expect_tx(&bars->full[s], 2u * static_cast<uint32_t>(n) * D * 2);
                for (int r0 = 0; r0 < np; r0 += 8) {
                    if (r0 > 0) id = (lane < 16 && r0 + pi < np) ? paged_block_id(p, sg.b, pg0 + r0 + pi) : 0;
                    const int page = pg0 + r0 + pi;
                    if (lane < 16 && r0 + pi < np) {
                        const int t = max(kc, page * P);
                        const int t1 = min(kc + n, page * P + P);
                        const uint16_t* src = seg_base + static_cast<int64_t>(id) * block_elems +
                                              static_cast<int64_t>(t - page * P) * D;
                        bulk_load(stage + (is_v ? kHalf : 0) + (t - kc) * D * 2, src,
                                  static_cast<uint32_t>(t1 - t) * D * 2, &bars->full[s]);
                    }
                }
            }
        }
        if (!ok && lane == 0) {
            // Let copies already in flight land before the CTA leaves.
            for (uint32_t i = (it > (uint32_t)kStreamStages ? it - kStreamStages : 0); i < it; ++i) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&bars->full[i % kStreamStages], (i / kStreamStages) & 1))
                    if (global_timer_ns() - t0 > 200000000ull) break;
            }
        }
    } else if (warp == kStreamWarps) {
        // Producer: bulk-copy every chunk of this CTA's slice into the ring.
        if (lane == 0) {
            uint32_t it = 0;
            long long v = v_begin;
            Segment sg;
            while (next(v, sg)) {
                const long long pair = static_cast<long long>(sg.b) * p.Hkv + sg.hkv;
                for (int kc = sg.k0; kc < sg.k1; kc += CK, ++it) {
                    const int n = min(CK, sg.k1 - kc);
                    const int s = it % kStreamStages;
                    if (it >= (uint32_t)kStreamStages &&
                        !mbar_wait(&bars->empty[s], ((it / kStreamStages) & 1) ^ 1, g, SITE_DEC_EMPTY))
                        goto drain;
                    const uint32_t bytes = static_cast<uint32_t>(n) * D * 2;
                    uint8_t* stage = smem + L::kRingOff + s * kStageBytes;
                    mbar_arrive_expect_tx(&bars->full[s], 2 * bytes);
                    const int64_t row = pair * p.Tk + kc;
                    bulk_load(stage, p.k + row * D, bytes, &bars->full[s]);
                    bulk_load(stage + kHalf, p.v + row * D, bytes, &bars->full[s]);
                }
            }
            goto out;
        drain:
            for (uint32_t i = (it > (uint32_t)kStreamStages ? it - kStreamStages : 0); i < it; ++i) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&bars->full[i % kStreamStages], (i / kStreamStages) & 1))
                    if (global_timer_ns() - t0 > 200000000ull) break;
            }
        out:;
        }
    } else if (warp < kStreamWarps) {
        const int grp = lane / LPK, sub = lane % LPK;
        uint32_t it = 0, nseg = 0;
        long long v = v_begin;
        Segment sg;
        while (next(v, sg)) {
            const int b = sg.b;
            const int hq0 = sg.hkv * p.group + sg.chunk * HC;
            // Query and output columns as packed fp32 pairs: the dot products
            // and the P.V updates run two columns per f32x2 instruction.
            uint64_t qf2[HC][4];
#pragma unroll
            for (int h = 0; h < HC; ++h) {
                const uint16_t* qp = p.q + (static_cast<int64_t>(b) * p.Hq + hq0 + h) * D + sub * 8;
                float qf[8];
                unpack8<kF16>(*reinterpret_cast<const uint4*>(qp), qf);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    qf2[h][e] = f2_pack(qf[2 * e] * p.scale_log2, qf[2 * e + 1] * p.scale_log2);
            }
            float m[HC], lsum[NV];
            uint64_t acc2[HC][4];
#pragma unroll
            for (int h = 0; h < HC; ++h) {
                m[h] = -INFINITY;
#pragma unroll
                for (int e = 0; e < 4; ++e) acc2[h][e] = 0ull;
            }
#pragma unroll
            for (int r = 0; r < NV; ++r) lsum[r] = 0.0f;

            for (int kc = sg.k0; kc < sg.k1; kc += CK, ++it) {
                const int n = min(CK, sg.k1 - kc);
                const int s = it % kStreamStages;
                if (!__all_sync(0xffffffffu, mbar_wait(&bars->full[s], (it / kStreamStages) & 1, g,
                                                       SITE_DEC_FULL)))
                    goto done;
                const uint8_t* ks = smem + L::kRingOff + s * kStageBytes;
                const uint8_t* vs = ks + kHalf;
                const int kb = warp * KW;
                // K rows now; V rows after the scores (fewer registers live).
                uint4 kr[kNK];
#pragma unroll
                for (int nn = 0; nn < kNK; ++nn) {
                    const int key = kb + nn * KPL + grp;
                    kr[nn] = key < n ? *reinterpret_cast<const uint4*>(ks + key * D * 2 + sub * 16)
                                     : make_uint4(0, 0, 0, 0);
                }
                float part[NV0];
#pragma unroll
                for (int nn = 0; nn < kNK; ++nn) {
                    float kf[8];
                    unpack8<kF16>(kr[nn], kf);
                    uint64_t kf2[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) kf2[e] = f2_pack(kf[2 * e], kf[2 * e + 1]);
#pragma unroll
                    for (int h = 0; h < HC; ++h) {
                        uint64_t s2 = f2_fma(qf2[h][0], kf2[0], 0ull);
#pragma unroll
                        for (int e = 1; e < 4; ++e) s2 = f2_fma(qf2[h][e], kf2[e], s2);
                        float s_lo, s_hi;
                        f2_unpack(s2, s_lo, s_hi);
                        part[nn * HC + h] = s_lo + s_hi;
                    }
                }
                group_reduce_scatter<NV0, LPK>(part, lane);
                float x[NV];
                int hown[NV];
                bool need = false;
#pragma unroll
                for (int r = 0; r < NV; ++r) {
                    const int idx = own_index<NV0, LPK>(sub, r);
                    hown[r] = idx % HC;
                    const int key = kb + (idx / HC) * KPL + grp;
                    x[r] = key < n ? part[r] : -INFINITY;
                    float mh = m[0];
#pragma unroll
                    for (int h = 1; h < HC; ++h) mh = (hown[r] == h) ? m[h] : mh;
                    need |= x[r] > mh + kRescaleThreshold;
                }
                if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                    for (int h = 0; h < HC; ++h) {
                        float cm = -INFINITY;
#pragma unroll
                        for (int r = 0; r < NV; ++r) cm = (hown[r] == h) ? fmaxf(cm, x[r]) : cm;
                        cm = warp_allmax(cm);
                        const float mnew = fmaxf(m[h], cm);
                        const float alpha = (m[h] == -INFINITY) ? 0.0f : ex2_approx(m[h] - mnew);
                        const uint64_t alpha2 = f2_pack(alpha, alpha);
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc2[h][e] = f2_fma(acc2[h][e], alpha2, 0ull);
#pragma unroll
                        for (int r = 0; r < NV; ++r) lsum[r] = (hown[r] == h) ? lsum[r] * alpha : lsum[r];
                        m[h] = mnew;
                    }
                }
#pragma unroll
                for (int r = 0; r < NV; ++r) {
                    float mh = m[0];
#pragma unroll
                    for (int h = 1; h < HC; ++h) mh = (hown[r] == h) ? m[h] : mh;
                    const float pr = (x[r] == -INFINITY) ? 0.0f : ex2_approx(x[r] - mh);
                    lsum[r] += pr;
                    if (own_canonical<NV0, LPK>(sub)) s_p[warp][grp][own_index<NV0, LPK>(sub, r)] = pr;
                }
                __syncwarp();
#pragma unroll
                for (int nn = 0; nn < kNK; ++nn) {
                    const int key = kb + nn * KPL + grp;
                    const uint4 vr = key < n ? *reinterpret_cast<const uint4*>(vs + key * D * 2 + sub * 16)
                                             : make_uint4(0, 0, 0, 0);
                    // This key's weights for the HC heads (one key at a time: fewer
                    // registers live than all NV0 at once).
                    float pk[HC];
#pragma unroll
                    for (int h = 0; h < HC; ++h) pk[h] = s_p[warp][grp][nn * HC + h];
                    float vf[8];
                    unpack8<kF16>(vr, vf);
                    uint64_t vf2[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) vf2[e] = f2_pack(vf[2 * e], vf[2 * e + 1]);
#pragma unroll
                    for (int h = 0; h < HC; ++h) {
                        const float pw = pk[h];
                        const uint64_t pw2 = f2_pack(pw, pw);
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc2[h][e] = f2_fma(pw2, vf2[e], acc2[h][e]);
                    }
                }
                // Every value read from the stage has been used: release it.
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->empty[s]);
            }

            // Segment end: merge lane groups, then warps (block-merge rule).
            float acc[HC][8];
#pragma unroll
            for (int h = 0; h < HC; ++h)
#pragma unroll
                for (int e = 0; e < 4; ++e) f2_unpack(acc2[h][e], acc[h][2 * e], acc[h][2 * e + 1]);
#pragma unroll
            for (int mask = LPK; mask < 32; mask <<= 1) {
#pragma unroll
                for (int h = 0; h < HC; ++h)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], mask);
            }
#pragma unroll
            for (int h = 0; h < HC; ++h) {
                float t = 0.0f;
                if (own_canonical<NV0, LPK>(sub)) {
#pragma unroll
                    for (int r = 0; r < NV; ++r)
                        t += ((own_index<NV0, LPK>(sub, r) % HC) == h) ? lsum[r] : 0.0f;
                }
                const float lw = warp_allsum(t);
                if (lane == 0) {
                    s_m[warp][h] = m[h];
                    s_l[warp][h] = lw;
                }
            }
            if (lane < LPK) {
#pragma unroll
                for (int h = 0; h < HC; ++h)
#pragma unroll
                    for (int e = 0; e < 8; ++e) s_acc[warp][h][sub * 8 + e] = acc[h][e];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->seg_in);
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->seg_in, nseg & 1, g, SITE_DEC_SEG)))
                goto done;
            {
                const bool whole = sg.k0 == 0 && sg.k1 == sg.L;
                // Fragment slot: dense, by unit and slice; paged, by CTA.
                const long long slot0 =
                    kPaged ? (2LL * blockIdx.x + (nseg == 0 ? 0 : 1)) * HC
                           : (sg.u * p.nseg_max +
                              (static_cast<long long>(blockIdx.x) - (sg.u * p.Tk) / p.per_cta)) * HC;
                for (int idx = threadIdx.x; idx < HC * D; idx += kStreamWarps * 32) {
                    const int h = idx / D, d = idx % D;
                    float M = -INFINITY;
#pragma unroll
                    for (int w = 0; w < kStreamWarps; ++w) M = fmaxf(M, s_m[w][h]);
                    float Ls = 0.0f, O = 0.0f;
#pragma unroll
                    for (int w = 0; w < kStreamWarps; ++w) {
                        const float wt = (s_m[w][h] == -INFINITY) ? 0.0f : ex2_approx(s_m[w][h] - M);
                        Ls = fmaf(s_l[w][h], wt, Ls);
                        O = fmaf(s_acc[w][h][d], wt, O);
                    }
                    const float out = O / Ls;
                    const float lse2 = M + __log2f(Ls);
                    if (whole) {
                        const int64_t row = static_cast<int64_t>(b) * p.Hq + hq0 + h;
                        const uint32_t pk = Elem16<kF16>::pack(out, 0.0f);
                        p.o[row * D + d] = static_cast<uint16_t>(pk & 0xffffu);
                        if (d == 0 && p.lse != nullptr) p.lse[row] = lse2 * kLn2;
                    } else {
                        const int64_t slot = slot0 + h;
                        p.ws_o[slot * D + d] = out;
                        if (d == 0) p.ws_lse[slot] = lse2;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->seg_out);
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->seg_out, nseg & 1, g, SITE_DEC_SEG)))
                goto done;
            ++nseg;
        }
    done:;
    }
    __syncthreads();
}

// Merge the fragments of the units that slice boundaries cut; units a single
// CTA covered were written directly.  Block j takes the boundary at virtual
// key (j + 1) * per_cta and merges the unit it cuts, if that is the unit's
// first cut boundary; its hc * D threads take one (head, column) each, so
// every load is issued at once.  Launched with programmatic stream
// serialisation: it waits for the stream kernel before reading the fragments.
template <int D, bool kF16 = false>
__global__ void __launch_bounds__(1024)
decode_stream_combine_kernel(const StreamParams p, int hc) {
    grid_dependency_wait();
    const int d = threadIdx.x % D, h = threadIdx.x / D;
    const long long pos = (blockIdx.x + 1LL) * p.per_cta;
    if (pos >= p.total) return;
    const long long u = pos / p.Tk;
    const long long start = u * p.Tk;
    if (start == pos || start < pos - p.per_cta) return;  // not cut here, or cut earlier
    const long long c0 = start / p.per_cta;
    const long long c1 = (start + p.Tk - 1) / p.per_cta;
    const int nseg = static_cast<int>(c1 - c0 + 1);
    const long long pair = u / p.chunks;
    const int chunk = static_cast<int>(u - pair * p.chunks);
    const int b = static_cast<int>(pair / p.Hkv), hkv = static_cast<int>(pair % p.Hkv);
    float M = -INFINITY;
    for (int s = 0; s < nseg; ++s) M = fmaxf(M, p.ws_lse[(u * p.nseg_max + s) * hc + h]);
    float Ls = 0.0f, acc = 0.0f;
    for (int s = 0; s < nseg; ++s) {
        const int64_t slot = (u * p.nseg_max + s) * hc + h;
        const float w = ex2_approx(p.ws_lse[slot] - M);
        Ls += w;
        acc = fmaf(w, p.ws_o[slot * D + d], acc);
    }
    const int64_t row = static_cast<int64_t>(b) * p.Hq + hkv * p.group + chunk * hc + h;
    const uint32_t pk = Elem16<kF16>::pack(acc / Ls, 0.0f);
    p.o[row * D + d] = static_cast<uint16_t>(pk & 0xffffu);
    if (d == 0 && p.lse != nullptr) p.lse[row] = (M + __log2f(Ls)) * kLn2;
}

// Paged mode: prefix of the clamped request lengths and the slice geometry
// (one block).  A length outside 0 .. max_pages * page is reported in the
// status word and clamped into that range.
__global__ void __launch_bounds__(1024)
paged_prefix_kernel(const int32_t* seq_lens, int B, int max_keys, long long units_per_req,
                    int grid, long long* cum, long long* geom, unsigned* status) {
    __shared__ long long warp_tot[32];
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (B + nt - 1) / nt;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    long long mine = 0;
    for (int b = b0; b < b1; ++b) {
        int L = seq_lens[b];
        if (L < 0 || L > max_keys) {
            atomicOr(status, ATTN_DEV_BAD_INPUT);
            L = L < 0 ? 0 : max_keys;
        }
        mine += L;
    }
    // Exclusive scan of the per-thread sums: within warps, then across warps.
    const int lane = tid & 31, warp = tid >> 5;
    long long incl = mine;
    for (int o = 1; o < 32; o <<= 1) {
        const long long t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        long long w = lane < nt / 32 ? warp_tot[lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            const long long t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    long long run = incl - mine + (warp > 0 ? warp_tot[warp - 1] : 0);
    for (int b = b0; b < b1; ++b) {
        cum[b] = run;
        int L = seq_lens[b];
        L = L < 0 ? 0 : (L > max_keys ? max_keys : L);
        run += L;
    }
    if (tid == nt - 1) {
        cum[B] = run;  // the last thread's range ends at B (or is empty and run is the total)
        const long long total = run * units_per_req;
        geom[0] = total;
        geom[1] = total > 0 ? (total + grid - 1) / grid : 1;
    }
}

// Paged mode: merge the fragments of cut units (CTA slots; requests without
// keys were written by the stream kernel).  Block j takes the boundary at
// virtual key (j + 1) * per_cta, which CTA j + 1's slice starts at; that CTA
// recorded the unit its slice starts in.  Threads and launch as in the dense
// combine.
template <int D, bool kF16 = false>
__global__ void __launch_bounds__(1024)
decode_paged_combine_kernel(const StreamParams p, int hc) {
    grid_dependency_wait();
    const int d = threadIdx.x % D, h = threadIdx.x / D;
    const long long total = p.pg.geom[0], per = p.pg.geom[1];
    const long long pos = (blockIdx.x + 1LL) * per;
    if (pos >= total) return;
    const int4 fu = p.pg.first_unit[blockIdx.x + 1];  // {b, unit in request, offset, length}
    const long long k0 = fu.z, L = fu.w;
    if (k0 == 0 || k0 > per) return;  // not cut here, or cut at an earlier boundary
    const long long start = pos - k0;
    const int hkv = fu.y / p.chunks;
    const int chunk = fu.y - hkv * p.chunks;
    const long long c0 = start / per, c1 = (start + L - 1) / per;
    const int first = start != c0 * per ? 1 : 0;  // CTA c0 holds the unit in its last slot
    float M = -INFINITY;
    for (long long c = c0; c <= c1; ++c)
        M = fmaxf(M, p.ws_lse[(2 * c + (c == c0 ? first : 0)) * hc + h]);
    float Ls = 0.0f, acc = 0.0f;
    for (long long c = c0; c <= c1; ++c) {
        const long long slot = (2 * c + (c == c0 ? first : 0)) * hc + h;
        const float wt = ex2_approx(p.ws_lse[slot] - M);
        Ls += wt;
        acc = fmaf(wt, p.ws_o[slot * D + d], acc);
    }
    const int64_t row = static_cast<int64_t>(fu.x) * p.Hq + hkv * p.group + chunk * hc + h;
    const uint32_t pk = Elem16<kF16>::pack(acc / Ls, 0.0f);
    p.o[row * D + d] = static_cast<uint16_t>(pk & 0xffffu);
    if (d == 0 && p.lse != nullptr) p.lse[row] = (M + __log2f(Ls)) * kLn2;
}

// Launches a combine kernel (grid = slice boundaries) with programmatic
// stream serialisation, so that it is scheduled while the stream kernel
// before it runs.
cudaError_t launch_combine_after_stream(void (*kern)(const StreamParams, int), int blocks,
                                        int threads, const StreamParams& p, int hc,
                                        cudaStream_t st) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, hc);
}

template <int D, int HC, bool kPaged = false, bool kF16 = false>
cudaError_t launch_stream(const StreamParams& p, int grid, cudaStream_t st) {
    using L = StreamLayout<D, HC, kPaged>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(decode_stream_kernel<D, HC, kPaged, kF16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    decode_stream_kernel<D, HC, kPaged, kF16><<<grid, kStreamThreads, L::kBytes, st>>>(p);
    return cudaGetLastError();
}

template <int D, bool kPaged = false, bool kF16 = false>
cudaError_t launch_stream_d(const StreamParams& p, int hc, int grid, cudaStream_t st) {
    switch (hc) {
        case 8: return launch_stream<D, 8, kPaged, kF16>(p, grid, st);
        case 4: return launch_stream<D, 4, kPaged, kF16>(p, grid, st);
        case 2: return launch_stream<D, 2, kPaged, kF16>(p, grid, st);
        default: return launch_stream<D, 1, kPaged, kF16>(p, grid, st);
    }
}

// Slice geometry shared by the workspace size and the launch.
struct StreamGeom {
    long long total, per_cta;
    int grid, nseg_max, hc, chunks;
};

StreamGeom stream_geom(const Shape& s, int num_sms) {
    StreamGeom g;
    const int group = s.Hq / s.Hkv;
    g.hc = heads_per_cta(group);
    g.chunks = group / g.hc;
    g.total = static_cast<long long>(s.B) * s.Hkv * g.chunks * s.Tk;
    g.per_cta = (g.total + num_sms - 1) / num_sms;
    g.grid = static_cast<int>((g.total + g.per_cta - 1) / g.per_cta);
    g.nseg_max = static_cast<int>((s.Tk + g.per_cta - 1) / g.per_cta) + 1;
    return g;
}

}  // namespace

size_t decode_stream_workspace_bytes(const Shape& s, int num_sms) {
    const StreamGeom g = stream_geom(s, num_sms);
    const size_t slots = static_cast<size_t>(s.B) * s.Hq * g.nseg_max;
    return slots * s.D * sizeof(float) + slots * sizeof(float) + 256;
}

// Paged workspace: cum [B + 1] and geom [2] (int64), first_unit [grid] (int4),
// then the fragment slots' outputs [2 * grid * hc, D] and lse values.
struct PagedWsLayout {
    size_t geom, first_unit, ws_o, ws_lse, bytes;
    PagedWsLayout(const PagedShape& s, int grid) {
        const size_t frag = 2ull * grid * heads_per_cta(s.Hq / s.Hkv);
        auto up16 = [](size_t x) { return (x + 15) / 16 * 16; };
        geom = 8ull * (s.B + 1);
        first_unit = up16(geom + 16);
        ws_o = up16(first_unit + 16ull * grid);
        ws_lse = ws_o + frag * s.D * sizeof(float);
        bytes = ws_lse + frag * sizeof(float) + 256;
    }
};

size_t decode_paged_workspace_bytes(const PagedShape& s, int num_sms) {
    return PagedWsLayout(s, num_sms).bytes;
}

cudaError_t launch_decode_paged_bf16(const uint16_t* q, const uint16_t* kv,
                                     const int32_t* block_table, const int32_t* seq_lens,
                                     uint16_t* o, float* lse, void* ws, const PagedShape& s,
                                     const LaunchEnv& env, int* grid_out, int* kernels_launched) {
    const int group = s.Hq / s.Hkv;
    const int hc = heads_per_cta(group);
    const int grid = env.num_sms;
    const PagedWsLayout lay(s, grid);
    uint8_t* base = static_cast<uint8_t*>(ws);
    long long* cum = reinterpret_cast<long long*>(base);
    long long* geom = reinterpret_cast<long long*>(base + lay.geom);
    float* ws_o = reinterpret_cast<float*>(base + lay.ws_o);
    float* ws_lse = reinterpret_cast<float*>(base + lay.ws_lse);

    StreamParams p{};
    p.q = q; p.k = nullptr; p.v = nullptr; p.o = o; p.lse = lse;
    p.ws_o = ws_o; p.ws_lse = ws_lse;
    p.Hq = s.Hq; p.Hkv = s.Hkv; p.Tk = 0; p.group = group; p.chunks = group / hc;
    p.nseg_max = 0; p.total = 0; p.per_cta = 0;
    p.scale_log2 = s.scale * 1.4426950408889634f;
    p.status = env.status;
    p.limit_ns = env.wait_limit_ns;
    p.pg.kv = kv; p.pg.block_table = block_table; p.pg.seq_lens = seq_lens;
    p.pg.cum = cum; p.pg.geom = geom;
    p.pg.first_unit = reinterpret_cast<int4*>(base + lay.first_unit);
    p.pg.B = s.B; p.pg.page = s.page; p.pg.max_pages = s.max_pages; p.pg.num_blocks = s.num_blocks;
    p.pg.in_kernel = s.B <= kMaxPrefixB ? 1 : 0;

    int launched = 2;
    cudaError_t e = cudaSuccess;
    if (!p.pg.in_kernel) {
        const long long units_per_req = static_cast<long long>(s.Hkv) * p.chunks;
        paged_prefix_kernel<<<1, 1024, 0, env.stream>>>(seq_lens, s.B, s.max_pages * s.page,
                                                        units_per_req, grid, cum, geom, env.status);
        e = cudaGetLastError();
        launched = 3;
    }
    if (e == cudaSuccess) {
        if (s.f16)
            e = (s.D == 64) ? launch_stream_d<64, true, true>(p, hc, grid, env.stream)
                            : launch_stream_d<128, true, true>(p, hc, grid, env.stream);
        else
            e = (s.D == 64) ? launch_stream_d<64, true>(p, hc, grid, env.stream)
                            : launch_stream_d<128, true>(p, hc, grid, env.stream);
    }
    if (e == cudaSuccess && grid > 1) {
        auto kern = s.f16 ? (s.D == 64 ? decode_paged_combine_kernel<64, true>
                                       : decode_paged_combine_kernel<128, true>)
                          : (s.D == 64 ? decode_paged_combine_kernel<64>
                                       : decode_paged_combine_kernel<128>);
        e = launch_combine_after_stream(kern, grid - 1, s.D * hc, p, hc, env.stream);
    } else {
        --launched;
    }
    if (grid_out) *grid_out = grid;
    if (kernels_launched) *kernels_launched = launched;
    return e;
}

cudaError_t launch_decode_stream_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                      uint16_t* o, float* lse, float* ws, const Shape& s,
                                      const LaunchEnv& env, int* grid_out, int* kernels_launched) {
    const StreamGeom g = stream_geom(s, env.num_sms);
    StreamParams p;
    p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
    const size_t slots = static_cast<size_t>(s.B) * s.Hq * g.nseg_max;
    p.ws_o = ws;
    p.ws_lse = ws + slots * s.D;
    p.Hq = s.Hq; p.Hkv = s.Hkv; p.Tk = s.Tk; p.group = s.Hq / s.Hkv; p.chunks = g.chunks;
    p.nseg_max = g.nseg_max;
    p.total = g.total;
    p.per_cta = g.per_cta;
    p.scale_log2 = s.scale * 1.4426950408889634f;
    p.status = env.status;
    p.limit_ns = env.wait_limit_ns;
    cudaError_t e;
    if (s.f16)
        e = (s.D == 64) ? launch_stream_d<64, false, true>(p, g.hc, g.grid, env.stream)
                        : launch_stream_d<128, false, true>(p, g.hc, g.grid, env.stream);
    else
        e = (s.D == 64) ? launch_stream_d<64>(p, g.hc, g.grid, env.stream)
                        : launch_stream_d<128>(p, g.hc, g.grid, env.stream);
    int launched = 1;
    if (e == cudaSuccess && g.grid > 1) {
        auto kern = s.f16 ? (s.D == 64 ? decode_stream_combine_kernel<64, true>
                                       : decode_stream_combine_kernel<128, true>)
                          : (s.D == 64 ? decode_stream_combine_kernel<64>
                                       : decode_stream_combine_kernel<128>);
        e = launch_combine_after_stream(kern, g.grid - 1, s.D * g.hc, p, g.hc, env.stream);
        launched = 2;
    }
    if (grid_out) *grid_out = g.grid;
    if (kernels_launched) *kernels_launched = launched;
    return e;
}

}  // namespace attn
