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

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    f[0] = bf16_lo_to_f32(u.x); f[1] = bf16_hi_to_f32(u.x);
    f[2] = bf16_lo_to_f32(u.y); f[3] = bf16_hi_to_f32(u.y);
    f[4] = bf16_lo_to_f32(u.z); f[5] = bf16_hi_to_f32(u.z);
    f[6] = bf16_lo_to_f32(u.w); f[7] = bf16_hi_to_f32(u.w);
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
template <int D>
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
    const uint32_t pk = pack_bf16x2(acc / L, 0.0f);
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

}  // namespace attn
