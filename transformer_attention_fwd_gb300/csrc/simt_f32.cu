// simt_f32.cu -- float32 attention forward on the CUDA cores.
//
// fp32 I/O must agree with a float64 evaluation to 1e-5, which rules out the
// tensor cores (tf32 carries ~1e-3 relative error); the fp32 workloads are
// also tiny (latency bound), so this kernel favours clarity: one CTA takes 16
// query rows of one (b, hq), stages 32-key tiles of K and V in shared memory
// and keeps a running row maximum, row sum and output accumulator
// ("3.3 Self-Attention机制深入理解" §7.3 online softmax, §12.2 tiling, §12.3
// rescaling of the partial output).  Exponentials use expf (natural base) for
// accuracy.
#include <cuda_runtime.h>
#include <cmath>
#include <cstdint>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRows = kWarps * kRowsPerWarp;  // 16 query rows per CTA
constexpr int kKeys = 32;                      // keys per shared-memory tile

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, m));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
simt_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                const float* __restrict__ v, float* __restrict__ o, float* __restrict__ lse,
                int Hq, int Hkv, int Tq, int Tk, int causal, float scale) {
    constexpr int DPL = D / 32;  // output columns per lane
    __shared__ float sQ[kRows][D];
    __shared__ float sK[kKeys][D + 1];
    __shared__ float sV[kKeys][D];

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int bh = blockIdx.x;
    const int b = bh / Hq, hq = bh % Hq;
    const int hkv = hq / (Hq / Hkv);
    const int row0 = blockIdx.y * kRows;
    const float* qh = q + static_cast<int64_t>(bh) * Tq * D;
    const float* kh = k + (static_cast<int64_t>(b) * Hkv + hkv) * Tk * D;
    const float* vh = v + (static_cast<int64_t>(b) * Hkv + hkv) * Tk * D;
    const int off = Tk - Tq;  // causal alignment: row i sees keys j <= i + off

    for (int idx = tid; idx < kRows * D; idx += blockDim.x) {
        const int r = idx / D, d = idx % D;
        sQ[r][d] = (row0 + r < Tq) ? qh[static_cast<int64_t>(row0 + r) * D + d] : 0.0f;
    }

    const int last_row = min(row0 + kRows - 1, Tq - 1);
    const int kend = causal ? min(Tk, last_row + off + 1) : Tk;

    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][DPL];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.0f;
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[r][i] = 0.0f;
    }

    for (int kt = 0; kt < kend; kt += kKeys) {
        __syncthreads();
        for (int idx = tid; idx < kKeys * D; idx += blockDim.x) {
            const int j = idx / D, d = idx % D;
            const bool in = kt + j < Tk;
            sK[j][d] = in ? kh[static_cast<int64_t>(kt + j) * D + d] : 0.0f;
            sV[j][d] = in ? vh[static_cast<int64_t>(kt + j) * D + d] : 0.0f;
        }
        __syncthreads();

        const int kj = kt + lane;  // this lane's key
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int lr = warp * kRowsPerWarp + r;
            const int row = row0 + lr;
            const bool vis = kj < Tk && (!causal || kj <= row + off);
            float s = 0.0f;
#pragma unroll 16
            for (int d = 0; d < D; ++d) s = fmaf(sQ[lr][d], sK[lane][d], s);
            s = vis ? s * scale : -INFINITY;
            const float m_new = fmaxf(m[r], warp_max(s));
            if (m_new == -INFINITY) continue;  // nothing visible yet (warp-uniform)
            const float alpha = (m[r] == -INFINITY) ? 0.0f : expf(m[r] - m_new);
            const float p = vis ? expf(s - m_new) : 0.0f;
            l[r] = l[r] * alpha + warp_sum(p);
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[r][i] *= alpha;
#pragma unroll 8
            for (int j = 0; j < kKeys; ++j) {
                const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
                for (int i = 0; i < DPL; ++i) acc[r][i] = fmaf(pj, sV[j][lane + 32 * i], acc[r][i]);
            }
            m[r] = m_new;
        }
    }

#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int row = row0 + warp * kRowsPerWarp + r;
        if (row >= Tq) continue;
        const float inv = 1.0f / l[r];
        float* orow = o + (static_cast<int64_t>(bh) * Tq + row) * D;
#pragma unroll
        for (int i = 0; i < DPL; ++i) orow[lane + 32 * i] = acc[r][i] * inv;
        if (lse != nullptr && lane == 0) lse[static_cast<int64_t>(bh) * Tq + row] = m[r] + logf(l[r]);
    }
}

}  // namespace

cudaError_t launch_simt_f32(const float* q, const float* k, const float* v, float* o,
                            float* lse, const Shape& s, const LaunchEnv& env,
                            int* kernels_launched) {
    const int row_blocks = (s.Tq + kRows - 1) / kRows;
    if (row_blocks > 65535) return cudaErrorInvalidConfiguration;
    dim3 grid(s.B * s.Hq, row_blocks);
    dim3 block(kWarps * 32);
    if (s.D == 64)
        simt_f32_kernel<64><<<grid, block, 0, env.stream>>>(q, k, v, o, lse, s.Hq, s.Hkv, s.Tq,
                                                            s.Tk, s.causal, s.scale);
    else
        simt_f32_kernel<128><<<grid, block, 0, env.stream>>>(q, k, v, o, lse, s.Hq, s.Hkv, s.Tq,
                                                             s.Tk, s.causal, s.scale);
    if (kernels_launched) *kernels_launched = 1;
    return cudaGetLastError();
}

}  // namespace attn
