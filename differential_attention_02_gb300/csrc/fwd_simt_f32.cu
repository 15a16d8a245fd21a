// fp32 prefill of differential attention on the CUDA cores (FFMA), for fp32
// inputs where tensor-core precision would not meet an fp32 tolerance.
//
// Computes, per head and query row i, the DiffAttn formula of "Differential
// Transformer: Transformer que cancela ruído de atenção" (section "Como a
// atenção diferencial funciona"): (softmax(Q1K1^T/sqrt d) - lambda
// softmax(Q2K2^T/sqrt d)) V with the causal mask of the intoai.pub page
// ("A Deeper Dive Into Attention Calculations"), then the per-head RMSNorm and
// (1 - lambda_init) scale ("Estrutura multi-head e arquitetura completa").
//
// Layout: one warp per query row, kRows rows per CTA. Keys stream through
// shared memory 32 at a time; lane l scores key (chunk + l) for both maps,
// each map keeps its own online-softmax state (running max, running sum), and
// lane l accumulates value columns l, l+32, ... of both maps' outputs.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

constexpr int kRows = 8;      // query rows (warps) per CTA
constexpr int kChunk = 32;    // keys per shared-memory chunk
constexpr int kMaxD = 128;
constexpr int kMaxDv = 256;

template <int DVL>  // value columns per lane = Dv / 32
__global__ void __launch_bounds__(kRows * 32) fwd_simt_f32_kernel(const SimtF32Params p) {
    extern __shared__ float smem[];
    const int d = p.d, Dv = p.Dv;
    const int dp = d + 1;  // padded key row: lane-strided reads hit distinct banks
    float* q1s = smem;                  // [kRows][d]
    float* q2s = q1s + kRows * d;       // [kRows][d]
    float* k1s = q2s + kRows * d;       // [kChunk][d+1]
    float* k2s = k1s + kChunk * dp;     // [kChunk][d+1]
    float* vs = k2s + kChunk * dp;      // [kChunk][Dv]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, h = blockIdx.y;
    const int row0 = blockIdx.x * kRows;
    const int i = row0 + warp;

    const float* q1 = p.q1 + b * p.sq1[0] + h * p.sq1[1];
    const float* q2 = p.q2 + b * p.sq2[0] + h * p.sq2[1];
    const float* k1 = p.k1 + b * p.sk1[0] + h * p.sk1[1];
    const float* k2 = p.k2 + b * p.sk2[0] + h * p.sk2[1];
    const float* v = p.v + b * p.sv[0] + h * p.sv[1];

    for (int t = threadIdx.x; t < kRows * d; t += blockDim.x) {
        const int r = t / d, c = t % d;
        const bool ok = row0 + r < p.N;
        q1s[t] = ok ? q1[(int64_t)(row0 + r) * p.sq1[2] + c] : 0.f;
        q2s[t] = ok ? q2[(int64_t)(row0 + r) * p.sq2[2] + c] : 0.f;
    }

    const float scale = 1.0f / sqrtf((float)d);
    float m1 = -INFINITY, m2 = -INFINITY, l1 = 0.f, l2 = 0.f;
    float o1[DVL], o2[DVL];
#pragma unroll
    for (int t = 0; t < DVL; ++t) o1[t] = o2[t] = 0.f;

    // Keys any row of this CTA may see.
    const int kend = p.causal ? min(p.N, row0 + kRows) : p.N;
    for (int c0 = 0; c0 < kend; c0 += kChunk) {
        __syncthreads();
        for (int t = threadIdx.x; t < kChunk * d; t += blockDim.x) {
            const int r = t / d, c = t % d;
            const bool ok = c0 + r < p.N;
            k1s[r * dp + c] = ok ? k1[(int64_t)(c0 + r) * p.sk1[2] + c] : 0.f;
            k2s[r * dp + c] = ok ? k2[(int64_t)(c0 + r) * p.sk2[2] + c] : 0.f;
        }
        for (int t = threadIdx.x; t < kChunk * Dv; t += blockDim.x) {
            const int r = t / Dv, c = t % Dv;
            vs[t] = (c0 + r < p.N) ? v[(int64_t)(c0 + r) * p.sv[2] + c] : 0.f;
        }
        __syncthreads();
        if (i >= p.N) continue;

        const int j = c0 + lane;
        const bool visible = (j < p.N) && (!p.causal || j <= i);
        float s1 = 0.f, s2 = 0.f;
        for (int c = 0; c < d; ++c) {
            s1 = fmaf(q1s[warp * d + c], k1s[lane * dp + c], s1);
            s2 = fmaf(q2s[warp * d + c], k2s[lane * dp + c], s2);
        }
        s1 = visible ? s1 * scale : -INFINITY;
        s2 = visible ? s2 * scale : -INFINITY;

        const float n1 = fmaxf(m1, warp_max(s1));
        const float n2 = fmaxf(m2, warp_max(s2));
        if (n1 == -INFINITY) continue;  // no visible key yet (cannot happen for causal rows)
        const float a1 = expf(m1 - n1), a2 = expf(m2 - n2);
        const float p1 = visible ? expf(s1 - n1) : 0.f;
        const float p2 = visible ? expf(s2 - n2) : 0.f;
        l1 = l1 * a1 + warp_sum(p1);
        l2 = l2 * a2 + warp_sum(p2);
        m1 = n1;
        m2 = n2;
#pragma unroll
        for (int t = 0; t < DVL; ++t) {
            o1[t] *= a1;
            o2[t] *= a2;
        }
        const int nk = min(kChunk, kend - c0);
        for (int jj = 0; jj < nk; ++jj) {
            const float w1 = __shfl_sync(0xffffffffu, p1, jj);
            const float w2 = __shfl_sync(0xffffffffu, p2, jj);
#pragma unroll
            for (int t = 0; t < DVL; ++t) {
                const float vv = vs[jj * Dv + lane + 32 * t];
                o1[t] = fmaf(w1, vv, o1[t]);
                o2[t] = fmaf(w2, vv, o2[t]);
            }
        }
    }
    if (i >= p.N) return;

    // Combine the maps, then RMSNorm over the Dv channels and the (1 - lambda_init) scale.
    float oh[DVL], ss = 0.f;
#pragma unroll
    for (int t = 0; t < DVL; ++t) {
        oh[t] = o1[t] / l1 - p.lambda * (o2[t] / l2);
        ss = fmaf(oh[t], oh[t], ss);
    }
    ss = warp_sum(ss);
    const float r = (1.0f - p.lambda_init) / sqrtf(ss / (float)Dv + p.eps);
    const int64_t obase = (((int64_t)b * p.N + i) * p.H + h) * Dv;
#pragma unroll
    for (int t = 0; t < DVL; ++t) {
        const int c = lane + 32 * t;
        float y = oh[t] * r;
        if (p.norm_w) y *= p.norm_w[c];
        if (p.out_bf16)
            reinterpret_cast<__nv_bfloat16*>(p.out)[obase + c] = __float2bfloat16_rn(y);
        else
            reinterpret_cast<float*>(p.out)[obase + c] = y;
    }
}

template <int DVL>
cudaError_t launch_dvl(const SimtF32Params& p, cudaStream_t stream) {
    const size_t smem = sizeof(float) * (size_t)(2 * kRows * p.d + 2 * kChunk * (p.d + 1) + kChunk * p.Dv);
    auto k = fwd_simt_f32_kernel<DVL>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.N + kRows - 1) / kRows, p.H, p.B);
    k<<<grid, kRows * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt_f32(const SimtF32Params& p, cudaStream_t stream) {
    if (p.d > kMaxD || p.Dv > kMaxDv) return cudaErrorInvalidValue;
    switch (p.Dv / 32) {
        case 1: return launch_dvl<1>(p, stream);
        case 2: return launch_dvl<2>(p, stream);
        case 3: return launch_dvl<3>(p, stream);
        case 4: return launch_dvl<4>(p, stream);
        case 5: return launch_dvl<5>(p, stream);
        case 6: return launch_dvl<6>(p, stream);
        case 7: return launch_dvl<7>(p, stream);
        case 8: return launch_dvl<8>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace da
