// Elementwise pieces of the DIFF Transformer layer around the attention module
// ("A Simple Principle From Noise-Cancelling Headphones Supercharges
// Transformers Like Never Before" (intoai.pub), section "The Overall
// Architecture Of The Multi-Head Differential Transformer"; "Differential
// Transformer: Transformer que cancela ruído de atenção", section "Estrutura
// multi-head e arquitetura completa"): each of the layer's two blocks is
// pre-normalised with RMSNorm and added back to its input, and the
// feed-forward block uses the SwiGLU activation.
//
// add_rmsnorm: y = x + z (z optional) and n = y / sqrt(mean(y^2) + eps) * g over
//   each row; y is written in fp32 when asked for (the residual stream), n in
//   bf16 or fp16 (the next GEMM's operand). One CTA per row; HBM-bound.
// swiglu: h = SiLU(g) * u for the two halves [g | u] of the gate/up GEMM's
//   fp16 output rows, written in bf16 or fp16. HBM-bound.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

constexpr int kNormThreads = 256;

// Eight consecutive elements of y = x + z.
__device__ __forceinline__ void load_y8(const AddNormParams& p, int64_t off, float* v) {
    if (p.x_f32) {
        const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(p.x) + off);
        const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(p.x) + off + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        const uint4 a = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.x) + off);
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = bf16lo_to_f32(w[i]);
            v[2 * i + 1] = bf16hi_to_f32(w[i]);
        }
    }
    if (p.z) {
        const float4 a = *reinterpret_cast<const float4*>(p.z + off);
        const float4 b = *reinterpret_cast<const float4*>(p.z + off + 4);
        v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w; v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
    }
}

__global__ void __launch_bounds__(kNormThreads) add_rmsnorm_kernel(const __grid_constant__ AddNormParams p) {
    pdl_trigger();
    pdl_wait();  // y and z may be the previous kernel's output
    __shared__ float red[kNormThreads / 32];
    const int64_t base = (int64_t)blockIdx.x * p.N;
    const int n8 = p.N / 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float ss = 0.f;
    for (int c = threadIdx.x; c < n8; c += kNormThreads) {
        float v[8];
        load_y8(p, base + c * 8, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(v[e], v[e], ss);
        if (p.y_out) {
            *reinterpret_cast<float4*>(p.y_out + base + c * 8) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4*>(p.y_out + base + c * 8 + 4) = make_float4(v[4], v[5], v[6], v[7]);
        }
    }
    if (p.n_out == nullptr) return;  // the same for every thread of the CTA
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < kNormThreads / 32; ++i) tot += red[i];
    const float rs = 1.0f / sqrtf(tot / (float)p.N + p.eps);
    for (int c = threadIdx.x; c < n8; c += kNormThreads) {
        float v[8];
        load_y8(p, base + c * 8, v);
        if (p.weight) {
            const float4 a = *reinterpret_cast<const float4*>(p.weight + c * 8);
            const float4 b = *reinterpret_cast<const float4*>(p.weight + c * 8 + 4);
            v[0] *= a.x; v[1] *= a.y; v[2] *= a.z; v[3] *= a.w; v[4] *= b.x; v[5] *= b.y; v[6] *= b.z; v[7] *= b.w;
        }
        const bool f16 = p.n_f16 != 0;
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.n_out) + base + c * 8) =
            make_uint4(pack_16x2(v[0] * rs, v[1] * rs, f16), pack_16x2(v[2] * rs, v[3] * rs, f16),
                       pack_16x2(v[4] * rs, v[5] * rs, f16), pack_16x2(v[6] * rs, v[7] * rs, f16));
    }
}

__device__ __forceinline__ float silu(float t) { return t / (1.0f + expf(-t)); }

__global__ void swiglu_kernel(const __half* __restrict__ gu, uint16_t* __restrict__ h, int h_f16, int64_t M, int H) {
    const int h8 = H / 8;
    const int64_t total = M * h8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / h8;
        const int c = (int)(i % h8);
        const uint4 gv = *reinterpret_cast<const uint4*>(gu + m * 2 * H + c * 8);
        const uint4 uv = *reinterpret_cast<const uint4*>(gu + m * 2 * H + H + c * 8);
        const __half2* g2 = reinterpret_cast<const __half2*>(&gv);
        const __half2* u2 = reinterpret_cast<const __half2*>(&uv);
        uint32_t out[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 g = __half22float2(g2[k]);
            const float2 u = __half22float2(u2[k]);
            out[k] = pack_16x2(silu(g.x) * u.x, silu(g.y) * u.y, h_f16 != 0);
        }
        *reinterpret_cast<uint4*>(h + m * H + c * 8) = make_uint4(out[0], out[1], out[2], out[3]);
    }
}

}  // namespace

cudaError_t launch_add_rmsnorm(const AddNormParams& p, cudaStream_t stream) {
    return launch_pdl(add_rmsnorm_kernel, dim3(p.M), dim3(kNormThreads), 0, stream, p);
}

cudaError_t launch_swiglu(const void* gate_up, void* h, int h_f16, int64_t M, int H, cudaStream_t stream) {
    int sms = 0;
    cudaError_t e = device_sm_count(&sms);
    if (e != cudaSuccess) return e;
    const int64_t total = M * (H / 8);
    const int64_t want = (total + 255) / 256;
    const int grid = (int)(want < (int64_t)sms * 16 ? want : (int64_t)sms * 16);
    swiglu_kernel<<<grid, 256, 0, stream>>>(static_cast<const __half*>(gate_up), static_cast<uint16_t*>(h), h_f16, M,
                                            H);
    return cudaGetLastError();
}

}  // namespace da
