// Backward pass of differential attention on the CUDA cores (fp32 arithmetic).
//
// The forward is, per head ("Differential Transformer: Transformer que cancela
// ruído de atenção", sections "Como a atenção diferencial funciona" and
// "Estrutura multi-head e arquitetura completa"; causal mask from "A Simple
// Principle From Noise-Cancelling Headphones...", "A Deeper Dive Into Attention
// Calculations"):
//   P_m = softmax(Q_m K_m^T / sqrt(d) + M),  A = P1 - lambda P2,  O = A V,
//   y = O / sqrt(mean(O^2) + eps) * w * (1 - lambda_init).
// The pages train the model but print no gradient; these kernels take the chain
// rule of that definition. With n = O / r, c = 1 - lambda_init and dy given:
//   dO = (g - n mean(g n)) / r, g = dy w c;       dw = sum_rows dy n c
//   dV = A^T dO;  dA = dO V^T;                      dlambda = -sum(dA P2)
//   dS1 = P1 (dA - D1), D1_i = dO_i . (P1 V)_i;     dS2 = P2 (-lambda dA - D2),
//   D2_i = -lambda dO_i . (P2 V)_i;  dQ_m = dS_m K_m / sqrt d;  dK_m = dS_m^T Q_m / sqrt d.
//
// Four launches, no atomics (results do not depend on scheduling):
//   rows   one warp per query row: recomputes both maps' softmax states and
//          outputs (as the fp32 forward does), then writes dO, the two
//          log-sum-exps and D1, D2 to the workspace, and per-CTA partial sums
//          of dlambda and dw;
//   kv     one warp per key row: streams the query rows it is visible to,
//          rebuilds P1, P2 from the log-sum-exps, and accumulates dV, dK1, dK2;
//   q      one warp per query row: streams its visible keys and accumulates
//          dQ1, dQ2;
//   reduce sums the partials of dlambda and dw in a fixed order.
// Lane l owns columns l, l + 32, ... of every row it accumulates; rows stream
// through shared memory 32 at a time, one warp per row, with a row stride of
// width + 4 floats: a lane reads its own row 16 bytes at a time and the eight
// lanes of a quarter-warp land on distinct banks. Dot products run in two
// independent FMA chains, in the same element order in every kernel, so the
// scores the key- and query-side passes rebuild equal the row pass's bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

constexpr int kRows = 8;    // rows (warps) per CTA
constexpr int kChunk = 32;  // streamed rows per shared-memory chunk
constexpr int kDL = 4;      // max d / 32
constexpr int kDVL = 8;     // max Dv / 32
constexpr int kThreads = kRows * 32;

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float ldf(const __half* p) { return __half2float(*p); }

// Row n of operand (b, h) with strides s = {b, h, n}, element c.
template <typename T>
__device__ __forceinline__ float ld_op(const void* base, const int64_t* s, int b, int h, int n, int c) {
    return ldf(static_cast<const T*>(base) + b * s[0] + h * s[1] + (int64_t)n * s[2] + c);
}

__device__ __forceinline__ int64_t row_index(const BwdParams& p, int b, int h, int i) {
    return ((int64_t)b * p.H + h) * p.N + i;
}

// Rows r0 .. r0 + rows - 1 of operand (b, h) into dst (row stride ld floats): warp w
// copies rows w, w + kRows, ..., lanes stride the columns. Rows at or past N read 0.
template <typename T>
__device__ __forceinline__ void stage_rows(float* dst, int ld, const void* src, const int64_t* s, int b, int h,
                                           int r0, int rows, int width, int N, int warp, int lane) {
    for (int r = warp; r < rows; r += kRows) {
        const bool ok = r0 + r < N;
        for (int c = lane; c < width; c += 32) dst[r * ld + c] = ok ? ld_op<T>(src, s, b, h, r0 + r, c) : 0.f;
    }
}

// The same from a workspace array of per-row records of `width` floats.
__device__ __forceinline__ void stage_ws_rows(float* dst, int ld, const float* src, const BwdParams& p, int b,
                                              int h, int r0, int rows, int width, int warp, int lane) {
    for (int r = warp; r < rows; r += kRows) {
        const bool ok = r0 + r < p.N;
        const float* row = src + (ok ? row_index(p, b, h, r0 + r) : 0) * width;
        for (int c = lane; c < width; c += 32) dst[r * ld + c] = ok ? row[c] : 0.f;
    }
}

// sum_c a[c] b[c] over n floats (n a multiple of 4, both 16-byte aligned), two chains.
__device__ __forceinline__ float dot4(const float* a, const float* b, int n) {
    const float4* a4 = reinterpret_cast<const float4*>(a);
    const float4* b4 = reinterpret_cast<const float4*>(b);
    float x = 0.f, y = 0.f;
    for (int i = 0; i < n / 4; ++i) {
        const float4 u = a4[i], v = b4[i];
        x = fmaf(u.x, v.x, x);
        y = fmaf(u.y, v.y, y);
        x = fmaf(u.z, v.z, x);
        y = fmaf(u.w, v.w, y);
    }
    return x + y;
}

// ------------------------------------------------------------------ rows pass
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_rows_kernel(const BwdParams p) {
    extern __shared__ float smem[];
    const int d = p.d, Dv = p.Dv, dp = d + 4;
    float* q1s = smem;               // [kRows][d]
    float* q2s = q1s + kRows * d;    // [kRows][d]
    float* k1s = q2s + kRows * d;    // [kChunk][d+4]
    float* k2s = k1s + kChunk * dp;  // [kChunk][d+4]
    float* vs = k2s + kChunk * dp;   // [kChunk][Dv]
    float* red_w = vs + kChunk * Dv;  // [kRows][Dv]
    float* red_l = red_w + kRows * Dv;  // [kRows]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, h = blockIdx.y;
    const int row0 = blockIdx.x * kRows;
    const int i = row0 + warp;
    const int dvl = Dv / 32;

    stage_rows<T>(q1s, d, p.q1, p.sq1, b, h, row0, kRows, d, p.N, warp, lane);
    stage_rows<T>(q2s, d, p.q2, p.sq2, b, h, row0, kRows, d, p.N, warp, lane);

    const float scale = 1.0f / sqrtf((float)d);
    float m1 = -INFINITY, m2 = -INFINITY, l1 = 0.f, l2 = 0.f;
    float o1[kDVL], o2[kDVL];
#pragma unroll
    for (int t = 0; t < kDVL; ++t) o1[t] = o2[t] = 0.f;

    const int kend = p.causal ? min(p.N, row0 + kRows) : p.N;
    for (int c0 = 0; c0 < kend; c0 += kChunk) {
        __syncthreads();
        stage_rows<T>(k1s, dp, p.k1, p.sk1, b, h, c0, kChunk, d, p.N, warp, lane);
        stage_rows<T>(k2s, dp, p.k2, p.sk2, b, h, c0, kChunk, d, p.N, warp, lane);
        stage_rows<T>(vs, Dv, p.v, p.sv, b, h, c0, kChunk, Dv, p.N, warp, lane);
        __syncthreads();
        if (i >= p.N) continue;

        const int j = c0 + lane;
        const bool visible = (j < p.N) && (!p.causal || j <= i);
        float s1 = dot4(q1s + warp * d, k1s + lane * dp, d);
        float s2 = dot4(q2s + warp * d, k2s + lane * dp, d);
        s1 = visible ? s1 * scale : -INFINITY;
        s2 = visible ? s2 * scale : -INFINITY;
        const float n1 = fmaxf(m1, warp_max(s1));
        const float n2 = fmaxf(m2, warp_max(s2));
        if (n1 == -INFINITY) continue;  // no visible key in this chunk yet
        const float a1 = expf(m1 - n1), a2 = expf(m2 - n2);
        const float e1 = visible ? expf(s1 - n1) : 0.f;
        const float e2 = visible ? expf(s2 - n2) : 0.f;
        l1 = l1 * a1 + warp_sum(e1);
        l2 = l2 * a2 + warp_sum(e2);
        m1 = n1;
        m2 = n2;
#pragma unroll
        for (int t = 0; t < kDVL; ++t) {
            o1[t] *= a1;
            o2[t] *= a2;
        }
        const int nk = min(kChunk, kend - c0);
        for (int jj = 0; jj < nk; ++jj) {
            const float w1 = __shfl_sync(0xffffffffu, e1, jj);
            const float w2 = __shfl_sync(0xffffffffu, e2, jj);
#pragma unroll
            for (int t = 0; t < kDVL; ++t) {
                if (t < dvl) {
                    const float vv = vs[jj * Dv + lane + 32 * t];
                    o1[t] = fmaf(w1, vv, o1[t]);
                    o2[t] = fmaf(w2, vv, o2[t]);
                }
            }
        }
    }

    // Per-row gradient of the RMSNorm, gain and (1 - lambda_init) scale.
    float dlam_row = 0.f;
    float dw_row[kDVL];
#pragma unroll
    for (int t = 0; t < kDVL; ++t) dw_row[t] = 0.f;
    if (i < p.N) {
        const float il1 = 1.0f / l1, il2 = 1.0f / l2;
        float oh[kDVL], ss = 0.f;
#pragma unroll
        for (int t = 0; t < kDVL; ++t) {
            o1[t] *= il1;  // the map-1 output P1 V
            o2[t] *= il2;  // the map-2 output P2 V
            oh[t] = o1[t] - p.lambda * o2[t];
            ss = fmaf(oh[t], oh[t], ss);  // zero beyond Dv
        }
        ss = warp_sum(ss);
        const float r = sqrtf(ss / (float)Dv + p.eps);
        const float ir = 1.0f / r;
        const float cs = 1.0f - p.lambda_init;
        const T* dy = static_cast<const T*>(p.dy) + (((int64_t)b * p.N + i) * p.H + h) * Dv;
        float g[kDVL], nn[kDVL], gn = 0.f;
#pragma unroll
        for (int t = 0; t < kDVL; ++t) {
            g[t] = nn[t] = 0.f;
            if (t < dvl) {
                const int c = lane + 32 * t;
                const float dyc = ldf(dy + c);
                nn[t] = oh[t] * ir;
                g[t] = dyc * (p.norm_w ? p.norm_w[c] : 1.f) * cs;
                dw_row[t] = dyc * nn[t] * cs;
                gn = fmaf(g[t], nn[t], gn);
            }
        }
        gn = warp_sum(gn) / (float)Dv;
        float* dorow = p.d_o + row_index(p, b, h, i) * Dv;
        float x1 = 0.f, x2 = 0.f;
#pragma unroll
        for (int t = 0; t < kDVL; ++t) {
            if (t < dvl) {
                const float dO = (g[t] - nn[t] * gn) * ir;
                dorow[lane + 32 * t] = dO;
                x1 = fmaf(dO, o1[t], x1);
                x2 = fmaf(dO, o2[t], x2);
            }
        }
        x1 = warp_sum(x1);
        x2 = warp_sum(x2);
        dlam_row = -x2;
        if (lane == 0) {
            float* st = p.stats + row_index(p, b, h, i) * 4;
            st[0] = m1 + logf(l1);
            st[1] = m2 + logf(l2);
            st[2] = x1;              // D1 = dO . P1 V
            st[3] = -p.lambda * x2;  // D2 = -lambda dO . P2 V
        }
    }

    // Per-CTA partial sums of dlambda and dw, in a fixed order.
#pragma unroll
    for (int t = 0; t < kDVL; ++t)
        if (t < dvl) red_w[warp * Dv + lane + 32 * t] = dw_row[t];
    if (lane == 0) red_l[warp] = dlam_row;
    __syncthreads();
    const int64_t cta = ((int64_t)b * p.H + h) * gridDim.x + blockIdx.x;
    for (int c = threadIdx.x; c < Dv; c += blockDim.x) {
        float s = 0.f;
        for (int w = 0; w < kRows; ++w) s += red_w[w * Dv + c];
        p.part_w[cta * Dv + c] = s;
    }
    if (threadIdx.x == 0) {
        float s = 0.f;
        for (int w = 0; w < kRows; ++w) s += red_l[w];
        p.part_lam[cta] = s;
    }
}

// ------------------------------------------------------------- key-side pass
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_kv_kernel(const BwdParams p) {
    extern __shared__ float smem[];
    const int d = p.d, Dv = p.Dv, dp = d + 4, dvp = Dv + 4;
    float* k1w = smem;                 // [kRows][d]   this CTA's keys
    float* k2w = k1w + kRows * d;      // [kRows][d]
    float* vw = k2w + kRows * d;       // [kRows][Dv]
    float* q1c = vw + kRows * Dv;      // [kChunk][d+4] streamed query rows
    float* q2c = q1c + kChunk * dp;    // [kChunk][d+4]
    float* doc = q2c + kChunk * dp;    // [kChunk][Dv+4]
    float* stc = doc + kChunk * dvp;   // [kChunk][4]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, h = blockIdx.y;
    const int key0 = blockIdx.x * kRows;
    const int j = key0 + warp;
    const int dl = d / 32, dvl = Dv / 32;

    stage_rows<T>(k1w, d, p.k1, p.sk1, b, h, key0, kRows, d, p.N, warp, lane);
    stage_rows<T>(k2w, d, p.k2, p.sk2, b, h, key0, kRows, d, p.N, warp, lane);
    stage_rows<T>(vw, Dv, p.v, p.sv, b, h, key0, kRows, Dv, p.N, warp, lane);

    const float scale = 1.0f / sqrtf((float)d);
    float dv[kDVL], dk1[kDL], dk2[kDL];
#pragma unroll
    for (int t = 0; t < kDVL; ++t) dv[t] = 0.f;
#pragma unroll
    for (int t = 0; t < kDL; ++t) dk1[t] = dk2[t] = 0.f;

    // Queries before this CTA's first key see none of its keys (causal).
    const int qbeg = p.causal ? (key0 / kChunk) * kChunk : 0;
    for (int c0 = qbeg; c0 < p.N; c0 += kChunk) {
        __syncthreads();
        stage_rows<T>(q1c, dp, p.q1, p.sq1, b, h, c0, kChunk, d, p.N, warp, lane);
        stage_rows<T>(q2c, dp, p.q2, p.sq2, b, h, c0, kChunk, d, p.N, warp, lane);
        stage_ws_rows(doc, dvp, p.d_o, p, b, h, c0, kChunk, Dv, warp, lane);
        if (threadIdx.x < kChunk * 4) {
            const int r = threadIdx.x / 4;
            stc[threadIdx.x] = (c0 + r < p.N) ? p.stats[row_index(p, b, h, c0 + r) * 4 + (threadIdx.x % 4)] : 0.f;
        }
        __syncthreads();
        if (j >= p.N) continue;

        const int i = c0 + lane;  // this lane's query row
        const bool visible = (i < p.N) && (!p.causal || j <= i);
        const float s1 = dot4(q1c + lane * dp, k1w + warp * d, d);
        const float s2 = dot4(q2c + lane * dp, k2w + warp * d, d);
        const float da = dot4(doc + lane * dvp, vw + warp * Dv, Dv);
        const float p1 = visible ? expf(s1 * scale - stc[lane * 4 + 0]) : 0.f;
        const float p2 = visible ? expf(s2 * scale - stc[lane * 4 + 1]) : 0.f;
        const float a = p1 - p.lambda * p2;
        const float ds1 = p1 * (da - stc[lane * 4 + 2]);
        const float ds2 = p2 * (-p.lambda * da - stc[lane * 4 + 3]);

        const int nq = min(kChunk, p.N - c0);
        for (int jj = 0; jj < nq; ++jj) {
            const float aa = __shfl_sync(0xffffffffu, a, jj);
            const float e1 = __shfl_sync(0xffffffffu, ds1, jj);
            const float e2 = __shfl_sync(0xffffffffu, ds2, jj);
#pragma unroll
            for (int t = 0; t < kDVL; ++t)
                if (t < dvl) dv[t] = fmaf(aa, doc[jj * dvp + lane + 32 * t], dv[t]);
#pragma unroll
            for (int t = 0; t < kDL; ++t) {
                if (t < dl) {
                    dk1[t] = fmaf(e1, q1c[jj * dp + lane + 32 * t], dk1[t]);
                    dk2[t] = fmaf(e2, q2c[jj * dp + lane + 32 * t], dk2[t]);
                }
            }
        }
    }
    if (j >= p.N) return;
    const int64_t ri = row_index(p, b, h, j);
#pragma unroll
    for (int t = 0; t < kDVL; ++t)
        if (t < dvl) p.dv[ri * Dv + lane + 32 * t] = dv[t];
#pragma unroll
    for (int t = 0; t < kDL; ++t) {
        if (t < dl) {
            p.dk1[ri * d + lane + 32 * t] = dk1[t] * scale;
            p.dk2[ri * d + lane + 32 * t] = dk2[t] * scale;
        }
    }
}

// ----------------------------------------------------------- query-side pass
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_q_kernel(const BwdParams p) {
    extern __shared__ float smem[];
    const int d = p.d, Dv = p.Dv, dp = d + 4, dvp = Dv + 4;
    float* q1w = smem;                 // [kRows][d]   this CTA's query rows
    float* q2w = q1w + kRows * d;      // [kRows][d]
    float* dow = q2w + kRows * d;      // [kRows][Dv]
    float* k1c = dow + kRows * Dv;     // [kChunk][d+4] streamed keys
    float* k2c = k1c + kChunk * dp;    // [kChunk][d+4]
    float* vc = k2c + kChunk * dp;     // [kChunk][Dv+4]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, h = blockIdx.y;
    const int row0 = blockIdx.x * kRows;
    const int i = row0 + warp;
    const int dl = d / 32;

    stage_rows<T>(q1w, d, p.q1, p.sq1, b, h, row0, kRows, d, p.N, warp, lane);
    stage_rows<T>(q2w, d, p.q2, p.sq2, b, h, row0, kRows, d, p.N, warp, lane);
    stage_ws_rows(dow, Dv, p.d_o, p, b, h, row0, kRows, Dv, warp, lane);
    float lse1 = 0.f, lse2 = 0.f, D1 = 0.f, D2 = 0.f;
    if (i < p.N) {
        const float* st = p.stats + row_index(p, b, h, i) * 4;
        lse1 = st[0];
        lse2 = st[1];
        D1 = st[2];
        D2 = st[3];
    }

    const float scale = 1.0f / sqrtf((float)d);
    float dq1[kDL], dq2[kDL];
#pragma unroll
    for (int t = 0; t < kDL; ++t) dq1[t] = dq2[t] = 0.f;

    const int kend = p.causal ? min(p.N, row0 + kRows) : p.N;
    for (int c0 = 0; c0 < kend; c0 += kChunk) {
        __syncthreads();
        stage_rows<T>(k1c, dp, p.k1, p.sk1, b, h, c0, kChunk, d, p.N, warp, lane);
        stage_rows<T>(k2c, dp, p.k2, p.sk2, b, h, c0, kChunk, d, p.N, warp, lane);
        stage_rows<T>(vc, dvp, p.v, p.sv, b, h, c0, kChunk, Dv, p.N, warp, lane);
        __syncthreads();
        if (i >= p.N) continue;

        const int j = c0 + lane;  // this lane's key
        const bool visible = (j < p.N) && (!p.causal || j <= i);
        const float s1 = dot4(q1w + warp * d, k1c + lane * dp, d);
        const float s2 = dot4(q2w + warp * d, k2c + lane * dp, d);
        const float da = dot4(dow + warp * Dv, vc + lane * dvp, Dv);
        const float p1 = visible ? expf(s1 * scale - lse1) : 0.f;
        const float p2 = visible ? expf(s2 * scale - lse2) : 0.f;
        const float ds1 = p1 * (da - D1);
        const float ds2 = p2 * (-p.lambda * da - D2);

        const int nk = min(kChunk, kend - c0);
        for (int jj = 0; jj < nk; ++jj) {
            const float e1 = __shfl_sync(0xffffffffu, ds1, jj);
            const float e2 = __shfl_sync(0xffffffffu, ds2, jj);
#pragma unroll
            for (int t = 0; t < kDL; ++t) {
                if (t < dl) {
                    dq1[t] = fmaf(e1, k1c[jj * dp + lane + 32 * t], dq1[t]);
                    dq2[t] = fmaf(e2, k2c[jj * dp + lane + 32 * t], dq2[t]);
                }
            }
        }
    }
    if (i >= p.N) return;
    const int64_t ri = row_index(p, b, h, i);
#pragma unroll
    for (int t = 0; t < kDL; ++t) {
        if (t < dl) {
            p.dq1[ri * d + lane + 32 * t] = dq1[t] * scale;
            p.dq2[ri * d + lane + 32 * t] = dq2[t] * scale;
        }
    }
}

// -------------------------------------------------------------- reductions
// Block 0: dlambda = sum of the row-pass partials; block 1 + c: dw[c].
__global__ void __launch_bounds__(256) bwd_reduce_kernel(const BwdParams p, int64_t n_part) {
    __shared__ float red[8];
    const int c = (int)blockIdx.x - 1;
    float s = 0.f;
    for (int64_t k = threadIdx.x; k < n_part; k += blockDim.x)
        s += c < 0 ? p.part_lam[k] : p.part_w[k * p.Dv + c];
    s = warp_sum(s);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < 8; ++w) t += red[w];
        if (c < 0)
            *p.dlambda = t;
        else
            p.dnorm_w[c] = t;
    }
}

template <typename T>
cudaError_t launch_typed(const BwdParams& p, cudaStream_t stream) {
    const int d = p.d, Dv = p.Dv;
    const size_t s_rows = sizeof(float) * (size_t)(2 * kRows * d + 2 * kChunk * (d + 4) + kChunk * Dv +
                                                   kRows * Dv + kRows);
    const size_t s_kv = sizeof(float) * (size_t)(2 * kRows * d + kRows * Dv + 2 * kChunk * (d + 4) +
                                                 kChunk * (Dv + 4) + kChunk * 4);
    const size_t s_q = sizeof(float) * (size_t)(2 * kRows * d + kRows * Dv + 2 * kChunk * (d + 4) +
                                                kChunk * (Dv + 4));
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(bwd_rows_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_rows)) ||
        (e = cudaFuncSetAttribute(bwd_kv_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_kv)) ||
        (e = cudaFuncSetAttribute(bwd_q_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_q)))
        return e;
    const dim3 grid((p.N + kRows - 1) / kRows, p.H, p.B);
    bwd_rows_kernel<T><<<grid, kThreads, s_rows, stream>>>(p);
    bwd_kv_kernel<T><<<grid, kThreads, s_kv, stream>>>(p);
    bwd_q_kernel<T><<<grid, kThreads, s_q, stream>>>(p);
    const int64_t n_part = (int64_t)grid.x * p.H * p.B;
    return launch_bwd_reduce(p, n_part, stream);
}

}  // namespace

int64_t bwd_partial_count(int B, int H, int N) { return (int64_t)((N + kRows - 1) / kRows) * H * B; }

cudaError_t launch_bwd_reduce(const BwdParams& p, int64_t n_part, cudaStream_t stream) {
    bwd_reduce_kernel<<<p.dnorm_w ? 1 + p.Dv : 1, 256, 0, stream>>>(p, n_part);
    return cudaGetLastError();
}

cudaError_t launch_bwd_simt(const BwdParams& p, cudaStream_t stream) {
    if (p.d % 32 || p.d > 32 * kDL || p.Dv % 32 || p.Dv > 32 * kDVL) return cudaErrorInvalidValue;
    switch (p.in_dtype) {
        case 0: return launch_typed<float>(p, stream);
        case 1: return launch_typed<__nv_bfloat16>(p, stream);
        case 2: return launch_typed<__half>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace da
