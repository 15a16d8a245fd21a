// Split-KV decode of differential attention: one new query token per
// sequence against its KV cache, bf16 or fp8 (e4m3) cache, fp32 arithmetic.
//
// What it computes: the last row of the DiffAttn formula of "Differential
// Transformer: Transformer que cancela ruído de atenção" (section "Como a
// atenção diferencial funciona") — both softmax maps over the cached keys,
// their lambda-weighted difference times V — then the per-head RMSNorm and the
// (1 - lambda_init) scale (section "Estrutura multi-head e arquitetura
// completa"). Reading the whole KV cache at every decoding step is the cost
// the priorstack.com article on Multi-Head Latent Attention describes, so this
// path is bound by HBM bandwidth.
//
// Kernel 1 (split): grid (splits, H, B). A producer warp streams 64-key
// stages of K1, K2 (128-byte-swizzled tiles) and V through a TMA + mbarrier
// ring; eight consumer warps score every stage (four lanes per key, eight keys
// per warp), keep an online-softmax state per map, accumulate P.V on the
// CUDA cores, and at the end the CTA merges its warps' states and writes one
// partial state (m, l, o[Dv]) per map to the workspace.
// Kernel 2 (merge): one CTA per (b, h) merges the split partials exactly,
// combines o1/l1 - lambda o2/l2, applies RMSNorm and (1 - lambda_init).
//
// fp8 cache: K1, K2 and V hold e4m3 values with one scale per tensor (cache
// value = stored value x scale). The pages point to lower-bit quantization as a
// use of the method's smaller activation outliers ("Differential Transformer:
// Transformer que cancela ruído de atenção", section "Resultados experimentais
// e efeitos de aplicação"); here the cache is quantized to halve the bytes the
// HBM-bound decode reads. The K scales are folded into the query, the V scale
// into the merged output. Per byte read the fp8 path has twice the arithmetic
// of the bf16 one (every e4m3 pair is converted to fp16 and then fp32), so its
// loop is kept lean: packed fp32 FMAs on element pairs for the scores and P.V,
// the eight keys of a warp unrolled, and a lazily moved running maximum.
#include <cuda_fp8.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

constexpr int kStageKeys = 64;
constexpr int kConsumerWarps = 8;
constexpr int kKeysPerWarp = kStageKeys / kConsumerWarps;  // 8: four lanes per key
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr float kLog2e = 1.4426950408889634f;

template <int D, int DV, bool FP8>
struct DecodeCfg {
    static constexpr int kEB = FP8 ? 1 : 2;                     // bytes per cached element
    // bf16: 64-element (128-byte) swizzled boxes per key row; fp8: one box of the whole row
    // (64 bytes unswizzled for d = 64, 128 bytes swizzled for d = 128).
    static constexpr int kBoxesK = FP8 ? 1 : D / 64;
    static constexpr int kKBytes = kStageKeys * D * kEB;        // one map's keys per stage
    static constexpr int kVBytes = kStageKeys * DV * kEB;
    static constexpr int kStageBytes = 2 * kKBytes + kVBytes;
    // fp8 stages are half the size: the same count keeps a d = 64 CTA at ~58 KB of shared
    // memory, so three CTAs (24 consumer warps) share an SM instead of two.
    static constexpr int kStages = (D == 64) ? 3 : 2;
    static constexpr int kQuarter = D / 4;                      // dot-product elements per lane
    static constexpr int kChunks = kQuarter * kEB / 16;         // 16-byte chunks per lane per key
    static constexpr int kDVL = DV / 32;                        // value columns per lane
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + 2 * kStages * 8 + 64 +
                                    (size_t)kConsumerWarps * (4 + 2 * DV) * 4;
};

// Element (key r, 16-byte chunk c) of a swizzled K tile: each 64-element box is
// [kStageKeys][128 bytes] with chunk c stored at position c ^ (r % 8).
__device__ __forceinline__ const uint4* k_chunk(const uint8_t* tile, int r, int c) {
    const int box = c >> 3, cc = c & 7;
    return reinterpret_cast<const uint4*>(tile + box * (kStageKeys * 128) + r * 128 + ((cc ^ (r & 7)) << 4));
}

// 16-byte chunk c of key row r in a stage's K tile of either element type.
template <int D, bool FP8>
__device__ __forceinline__ const uint4* key_chunk(const uint8_t* tile, int r, int c) {
    if constexpr (FP8 && D == 64) return reinterpret_cast<const uint4*>(tile + r * 64 + (c << 4));
    else return k_chunk(tile, r, c);
}

// Four e4m3 values packed in a 32-bit word (lowest byte first) as two float pairs.
__device__ __forceinline__ void fp8x4_to_f32x4(uint32_t w, float2* f) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
    f[0] = __half22float2(__half2(lo));
    f[1] = __half22float2(__half2(hi));
}

// Stale-maximum threshold (log2 units): a running maximum moves only when a score exceeds it
// by more than this, so the weights exp2(s - m) stay below 2^8 and most stages skip the
// rescale of the accumulators. The stale maximum is exact: l and o use the same one.
constexpr float kLazyMax = 8.f;

template <int D, int DV, bool FP8>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const __grid_constant__ DecodeParams p) {
    using C = DecodeCfg<D, DV, FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(stages + C::kStages * C::kStageBytes);
    uint64_t* empty = full + C::kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + C::kStages);
    float* red = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes + 2 * C::kStages * 8 + 64);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int len = p.seq_lens ? min(max(p.seq_lens[b], 0), p.L) : p.L;
    const int key_begin = split * p.keys_per_split;
    const int key_end = min(len, key_begin + p.keys_per_split);
    const int n_stages = key_end > key_begin ? (key_end - key_begin + kStageKeys - 1) / kStageKeys : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------- producer: one elected lane issues every TMA ----------------
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_k1);
            tma_prefetch_desc(&p.tm_k2);
            tma_prefetch_desc(&p.tm_v);
            const int hk = h / p.kv_group;  // the KV head this query head reads
            // Paged cache: stage t is the sequence's page key / 64; its physical page is
            // read from the block table one stage ahead, off the path to the copy.
            const int32_t* pages = p.block_table ? p.block_table + (int64_t)b * p.max_pages : nullptr;
            int next_page = (pages && n_stages > 0) ? pages[key_begin / kStageKeys] : 0;
            int t = 0;
            for (; t < n_stages; ++t) {
                const int s = t % C::kStages;
                const int page = next_page;
                if (pages && t + 1 < n_stages) next_page = pages[key_begin / kStageKeys + t + 1];
                if (!mbar_wait(&empty[s], ((t / C::kStages) & 1) ^ 1, abort_flag, p.err, 0x11)) break;
                uint8_t* st = stages + s * C::kStageBytes;
                // Coordinates (row, batch) of the stage: (key, b) in a contiguous cache,
                // (0, page) in a paged one.
                const int row = pages ? 0 : key_begin + t * kStageKeys;
                // The stage lies inside this split's keys, and a paged stage's page inside the pool
                // (a debug build that finds a page outside it reports it and reads page 0 instead).
                index_ok(key_begin + t * kStageKeys < key_end && hk < p.H / p.kv_group, p.err, 0xA0);
                const int bz = pages ? (index_ok(page >= 0 && page < p.num_pages, p.err, 0xA1) ? page : 0) : b;
                mbar_arrive_expect_tx(&full[s], C::kStageBytes);
#pragma unroll
                for (int x = 0; x < C::kBoxesK; ++x) {  // fp8: one box, x = 0
                    tma_load_4d(st + x * kStageKeys * 128, &p.tm_k1, &full[s], x * 64, row, hk, bz);
                    tma_load_4d(st + C::kKBytes + x * kStageKeys * 128, &p.tm_k2, &full[s], x * 64, row, hk, bz);
                }
                tma_load_4d(st + 2 * C::kKBytes, &p.tm_v, &full[s], 0, row, hk, bz);
            }
            // Do not leave while copies into this CTA's shared memory may still land.
            for (int u = max(0, t - C::kStages); u < t; ++u)
                mbar_wait(&full[u % C::kStages], (u / C::kStages) & 1, nullptr, p.err, 0x12);
        }
    } else {
        // ---------------- consumers ----------------
        const int kq = lane >> 2;      // key within the warp's 8
        const int quarter = lane & 3;  // quarter of the d elements this lane dots
        // Query halves, pre-scaled so scores come out in log2 units.
        float q1r[C::kQuarter], q2r[C::kQuarter];  // fp8: read in pairs by the packed FMAs
        {
            const __nv_bfloat16* q1 = reinterpret_cast<const __nv_bfloat16*>(p.q1) + ((int64_t)b * p.H + h) * D;
            const __nv_bfloat16* q2 = reinterpret_cast<const __nv_bfloat16*>(p.q2) + ((int64_t)b * p.H + h) * D;
            const float sc = kLog2e / sqrtf((float)D);
            const float sc1 = sc * p.k1_scale, sc2 = sc * p.k2_scale;  // 1 for a bf16 cache
#pragma unroll
            for (int e = 0; e < C::kQuarter; ++e) {
                q1r[e] = __bfloat162float(q1[quarter * C::kQuarter + e]) * sc1;
                q2r[e] = __bfloat162float(q2[quarter * C::kQuarter + e]) * sc2;
            }
        }
        float m1 = -INFINITY, m2 = -INFINITY, l1 = 0.f, l2 = 0.f;
        float o1[C::kDVL], o2[C::kDVL];
#pragma unroll
        for (int t = 0; t < C::kDVL; ++t) o1[t] = o2[t] = 0.f;

        for (int t = 0; t < n_stages; ++t) {
            const int s = t % C::kStages;
            if (!mbar_wait(&full[s], (t / C::kStages) & 1, abort_flag, p.err, 0x13)) break;
            const uint8_t* st = stages + s * C::kStageBytes;
            const int r = warp * kKeysPerWarp + kq;  // key row inside the stage
            const int key = key_begin + t * kStageKeys + r;
            // Scores: this lane's quarter of both dot products, reduced over the 4 lanes of the key.
            float s1 = 0.f, s2 = 0.f;
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
                const int chunk = quarter * C::kChunks + c;
                const uint4 a = *key_chunk<D, FP8>(st, r, chunk);
                const uint4 bb = *key_chunk<D, FP8>(st + C::kKBytes, r, chunk);
                const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {bb.x, bb.y, bb.z, bb.w};
                if constexpr (FP8) {
                    // packed fp32 FMAs on (even, odd) element pairs
                    float2 t1 = make_float2(0.f, 0.f), t2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float2 fa[2], fb[2];
                        fp8x4_to_f32x4(aw[e], fa);
                        fp8x4_to_f32x4(bw[e], fb);
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int i = c * 16 + 4 * e + 2 * u;
                            t1 = __ffma2_rn(make_float2(q1r[i], q1r[i + 1]), fa[u], t1);
                            t2 = __ffma2_rn(make_float2(q2r[i], q2r[i + 1]), fb[u], t2);
                        }
                    }
                    s1 += t1.x + t1.y;
                    s2 += t2.x + t2.y;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        s1 = fmaf(q1r[c * 8 + 2 * e], bf16lo_to_f32(aw[e]), s1);
                        s1 = fmaf(q1r[c * 8 + 2 * e + 1], bf16hi_to_f32(aw[e]), s1);
                        s2 = fmaf(q2r[c * 8 + 2 * e], bf16lo_to_f32(bw[e]), s2);
                        s2 = fmaf(q2r[c * 8 + 2 * e + 1], bf16hi_to_f32(bw[e]), s2);
                    }
                }
            }
            s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
            s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
            s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
            s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
            const bool ok = key < key_end;
            s1 = ok ? s1 : -INFINITY;
            s2 = ok ? s2 : -INFINITY;
            // Max over the warp's 8 keys (lanes 4 apart hold different keys).
            float c1 = s1, c2 = s2;
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                c1 = fmaxf(c1, __shfl_xor_sync(0xffffffffu, c1, o));
                c2 = fmaxf(c2, __shfl_xor_sync(0xffffffffu, c2, o));
            }
            const int nk = min(kKeysPerWarp, key_end - (key_begin + t * kStageKeys + warp * kKeysPerWarp));
            if (nk > 0) {
                if constexpr (FP8) {
                    // c1, c2 and the maxima are the same in every lane: the branch is warp-uniform
                    if (c1 > m1 + kLazyMax || c2 > m2 + kLazyMax) {
                        const float n1 = c1 > m1 + kLazyMax ? c1 : m1, n2 = c2 > m2 + kLazyMax ? c2 : m2;
                        const float a1 = fast_exp2(m1 - n1), a2 = fast_exp2(m2 - n2);
                        l1 *= a1;
                        l2 *= a2;
                        m1 = n1;
                        m2 = n2;
#pragma unroll
                        for (int u = 0; u < C::kDVL; ++u) {
                            o1[u] *= a1;
                            o2[u] *= a2;
                        }
                    }
                }
                float p1, p2;
                if constexpr (FP8) {
                    p1 = ok ? fast_exp2(s1 - m1) : 0.f;
                    p2 = ok ? fast_exp2(s2 - m2) : 0.f;
                    l1 += p1;  // per-lane partial; every key is counted by its 4 lanes
                    l2 += p2;
                } else {
                    const float n1 = fmaxf(m1, c1), n2 = fmaxf(m2, c2);
                    const float a1 = fast_exp2(m1 - n1), a2 = fast_exp2(m2 - n2);
                    p1 = ok ? fast_exp2(s1 - n1) : 0.f;
                    p2 = ok ? fast_exp2(s2 - n2) : 0.f;
                    l1 = l1 * a1 + p1;  // per-lane partial; every key is counted by its 4 lanes
                    l2 = l2 * a2 + p2;
                    m1 = n1;
                    m2 = n2;
#pragma unroll
                    for (int u = 0; u < C::kDVL; ++u) {
                        o1[u] *= a1;
                        o2[u] *= a2;
                    }
                }
                const uint8_t* vt = st + 2 * C::kKBytes;
                auto pv_key = [&](int kk) {
                    const float w1 = __shfl_sync(0xffffffffu, p1, kk * 4);
                    const float w2 = __shfl_sync(0xffffffffu, p2, kk * 4);
                    const uint8_t* vrow = vt + (size_t)(warp * kKeysPerWarp + kk) * DV * C::kEB;
                    if constexpr (FP8) {
                        // kDVL consecutive e4m3 values: columns lane * kDVL ...
                        float2 f[C::kDVL / 2];
                        if constexpr (C::kDVL == 4) {
                            fp8x4_to_f32x4(*reinterpret_cast<const uint32_t*>(vrow + lane * 4), f);
                        } else {
                            const uint2 vv = *reinterpret_cast<const uint2*>(vrow + lane * 8);
                            fp8x4_to_f32x4(vv.x, f);
                            fp8x4_to_f32x4(vv.y, f + 2);
                        }
                        // packed fp32 FMAs on column pairs, one weight broadcast to both halves
                        const float2 ww1 = make_float2(w1, w1), ww2 = make_float2(w2, w2);
#pragma unroll
                        for (int u = 0; u < C::kDVL / 2; ++u) {
                            const float2 r1 = __ffma2_rn(ww1, f[u], make_float2(o1[2 * u], o1[2 * u + 1]));
                            const float2 r2 = __ffma2_rn(ww2, f[u], make_float2(o2[2 * u], o2[2 * u + 1]));
                            o1[2 * u] = r1.x;
                            o1[2 * u + 1] = r1.y;
                            o2[2 * u] = r2.x;
                            o2[2 * u + 1] = r2.y;
                        }
                    } else if constexpr (C::kDVL == 4) {
                        const uint2 vv = *reinterpret_cast<const uint2*>(vrow + lane * 8);
                        const float f[4] = {bf16lo_to_f32(vv.x), bf16hi_to_f32(vv.x), bf16lo_to_f32(vv.y),
                                            bf16hi_to_f32(vv.y)};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            o1[u] = fmaf(w1, f[u], o1[u]);
                            o2[u] = fmaf(w2, f[u], o2[u]);
                        }
                    } else {
                        const uint4 vv = *reinterpret_cast<const uint4*>(vrow + lane * 16);
                        const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            o1[2 * u] = fmaf(w1, bf16lo_to_f32(vw[u]), o1[2 * u]);
                            o1[2 * u + 1] = fmaf(w1, bf16hi_to_f32(vw[u]), o1[2 * u + 1]);
                            o2[2 * u] = fmaf(w2, bf16lo_to_f32(vw[u]), o2[2 * u]);
                            o2[2 * u + 1] = fmaf(w2, bf16hi_to_f32(vw[u]), o2[2 * u + 1]);
                        }
                    }
                };
                if (nk == kKeysPerWarp) {  // warp-uniform: every key of the warp is in range
#pragma unroll
                    for (int kk = 0; kk < kKeysPerWarp; ++kk) pv_key(kk);
                } else {
                    for (int kk = 0; kk < nk; ++kk) pv_key(kk);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // Warp state -> shared memory: [warp][m1, l1, m2, l2, o1[DV], o2[DV]].
        l1 = warp_sum(l1) * 0.25f;
        l2 = warp_sum(l2) * 0.25f;
        float* w = red + warp * (4 + 2 * DV);
        if (lane == 0) {
            w[0] = m1;
            w[1] = l1;
            w[2] = m2;
            w[3] = l2;
        }
#pragma unroll
        for (int u = 0; u < C::kDVL; ++u) {
            w[4 + lane * C::kDVL + u] = o1[u];
            w[4 + DV + lane * C::kDVL + u] = o2[u];
        }
    }
    __syncthreads();
    if (*abort_flag) return;

    // Merge the consumer warps into this split's partial state.
    const int64_t slot = ((int64_t)b * p.H + h) * p.num_splits + split;
    float M1 = -INFINITY, M2 = -INFINITY;
    for (int w = 0; w < kConsumerWarps; ++w) {
        M1 = fmaxf(M1, red[w * (4 + 2 * DV) + 0]);
        M2 = fmaxf(M2, red[w * (4 + 2 * DV) + 2]);
    }
    for (int c = threadIdx.x; c < 2 * DV; c += blockDim.x) {
        const int map = c / DV;
        const float M = map ? M2 : M1;
        float acc = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = red[w * (4 + 2 * DV) + 2 * map];
            if (mw != -INFINITY) acc += red[w * (4 + 2 * DV) + 4 + c] * fast_exp2(mw - M);
        }
        p.part_o[slot * 2 * DV + c] = acc;
    }
    if (threadIdx.x < 2) {
        const int map = threadIdx.x;
        const float M = map ? M2 : M1;
        float l = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = red[w * (4 + 2 * DV) + 2 * map];
            if (mw != -INFINITY) l += red[w * (4 + 2 * DV) + 2 * map + 1] * fast_exp2(mw - M);
        }
        p.part_stats[slot * 4 + 2 * map] = M;
        p.part_stats[slot * 4 + 2 * map + 1] = l;
    }
}

// One CTA of DV threads per (b, h): exact merge of the split states of both
// maps, combination, RMSNorm over DV channels and the (1 - lambda_init) scale.
template <int DV>
__global__ void __launch_bounds__(DV) decode_merge_kernel(const __grid_constant__ DecodeParams p) {
    __shared__ float red[DV / 32];
    const int bh = blockIdx.x, c = threadIdx.x;
    const int S = p.num_splits;
    const float* st = p.part_stats + (int64_t)bh * S * 4;
    const float* po = p.part_o + (int64_t)bh * S * 2 * DV;
    float M1 = -INFINITY, M2 = -INFINITY;
    for (int s = 0; s < S; ++s) {
        M1 = fmaxf(M1, st[s * 4 + 0]);
        M2 = fmaxf(M2, st[s * 4 + 2]);
    }
    float l1 = 0.f, l2 = 0.f, o1 = 0.f, o2 = 0.f;
    for (int s = 0; s < S; ++s) {
        if (st[s * 4 + 0] != -INFINITY) {
            const float e = fast_exp2(st[s * 4 + 0] - M1);
            l1 += st[s * 4 + 1] * e;
            o1 += po[s * 2 * DV + c] * e;
        }
        if (st[s * 4 + 2] != -INFINITY) {
            const float e = fast_exp2(st[s * 4 + 2] - M2);
            l2 += st[s * 4 + 3] * e;
            o2 += po[s * 2 * DV + DV + c] * e;
        }
    }
    const float oh = (o1 / l1 - p.lambda * (o2 / l2)) * p.v_scale;  // v_scale 1 for a bf16 cache
    float ss = warp_sum(oh * oh);
    if ((c & 31) == 0) red[c >> 5] = ss;
    __syncthreads();
    ss = 0.f;
#pragma unroll
    for (int w = 0; w < DV / 32; ++w) ss += red[w];
    float y = oh * ((1.0f - p.lambda_init) / sqrtf(ss / (float)DV + p.eps));
    if (p.norm_w) y *= p.norm_w[c];
    const int64_t o = (int64_t)bh * DV + c;
    if (p.out_bf16)
        reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(y);
    else
        reinterpret_cast<float*>(p.out)[o] = y;
}

template <int D, int DV, bool FP8>
cudaError_t launch_t(const DecodeParams& p, cudaStream_t stream) {
    using C = DecodeCfg<D, DV, FP8>;
    auto k = decode_split_kernel<D, DV, FP8>;
    cudaError_t e = prepare_once<decode_split_kernel<D, DV, FP8>>((int)C::kSmem);
    if (e != cudaSuccess) return e;
    k<<<dim3(p.num_splits, p.H, p.B), kThreads, C::kSmem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_merge_kernel<DV><<<p.B * p.H, DV, 0, stream>>>(p);
    return cudaGetLastError();
}

// Appends each sequence's new token (K1, K2, V rows of every KV head) to a paged
// cache: position pos = seq_lens[b] - 1 goes to row pos % 64 of page
// block_table[b][pos / 64]. One warp per (sequence, KV head), 16-byte copies.
// Positions or pages outside the table or the pool are skipped.
__global__ void kv_append_paged_kernel(const __grid_constant__ KvAppendParams p) {
    const int b = blockIdx.x / p.H_kv, h = blockIdx.x % p.H_kv;
    const int pos = p.seq_lens[b] - 1;
    if (pos < 0 || pos / kStageKeys >= p.max_pages) return;
    const int page = p.block_table[(int64_t)b * p.max_pages + pos / kStageKeys];
    if (page < 0 || page >= p.num_pages) return;
    const int row = pos % kStageKeys;
    const int64_t src_k = ((int64_t)b * p.H_kv + h) * p.d, src_v = ((int64_t)b * p.H_kv + h) * p.Dv;
    const int64_t dst_k = page * p.k_stride_page + h * p.k_stride_h + row * p.k_stride_row;
    const int64_t dst_v = page * p.v_stride_page + h * p.v_stride_h + row * p.v_stride_row;
    const int ck = p.d / 8, cv = p.Dv / 8;  // 16-byte chunks per row
    for (int c = threadIdx.x; c < 2 * ck + cv; c += blockDim.x) {
        const uint4* src;
        uint4* dst;
        if (c < ck) {
            src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.k1_new) + src_k) + c;
            dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.k1_pages) + dst_k) + c;
        } else if (c < 2 * ck) {
            src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.k2_new) + src_k) + (c - ck);
            dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.k2_pages) + dst_k) + (c - ck);
        } else {
            src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.v_new) + src_v) + (c - 2 * ck);
            dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.v_pages) + dst_v) + (c - 2 * ck);
        }
        *dst = *src;
    }
}

// The same append into fp8 (e4m3) pages: each value is stored as
// sat_e4m3(x / scale), rounded to nearest even. 8 values per lane step.
__global__ void kv_append_paged_fp8_kernel(const __grid_constant__ KvAppendParams p) {
    const int b = blockIdx.x / p.H_kv, h = blockIdx.x % p.H_kv;
    const int pos = p.seq_lens[b] - 1;
    if (pos < 0 || pos / kStageKeys >= p.max_pages) return;
    const int page = p.block_table[(int64_t)b * p.max_pages + pos / kStageKeys];
    if (page < 0 || page >= p.num_pages) return;
    const int row = pos % kStageKeys;
    const int64_t src_k = ((int64_t)b * p.H_kv + h) * p.d, src_v = ((int64_t)b * p.H_kv + h) * p.Dv;
    const int64_t dst_k = page * p.k_stride_page + h * p.k_stride_h + row * p.k_stride_row;
    const int64_t dst_v = page * p.v_stride_page + h * p.v_stride_h + row * p.v_stride_row;
    const int ck = p.d / 8, cv = p.Dv / 8;  // 8-value groups per row
    for (int c = threadIdx.x; c < 2 * ck + cv; c += blockDim.x) {
        const __nv_bfloat16* src;
        uint8_t* dst;
        float scale;
        if (c < ck) {
            src = static_cast<const __nv_bfloat16*>(p.k1_new) + src_k + c * 8;
            dst = static_cast<uint8_t*>(p.k1_pages) + dst_k + c * 8;
            scale = p.k1_scale;
        } else if (c < 2 * ck) {
            src = static_cast<const __nv_bfloat16*>(p.k2_new) + src_k + (c - ck) * 8;
            dst = static_cast<uint8_t*>(p.k2_pages) + dst_k + (c - ck) * 8;
            scale = p.k2_scale;
        } else {
            src = static_cast<const __nv_bfloat16*>(p.v_new) + src_v + (c - 2 * ck) * 8;
            dst = static_cast<uint8_t*>(p.v_pages) + dst_v + (c - 2 * ck) * 8;
            scale = p.v_scale;
        }
        const uint4 x = *reinterpret_cast<const uint4*>(src);
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
        uint32_t q[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float2 a = make_float2(__fdiv_rn(bf16lo_to_f32(xw[2 * k]), scale),
                                         __fdiv_rn(bf16hi_to_f32(xw[2 * k]), scale));
            const float2 bb = make_float2(__fdiv_rn(bf16lo_to_f32(xw[2 * k + 1]), scale),
                                          __fdiv_rn(bf16hi_to_f32(xw[2 * k + 1]), scale));
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(bb, __NV_SATFINITE, __NV_E4M3);
            q[k] = lo | (hi << 16);
        }
        *reinterpret_cast<uint2*>(dst) = make_uint2(q[0], q[1]);
    }
}

}  // namespace

int decode_keys_per_stage(int) { return kStageKeys; }

cudaError_t launch_kv_append_paged(const KvAppendParams& p, cudaStream_t stream) {
    if (p.fp8)
        kv_append_paged_fp8_kernel<<<p.B * p.H_kv, 32, 0, stream>>>(p);
    else
        kv_append_paged_kernel<<<p.B * p.H_kv, 32, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_decode_bf16(const DecodeParams& p, cudaStream_t stream) {
    if (p.d == 64 && p.Dv == 128) return p.kv_fp8 ? launch_t<64, 128, true>(p, stream) : launch_t<64, 128, false>(p, stream);
    if (p.d == 128 && p.Dv == 256)
        return p.kv_fp8 ? launch_t<128, 256, true>(p, stream) : launch_t<128, 256, false>(p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace da
