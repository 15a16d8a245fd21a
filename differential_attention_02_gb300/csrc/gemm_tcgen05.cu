// bf16 or fp16 GEMM C[M, N] = A[M, K] . W[K, N] on the 5th-generation tensor cores
// (tcgen05.mma, fp32 accumulator in tensor memory), fed by TMA.
//
// Used for the projections of the multi-head differential attention module:
// [Q | K | V] = X W and Y = concat(heads) W_O, "A Simple Principle From
// Noise-Cancelling Headphones Supercharges Transformers Like Never Before"
// (intoai.pub), sections "Moving On To The Differential Transformer" and
// "Differential Attention With Multiple Heads".
//
// Persistent: one CTA per SM walks the 128 x 256 output tiles (M-block-major,
// so the CTAs running at once share W and each A row block through L2). Two
// 256-column TMEM accumulators let the epilogue of one tile overlap the MMAs
// of the next. Warp roles: warp 0 = TMA producer (one lane; A K-major
// 128 x 64 boxes, W N-major 64 x 64 boxes, both 128-byte swizzled, 4-stage
// ring), warp 1 = TMEM owner and MMA issuer (an elected lane of the converged warp; B given as MN-major),
// warps 2..5 = epilogue: warp w owns TMEM lanes (tile rows) 32*(w%4)..+31 and
// writes them through 128-byte-swizzled shared-memory boxes with TMA stores,
// 64 columns per pass.
//
// Epilogue modes for the DIFF Transformer layer ("The Overall Architecture Of The
// Multi-Head Differential Transformer", intoai.pub; "Estrutura multi-head e
// arquitetura completa", hada): the residual add Y = X + MultiHead(.) with the
// row sums of Y^2 its RMSNorm needs and a 16-bit copy of Y (times the norm's gain)
// as the next GEMM's operand, since RMSNorm(Y) W = (Y (g W)) / r row by row; and
// the SwiGLU of the gate/up product, scaled by 1/r, so that neither the
// normalised activations nor the gate/up output make a round trip through HBM.
#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

constexpr int BM = kGemmBM, BN = kGemmBN, BK = kGemmBK;
constexpr int kStages = 4;  // 48 KB each: ~2K cycles of MMA work in flight
constexpr int kABytes = BM * BK * 2;             // 16 KB
constexpr int kWBoxBytes = BK * 64 * 2;          // 8 KB: 64 K-rows x 64 N-columns
constexpr int kWBytes = (BN / 64) * kWBoxBytes;  // 32 KB
constexpr int kStageBytes = kABytes + kWBytes;
constexpr int kOutBoxBytes = 32 * 128;           // one [32 rows][128 bytes] output box
constexpr int kOutCols = 64;                     // output columns per epilogue pass
constexpr int kOutWarpBytes = 2 * kOutBoxBytes;  // one epilogue warp's staging: 64 columns of fp32
constexpr int kOffOut = kStages * kStageBytes;
constexpr int kOffBar = kOffOut + 4 * kOutWarpBytes;
constexpr int kThreads = 6 * 32;
constexpr uint32_t kTmemCols = 2 * BN;           // two fp32 accumulators
constexpr size_t kSmem = 1024 + (size_t)kOffBar + 256;
static_assert(kSmem <= 232448, "shared memory budget");

struct GemmBars {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(GemmBars) <= 256, "barrier block fits the 256 bytes past kOffBar");

__global__ void __launch_bounds__(kThreads, 1) gemm_bf16_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    GemmBars* bars = reinterpret_cast<GemmBars*>(smem + kOffBar);
    volatile int* abort_flag = &bars->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_n = (p.N + BN - 1) / BN;
    const int tiles = ((p.M + BM - 1) / BM) * tiles_n;
    const int kblocks = (p.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->acc_full[b], 1);
            mbar_init(&bars->acc_empty[b], 4);  // one arrival per epilogue warp
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // The setup above may overlap the previous kernel's tail; A (and R, the gain, the row
    // sums) may be that kernel's output.
    pdl_trigger();
    pdl_wait();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_a);
            tma_prefetch_desc(&p.tm_w);
            int it = 0;
            bool go = true;
            for (int t = blockIdx.x; go && t < tiles; t += gridDim.x) {
                const int m0 = (t / tiles_n) * BM, n0 = (t % tiles_n) * BN;
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % kStages;
                    if (!mbar_wait(&bars->empty[s], ((it / kStages) & 1) ^ 1, abort_flag, p.err, 0x21)) {
                        go = false;
                        break;
                    }
                    uint8_t* st = smem + s * kStageBytes;
                    mbar_arrive_expect_tx(&bars->full[s], kStageBytes);
                    index_ok(m0 < p.M && n0 < p.N && kb * BK < p.K, p.err, 0xB0);
                    tma_load_2d(st, &p.tm_a, &bars->full[s], kb * BK, m0);
#pragma unroll
                    for (int c = 0; c < BN / 64; ++c)
                        tma_load_2d(st + kABytes + c * kWBoxBytes, &p.tm_w, &bars->full[s], n0 + c * 64, kb * BK);
                }
            }
            // Drain: no copy may still be landing in shared memory when the CTA exits.
            for (int u = max(0, it - kStages); u < it; ++u)
                mbar_wait(&bars->full[u % kStages], (u / kStages) & 1, nullptr, p.err, 0x22);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp walks the loop and waits; one elected lane issues each
        // k-block's MMAs together with the commit that tracks them.
        const uint32_t idesc = idesc_kind_f16(BM, BN, /*A MN-major*/ 0, /*B MN-major*/ 1, p.ab_f16);
        // A: K-major, 128-byte rows; one K=16 step is 32 bytes along the row.
        // B: MN-major; 64-column boxes are kWBoxBytes apart (leading offset),
        // 8-row K groups 1024 bytes apart (stride offset); K=16 is 16 rows.
        const uint64_t da0 = sdesc_sw128(smem_u32(smem), 16, 1024);
        const uint64_t dw0 = sdesc_sw128(smem_u32(smem) + kABytes, kWBoxBytes, 1024);
        constexpr uint64_t kStep = kStageBytes >> 4;
        int it = 0, local = 0;
        bool go = true;
        for (int t = blockIdx.x; go && t < tiles; t += gridDim.x, ++local) {
            const int buf = local & 1;
            // The epilogue must have read this accumulator's previous tile.
            if (!mbar_wait_warp(&bars->acc_empty[buf], ((local >> 1) & 1) ^ 1, abort_flag, p.err, 0x23)) break;
            tc_fence_after();
            const uint32_t acc = tmem + buf * BN;
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int s = it % kStages;
                if (!mbar_wait_warp(&bars->full[s], (it / kStages) & 1, abort_flag, p.err, 0x24)) {
                    go = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_ss(acc, da0 + s * kStep + (uint64_t)(k * 2), dw0 + s * kStep + (uint64_t)(k * 128), idesc,
                                (kb > 0 || k > 0) ? 1u : 0u);
                    umma_commit(&bars->empty[s]);
                    if (kb == kblocks - 1) umma_commit(&bars->acc_full[buf]);
                }
                __syncwarp();
            }
        }
        // Every MMA issued (also before an abort) must finish before TMEM is freed.
        if (elect_one()) umma_commit(&bars->drain);
        __syncwarp();
        mbar_wait(&bars->drain, 0, nullptr, p.err, 0x25);
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int lg = warp & 3;  // TMEM lane group (tile rows) this warp may access
        uint8_t* stage = smem + kOffOut + lg * kOutWarpBytes;
        const int eb = p.out_bf16 || p.out_f16 ? 2 : 4;
        const int bw = 128 / eb;  // elements per 128-byte box row
        int local = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++local) {
            const int buf = local & 1;
            // tcgen05.ld is warp-collective: the decision to read TMEM is made per warp.
            bool ok = mbar_wait_warp(&bars->acc_full[buf], (local >> 1) & 1, abort_flag, p.err, 0x26);
            ok = __all_sync(0xffffffffu, ok && !*abort_flag);
            if (!ok) break;
            tc_fence_after();
            const int m0 = (t / tiles_n) * BM, n0 = (t % tiles_n) * BN;
            const uint32_t t_row = tmem + buf * BN + ((uint32_t)(lg * 32) << 16);
            const int row = m0 + lg * 32 + lane;  // this lane's output row
            const bool row_ok = row < p.M;
            if (p.mode == 2) {
                // SwiGLU: gate columns [0,128) and up columns [128,256) of the tile give output
                // columns n0/2 + [0,128), 64 per pass. The row scale 1/r from the partial sums.
                float ir = 1.f;
                if (p.row_sq_in) {
                    float ssum = 0.f;
                    if (row_ok)
                        for (int i = 0; i < p.n_sq; ++i) ssum += p.row_sq_in[(int64_t)row * p.n_sq + i];
                    ir = row_ok ? 1.0f / sqrtf(ssum / p.sq_count + p.eps) : 0.f;
                }
#pragma unroll 1
                for (int pass = 0; pass < 2; ++pass) {
                    if (lane == 0) tma_store_wait_read();
                    __syncwarp();
#pragma unroll 1
                    for (int c = 0; c < 2; ++c) {
                        uint32_t g[32], u[32];
                        tmem_ld32(t_row + pass * 64 + c * 32, g);
                        tmem_ld32(t_row + 128 + pass * 64 + c * 32, u);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint32_t w4[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                float hv[2];
#pragma unroll
                                for (int k = 0; k < 2; ++k) {
                                    const int i = 8 * j + 2 * e + k;
                                    const float gs = __uint_as_float(g[i]) * ir, us = __uint_as_float(u[i]) * ir;
                                    hv[k] = gs / (1.0f + expf(-gs)) * us;  // silu(g) * u
                                }
                                w4[e] = pack_16x2(hv[0], hv[1], p.out_f16 != 0);
                            }
                            *reinterpret_cast<uint4*>(stage + sw128_offset(lane, c * 4 + j)) =
                                make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                    if (pass == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars->acc_empty[buf]);
                    }
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        index_ok(m0 < p.M && n0 < p.N && m0 >= 0 && n0 >= 0, p.err, 0xB2);
                        tma_store_2d(&p.tm_c, stage, n0 / 2 + pass * 64, m0 + lg * 32);
                        tma_store_commit();
                    }
                }
                continue;
            }
            float sq = 0.f;  // mode 1: this row's sum of C^2 over the tile
            // Mode 1: this row's residual slice of a 64-column pass as raw 16-byte words (16 for
            // fp32, 8 for 16-bit R), loaded one pass ahead so a load's latency overlaps the
            // previous pass's work instead of stalling every 32-column chunk.
            uint4 rcur[16], rnext[16];
            auto load_resid = [&](int pass, uint4* dst) {
                if (p.mode != 1 || !row_ok) return;
                const int col0 = n0 + pass * kOutCols;
                if (p.r_dtype == 0) {
                    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const float*>(p.resid) + row * p.ld_r + col0);
#pragma unroll
                    for (int q = 0; q < 16; ++q) dst[q] = src[q];
                } else {
                    const uint4* src =
                        reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.resid) + row * p.ld_r + col0);
#pragma unroll
                    for (int q = 0; q < 8; ++q) dst[q] = src[q];
                }
            };
            load_resid(0, rcur);
#pragma unroll 1
            for (int pass = 0; pass < BN / kOutCols; ++pass) {
                if (pass + 1 < BN / kOutCols) load_resid(pass + 1, rnext);
                // The staging boxes of this warp must be free (its previous stores read them).
                if (lane == 0) tma_store_wait_read();
                __syncwarp();
#pragma unroll
                for (int c = 0; c < kOutCols / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(t_row + pass * kOutCols + c * 32, r);
                    const int col0 = n0 + pass * kOutCols + c * 32;  // first of these 32 columns
                    float res[32];
                    if (p.mode == 1) {
                        if (row_ok) {
                            if (p.r_dtype == 0) {
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    const uint4 v = rcur[c * 8 + q];
                                    res[4 * q] = __uint_as_float(v.x); res[4 * q + 1] = __uint_as_float(v.y);
                                    res[4 * q + 2] = __uint_as_float(v.z); res[4 * q + 3] = __uint_as_float(v.w);
                                }
                            } else {
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const uint4 v = rcur[c * 4 + q];
                                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        float2 f2;
                                        if (p.r_dtype == 2) f2 = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
                                        else f2 = make_float2(bf16lo_to_f32(w4[e]), bf16hi_to_f32(w4[e]));
                                        res[8 * q + 2 * e] = f2.x;
                                        res[8 * q + 2 * e + 1] = f2.y;
                                    }
                                }
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) res[i] = 0.f;
                        }
                    }
                    tmem_ld_wait();
                    if (p.mode == 1) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float y = __uint_as_float(r[i]) + res[i];
                            r[i] = __float_as_uint(y);
                            sq = fmaf(y, y, sq);
                        }
                        if (p.c16 && row_ok) {
                            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.c16) + row * p.ld_c16 + col0);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint32_t w4[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int i = 8 * q + 2 * e;
                                    float a0 = __uint_as_float(r[i]), a1 = __uint_as_float(r[i + 1]);
                                    if (p.c16_gain) {
                                        a0 *= p.c16_gain[col0 + i];
                                        a1 *= p.c16_gain[col0 + i + 1];
                                    }
                                    w4[e] = pack_16x2(a0, a1, p.c16_f16 != 0);
                                }
                                dst[q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                            }
                        }
                    }
                    if (eb == 2) {
                        // 32 columns = half a box row: 16-byte chunks c*4 .. c*4+3 of the one box.
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float* f = reinterpret_cast<const float*>(r + 8 * j);
                            uint4 v;
                            if (p.out_f16)
                                v = make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]),
                                               pack_f16x2(f[6], f[7]));
                            else
                                v = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                               pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
                            *reinterpret_cast<uint4*>(stage + sw128_offset(lane, c * 4 + j)) = v;
                        }
                    } else {
                        // 32 fp32 columns = one box row.
                        uint8_t* box = stage + c * kOutBoxBytes;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<uint4*>(box + sw128_offset(lane, j)) =
                                make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                    }
                }
                if (pass == BN / kOutCols - 1) {
                    // Done reading this accumulator: the MMA warp may reuse it.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->acc_empty[buf]);
                }
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {
                    const int nbox = kOutCols / bw;
                    for (int i = 0; i < nbox; ++i) {
                        // The tile starts inside C; boxes past its end are clipped by the store.
                        index_ok(m0 < p.M && n0 < p.N && m0 >= 0 && n0 >= 0, p.err, 0xB1);
                        tma_store_2d(&p.tm_c, stage + i * kOutBoxBytes, n0 + pass * kOutCols + i * bw, m0 + lg * 32);
                    }
                    tma_store_commit();
                }
#pragma unroll
                for (int q = 0; q < 16; ++q) rcur[q] = rnext[q];
            }
            if (p.mode == 1 && p.row_sq && row_ok) p.row_sq[(int64_t)row * tiles_n + n0 / BN] = sq;
        }
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_gemm_bf16(const GemmParams& p, cudaStream_t stream) {
    cudaError_t e = prepare_once<gemm_bf16_kernel>((int)kSmem);
    if (e != cudaSuccess) return e;
    int sms = 0;
    if ((e = device_sm_count(&sms)) != cudaSuccess) return e;
    const int tiles = ((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
    return launch_pdl(gemm_bf16_kernel, dim3(tiles < sms ? tiles : sms), dim3(kThreads), kSmem, stream, p);
}

}  // namespace da
