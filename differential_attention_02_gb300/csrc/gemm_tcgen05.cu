// bf16 GEMM C[M, N] = A[M, K] . W[K, N] on the 5th-generation tensor cores
// (tcgen05.mma, fp32 accumulator in tensor memory), fed by TMA.
//
// Used for the projections of the multi-head differential attention module:
// [Q | K | V] = X W and Y = concat(heads) W_O, "A Simple Principle From
// Noise-Cancelling Headphones Supercharges Transformers Like Never Before"
// (intoai.pub), sections "Moving On To The Differential Transformer" and
// "Differential Attention With Multiple Heads".
//
// One CTA per 128 x 256 output tile. Warp roles: warp 0 = TMA producer (one
// lane), warp 1 = MMA issuer (one lane) and TMEM owner, warps 2..5 = epilogue
// (warp w reads TMEM lanes 32*(w%4) .. +31). A is K-major (128-byte swizzled
// 128 x 64 boxes); W is N-major, so B is given to the MMA as MN-major (four
// 64 x 64 boxes per stage, 128-byte swizzled).
#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

constexpr int BM = kGemmBM, BN = kGemmBN, BK = kGemmBK;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK * 2;           // 16 KB
constexpr int kWBoxBytes = BK * 64 * 2;        // 8 KB: 64 K-rows x 64 N-columns
constexpr int kWBytes = (BN / 64) * kWBoxBytes;  // 32 KB
constexpr int kStageBytes = kABytes + kWBytes;
constexpr int kThreads = 6 * 32;
constexpr uint32_t kTmemCols = BN;  // fp32 accumulator, one column per output column
constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + 256;

__global__ void __launch_bounds__(kThreads, 1) gemm_bf16_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* acc_full = empty + kStages;
    uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int kblocks = (p.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_base_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_slot;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&p.tm_a);
            tma_prefetch_desc(&p.tm_w);
            int kb = 0;
            for (; kb < kblocks; ++kb) {
                const int s = kb % kStages;
                if (!mbar_wait(&empty[s], ((kb / kStages) & 1) ^ 1, abort_flag, p.err, 0x21)) break;
                uint8_t* st = smem + s * kStageBytes;
                mbar_arrive_expect_tx(&full[s], kStageBytes);
                tma_load_2d(st, &p.tm_a, &full[s], kb * BK, m0);
#pragma unroll
                for (int c = 0; c < BN / 64; ++c)
                    tma_load_2d(st + kABytes + c * kWBoxBytes, &p.tm_w, &full[s], n0 + c * 64, kb * BK);
            }
            for (int u = max(0, kb - kStages); u < kb; ++u)
                mbar_wait(&full[u % kStages], (u / kStages) & 1, nullptr, p.err, 0x22);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, /*A MN-major*/ 0, /*B MN-major*/ 1);
            bool ok = true;
            for (int kb = 0; kb < kblocks; ++kb) {
                const int s = kb % kStages;
                if (!mbar_wait(&full[s], (kb / kStages) & 1, abort_flag, p.err, 0x23)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(smem + s * kStageBytes);
                const uint32_t w_addr = a_addr + kABytes;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    // A: K-major, 128-byte rows; one K=16 step is 32 bytes along the row.
                    const uint64_t ad = sdesc_sw128(a_addr + k * 32, 16, 1024);
                    // B: MN-major; 64-column boxes are kWBoxBytes apart (leading offset),
                    // 8-row K groups are 1024 bytes apart (stride offset); K=16 is 16 rows.
                    const uint64_t bd = sdesc_sw128(w_addr + k * 16 * 128, kWBoxBytes, 1024);
                    umma_ss(tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit(&empty[s]);
            }
            umma_commit(acc_full);  // also drains the MMAs issued before an abort
            mbar_wait(acc_full, 0, nullptr, p.err, ok ? 0x24 : 0x25);
        }
    } else {
        // Epilogue: TMEM -> registers -> global.
        const int lg = warp & 3;  // TMEM lane group this warp may access
        // tcgen05.ld is warp-collective: the decision to read TMEM is made per warp.
        bool ok = mbar_wait_warp(acc_full, 0, abort_flag, p.err, 0x26);
        tc_fence_after();
        ok = __all_sync(0xffffffffu, ok && !*abort_flag);
        if (ok) {
            const int row = m0 + lg * 32 + lane;
            const uint32_t t_row = tmem + ((uint32_t)(lg * 32) << 16);
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(t_row + c0, r);
                tmem_ld_wait();
                const int col = n0 + c0;
                if (row < p.M && col < p.N) {
                    if (p.out_f16) {
                        __half* dst = reinterpret_cast<__half*>(p.C) + (int64_t)row * p.ldc + col;
                        if (col + 32 <= p.N) {
#pragma unroll
                            for (int j = 0; j < 32; j += 8) {
                                uint4 v;
                                v.x = pack_f16x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
                                v.y = pack_f16x2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                                v.z = pack_f16x2(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5]));
                                v.w = pack_f16x2(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7]));
                                *reinterpret_cast<uint4*>(dst + j) = v;
                            }
                        } else {
                            for (int j = 0; j < p.N - col; ++j) dst[j] = __float2half_rn(__uint_as_float(r[j]));
                        }
                    } else if (p.out_bf16) {
                        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.C) + (int64_t)row * p.ldc + col;
                        if (col + 32 <= p.N) {
#pragma unroll
                            for (int j = 0; j < 32; j += 8) {
                                uint4 v;
                                v.x = pack_bf16x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
                                v.y = pack_bf16x2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                                v.z = pack_bf16x2(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5]));
                                v.w = pack_bf16x2(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7]));
                                *reinterpret_cast<uint4*>(dst + j) = v;
                            }
                        } else {
                            for (int j = 0; j < p.N - col; ++j) dst[j] = __float2bfloat16_rn(__uint_as_float(r[j]));
                        }
                    } else {
                        float* dst = reinterpret_cast<float*>(p.C) + (int64_t)row * p.ldc + col;
                        if (col + 32 <= p.N) {
#pragma unroll
                            for (int j = 0; j < 32; j += 4)
                                *reinterpret_cast<float4*>(dst + j) =
                                    make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                                __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                        } else {
                            for (int j = 0; j < p.N - col; ++j) dst[j] = __uint_as_float(r[j]);
                        }
                    }
                }
            }
        }
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
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.N + BN - 1) / BN, (p.M + BM - 1) / BM);
    gemm_bf16_kernel<<<grid, kThreads, kSmem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace da
