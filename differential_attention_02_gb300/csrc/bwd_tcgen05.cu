// Backward pass of differential attention on the 5th-generation tensor cores
// (tcgen05.mma, TMEM accumulators, TMA), d = 64 and Dv = 128.
//
// The forward is, per head ("Differential Transformer: Transformer que cancela
// ruído de atenção", sections "Como a atenção diferencial funciona" and
// "Estrutura multi-head e arquitetura completa"; causal mask from the intoai.pub
// page, "A Deeper Dive Into Attention Calculations"):
//   P_m = softmax(Q_m K_m^T / sqrt(d) + M),  A = P1 - lambda P2,  O = A V,
//   y = O / sqrt(mean(O^2) + eps) * w * (1 - lambda_init).
// The pages train the model but print no gradient; this is the chain rule of
// that definition. The preparation pass (the forward kernel with another
// epilogue, launch_bwd_prep, or from a training forward's saved state,
// launch_bwd_prep_saved) leaves per query row: dO (the gradient of O, in the
// operand type), L_m (so that P_m = exp2(S_m log2(e)/sqrt(d) - L_m)),
// D1 = dO . (P1 V) and D2 = -lambda dO . (P2 V). Then, with dA = dO V^T:
//   dS1 = P1 (dA - D1),  dS2 = P2 (-lambda dA - D2)
//   dQ_m = dS_m K_m / sqrt(d)      (this file, kernel bwd_dq: one query tile per CTA)
//   dK_m = dS_m^T Q_m / sqrt(d),  dV = A^T dO
//                                  (kernel bwd_dkdv: one key tile per CTA)
// Each gradient row is written by exactly one CTA, so there are no atomics and
// the result does not depend on scheduling. The key side follows the preparation
// as a programmatic dependent launch (its setup and K/V loads overlap the
// preparation's last wave); the query side runs beside it on a forked stream.
//
// Both kernels keep S, dA and the gradient accumulators in TMEM. The products
// whose left operand is elementwise data (dS or A, rounded to the operand type)
// read it from TMEM in bwd_dq, like the forward's P.V (written over the score
// columns), and in bwd_dkdv from columns of its own (A, dS1) or shared memory (dS2),
// so that the score columns are free for the next step's products.
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

constexpr int BM = 128;               // query rows (bwd_dq) or keys (bwd_dkdv) per CTA
constexpr int kD = 64, kDV = 128;     // the supported head widths
constexpr int kThreads = 12 * 32;     // 8 elementwise warps, producer, MMA, 2 idle
constexpr int kWarpProducer = 8, kWarpMma = 9;
constexpr int kRegsLaunch = 168, kRegsMath = 224, kRegsOther = 56;
static_assert(2 * 128 * kRegsMath + 128 * kRegsOther <= kThreads * kRegsLaunch, "register split");

// One MMA group: K-major A and B tiles built from 128-byte-swizzled boxes of 64
// 16-bit elements per row. a_box / b_box: bytes between consecutive 64-element
// boxes of A / B; one K=16 step advances 32 bytes inside a box.
template <int KSTEPS, bool F16>
__device__ __forceinline__ void mma_kmajor(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, int a_box, int b_box,
                                           uint32_t idesc, bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
        const uint64_t oa = (uint64_t)(((kk >> 2) * a_box + (kk & 3) * 32) >> 4);
        const uint64_t ob = (uint64_t)(((kk >> 2) * b_box + (kk & 3) * 32) >> 4);
        umma_ss(d_tmem, a_desc + oa, b_desc + ob, idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
}

// D (+)= A[TMEM] * B[smem, MN-major]: A holds 16-bit pairs, K=16 per 8 columns;
// one K=16 step of B advances 16 rows of 128 bytes.
template <int KSTEPS>
__device__ __forceinline__ void mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk)
        umma_ts(d_tmem, a_tmem + kk * 8, b_desc + (uint64_t)(kk * 128), idesc, (accumulate || kk > 0) ? 1u : 0u);
}

// ============================================================================
// bwd_dq: one CTA per 128-row query tile of one (b, h).
// ============================================================================
// TMEM: S1 [0,128), S2 [128,256), dA [256,384), dQ1 [384,448), dQ2 [448,512).
// dS_m is written as 16-bit pairs into the first 64 columns of S_m.
// Warps 0..3 compute dS1 and warps 4..7 dS2 for row 32*(w%4)+lane; warp 8 loads,
// warp 9 issues the MMAs. Per key tile j the issue order is
//   dA(j), S1(j), S2(j)  ...  dQ1 += dS1(j) K1(j), dA(j+1), S1(j+1), dQ2 += dS2(j) K2(j), S2(j+1)
// so one group's elementwise work overlaps the other group's products; each dQ_m
// product runs in two halves of 64 keys, the first while the group computes the
// second half's dS_m.

// 16 lanes x 256 bits, four times along the columns: thread t gets lanes t/4 and t/4 + 8 of
// the addressed 16, columns 2(t%4) and 2(t%4)+1 of each 8-column block (registers
// 4i + {0, 1} from lane t/4, 4i + {2, 3} from lane t/4 + 8, block i).
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Shared-space load and store by 32-bit shared address (ld.shared / st.shared rather than
// generic accesses through a pointer whose address space the compiler cannot see).
__device__ __forceinline__ float4 lds_f4(uint32_t saddr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(saddr)
                 : "memory");
    return v;
}
// 16 lanes x 128 bits, four times along the columns: register 2i + a goes to lane t/4 + 8a
// of the addressed 16, column 4i + t%4.
__device__ __forceinline__ void tmem_st_16x128b_x4(uint32_t taddr, const uint32_t* r) {
    asm volatile("tcgen05.st.sync.aligned.16x128b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void sts_u32(uint32_t saddr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(saddr), "r"(v) : "memory");
}

namespace dq {
constexpr int kStages = 2;
constexpr int kQBytes = BM * kD * 2;           // 16 KB
constexpr int kOBytes = BM * kDV * 2;          // dO tile, 32 KB
constexpr int kKBytes = BM * kD * 2;           // one K tile of 128 keys, 16 KB
constexpr int kVBytes = BM * kDV * 2;          // 32 KB
constexpr int kStageBytes = 2 * kKBytes + kVBytes;
constexpr int kOffQ1 = 0, kOffQ2 = kQBytes, kOffO = 2 * kQBytes, kOffStages = 2 * kQBytes + kOBytes;
constexpr int kOffBar = kOffStages + kStages * kStageBytes;
constexpr size_t kSmem = 1024 + (size_t)kOffBar + 256;
static_assert(kSmem <= 232448, "shared memory budget");
constexpr uint32_t kColS = 0, kColA = 256, kColQ = 384;

struct Bars {
    uint64_t q_full;
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[2];   // S_m(j) and dA(j) in TMEM
    uint64_t ds_half[2];  // dS_m(j) of keys 0..63 in TMEM (4 warps each)
    uint64_t ds_full[2];  // dS_m(j) of keys 64..127 too
    uint64_t da_free;     // every elementwise warp has read dA(j) (8 warps)
    uint64_t dq_done;     // the last dQ products completed
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block fits the 256 bytes past kOffBar");
}  // namespace dq

template <bool F16>
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdTcParams p) {
    using namespace dq;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
    volatile int* abort_flag = &bars->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = (p.N + BM - 1) / BM;
    const int BH = p.B * p.H;
    const int qt = n_tiles - 1 - (int)(blockIdx.x / BH);  // heaviest tiles first
    const int bh = blockIdx.x % BH, b = bh / p.H, h = bh % p.H;
    const int q0 = qt * BM;
    const int nkv = p.causal ? qt + 1 : n_tiles;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->kv_full[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(&bars->s_full[g], 1);
            mbar_init(&bars->ds_half[g], 4);
            mbar_init(&bars->ds_full[g], 4);
        }
        mbar_init(&bars->da_free, 8);
        mbar_init(&bars->dq_done, 1);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbarrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&bars->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    uint8_t* stages = smem + kOffStages;

    if (warp >= 8) {
        setmaxnreg_dec<kRegsOther>();
        if (warp == kWarpProducer) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars->q_full, 2 * kQBytes + kOBytes);
                index_ok(q0 < p.N && h < p.H && b < p.B, p.err, 0xC0);
                tma_load_4d(smem + kOffQ1, &p.tm_q1, &bars->q_full, 0, q0, h, b);
                tma_load_4d(smem + kOffQ2, &p.tm_q2, &bars->q_full, 0, q0, h, b);
                for (int x = 0; x < kDV / 64; ++x)
                    tma_load_4d(smem + kOffO + x * BM * 128, &p.tm_do, &bars->q_full, x * 64, q0, h, b);
                int j = 0;
                for (; j < nkv; ++j) {
                    const int s = j % kStages;
                    if (!mbar_wait(&bars->kv_empty[s], ((j / kStages) & 1) ^ 1, abort_flag, p.err, 0xC1)) break;
                    uint8_t* st = stages + s * kStageBytes;
                    mbar_arrive_expect_tx(&bars->kv_full[s], kStageBytes);
                    index_ok(j * BM < p.N, p.err, 0xC2);
                    tma_load_4d(st, &p.tm_k1, &bars->kv_full[s], 0, j * BM, h, b);
                    tma_load_4d(st + kKBytes, &p.tm_k2, &bars->kv_full[s], 0, j * BM, h, b);
                    for (int x = 0; x < kDV / 64; ++x)
                        tma_load_4d(st + 2 * kKBytes + x * BM * 128, &p.tm_v, &bars->kv_full[s], x * 64, j * BM, h, b);
                }
                mbar_wait(&bars->q_full, 0, nullptr, p.err, 0xC3);
                for (int u = max(0, j - kStages); u < j; ++u)
                    mbar_wait(&bars->kv_full[u % kStages], (u / kStages) & 1, nullptr, p.err, 0xC4);
            }
        } else if (warp == kWarpMma) {
            const bool lead = elect_one();
            // K-major descriptors differ only in the start address: one base plus offsets.
            const uint64_t dq1 = sdesc_sw128(smem_u32(smem), 16, 1024);
            const uint64_t dq2 = dq1 + (kOffQ2 >> 4), ddo = dq1 + (kOffO >> 4);
            const uint64_t dk0 = dq1 + (kOffStages >> 4);                            // K-major K / V tiles
            const uint64_t dkn0 = sdesc_sw128(smem_u32(stages), BM * 128, 1024);      // K as an MN-major operand
            constexpr uint64_t kStep = kStageBytes >> 4, kK2 = kKBytes >> 4, kV = (2 * kKBytes) >> 4;
            constexpr uint32_t id_s = idesc_kind_f16(BM, BM, 0, 0, F16);    // S, dA: 128 x 128
            constexpr uint32_t id_q = idesc_kind_f16(BM, kD, 0, 1, F16);    // dQ: 128 x 64, B MN-major
            const uint32_t tS1 = tmem + kColS, tS2 = tmem + kColS + BM, tA = tmem + kColA;
            const uint32_t tQ1 = tmem + kColQ, tQ2 = tmem + kColQ + kD;
            auto issue_scores = [&](int s, bool second_map) {  // dA and S1, or S2, of stage s
                const uint64_t st = (uint64_t)s * kStep;
                if (!second_map) {
                    mma_kmajor<kDV / 16, F16>(tA, ddo, dk0 + st + kV, BM * 128, BM * 128, id_s, false);
                    mma_kmajor<kD / 16, F16>(tS1, dq1, dk0 + st, 0, 0, id_s, false);
                    umma_commit(&bars->s_full[0]);
                } else {
                    mma_kmajor<kD / 16, F16>(tS2, dq2, dk0 + st + kK2, 0, 0, id_s, false);
                    umma_commit(&bars->s_full[1]);
                }
            };
            bool ok = mbar_wait_warp(&bars->q_full, 0, abort_flag, p.err, 0xC5) &&
                      mbar_wait_warp(&bars->kv_full[0], 0, abort_flag, p.err, 0xC6);
            if (ok) {
                tc_fence_after();
                if (lead) {
                    issue_scores(0, false);
                    issue_scores(0, true);
                }
                __syncwarp();
            }
            for (int j = 0; ok && j < nkv; ++j) {
                const int s = j % kStages, s1 = (j + 1) % kStages;
                const bool more = j + 1 < nkv;
                const uint64_t st = (uint64_t)s * kStep;
                // Each map's dQ_m += dS_m K_m in two halves of four K-steps: keys 0..63 as soon
                // as the group has written them (ds_half), while it computes keys 64..127.
                constexpr uint64_t kHalfB = (uint64_t)(BM / 2 / 16) * 128;  // 4 K-steps of B
                // map 1: dQ1 += dS1 K1, then dA(j+1) and S1(j+1)
                if (!(ok = mbar_wait_warp(&bars->ds_half[0], j & 1, abort_flag, p.err, 0xCC))) break;
                tc_fence_after();
                if (lead) mma_tmem_a<BM / 32>(tQ1, tS1, dkn0 + st, id_q, j > 0);
                __syncwarp();
                ok = mbar_wait_warp(&bars->ds_full[0], j & 1, abort_flag, p.err, 0xC7);
                if (ok && more)
                    ok = mbar_wait_warp(&bars->kv_full[s1], ((j + 1) / kStages) & 1, abort_flag, p.err, 0xC8) &&
                         mbar_wait_warp(&bars->da_free, j & 1, abort_flag, p.err, 0xC9);
                if (!ok) break;
                tc_fence_after();
                if (lead) {
                    mma_tmem_a<BM / 32>(tQ1, tS1 + BM / 4, dkn0 + st + kHalfB, id_q, true);
                    if (more) issue_scores(s1, false);
                }
                __syncwarp();
                // map 2: dQ2 += dS2 K2, release the stage, then S2(j+1)
                if (!(ok = mbar_wait_warp(&bars->ds_half[1], j & 1, abort_flag, p.err, 0xCD))) break;
                tc_fence_after();
                if (lead) mma_tmem_a<BM / 32>(tQ2, tS2, dkn0 + st + kK2, id_q, j > 0);
                __syncwarp();
                if (!(ok = mbar_wait_warp(&bars->ds_full[1], j & 1, abort_flag, p.err, 0xCA))) break;
                tc_fence_after();
                if (lead) {
                    mma_tmem_a<BM / 32>(tQ2, tS2 + BM / 4, dkn0 + st + kK2 + kHalfB, id_q, true);
                    umma_commit(&bars->kv_empty[s]);
                    if (more) issue_scores(s1, true);
                    else umma_commit(&bars->dq_done);
                }
                __syncwarp();
            }
            if (lead) umma_commit(&bars->drain);
            __syncwarp();
            mbar_wait(&bars->drain, 0, nullptr, p.err, 0xCB);
        }
        tc_fence_before();
        named_bar_sync(2, kThreads);
        if (warp == kWarpMma) {
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
        return;
    }

    // ---------------------------------------------------------------- elementwise (map g)
    setmaxnreg_inc<kRegsMath>();
    const int g = warp >> 2, lg = warp & 3;
    const int r = lg * 32 + lane;
    const int qrow = q0 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(lg * 32) << 16);
    const uint32_t tS = lane_base + kColS + g * BM, tA = lane_base + kColA;
    const float sl2 = p.scale_log2, lam = p.lambda;
    // This row's L_g and D_g (rows past N read zeros and are never stored).
    float L = 0.f, Dg = 0.f;
    if (qrow < p.N) {
        const float4 st = *reinterpret_cast<const float4*>(p.stats + (((int64_t)b * p.H + h) * p.N + qrow) * 4);
        L = g ? st.y : st.x;
        Dg = g ? st.w : st.z;
    }
    const int lim = p.causal ? min(qrow + 1, p.N) : p.N;  // visible keys: key < lim
    const float ca = g ? -lam : 1.0f;                     // dA's factor in dP_g
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
        if (!(ok = mbar_wait_warp(&bars->s_full[g], j & 1, abort_flag, p.err, 0xD0 + g))) break;
        tc_fence_after();
        const int kbase = j * BM;
        // Masks only where some row of the tile may not see every key of the tile (the
        // causal diagonal, or keys past N): a warp-uniform test.
        const bool need_mask = (p.causal && kbase + BM > q0 + 1) || kbase + BM > p.N;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            uint32_t s[64], a[64];
            tmem_ld32(tS + hf * 64, s);
            tmem_ld32(tS + hf * 64 + 32, s + 32);
            tmem_ld32(tA + hf * 64, a);
            tmem_ld32(tA + hf * 64 + 32, a + 32);
            tmem_ld_wait();
            if (hf == 1) {  // dA(j) fully read: the next dA may overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->da_free);
            }
            uint32_t pk[32];
            // dS_g = P_g (c dA - D_g) with c = 1 (map 1) or -lambda (map 2)
            auto elementwise = [&](auto masked) {
#pragma unroll
                for (int i = 0; i < 64; i += 2) {
                    float ds[2];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        float pr = fast_exp2(fmaf(__uint_as_float(s[i + k]), sl2, -L));
                        if constexpr (decltype(masked)::value) {
                            if (kbase + hf * 64 + i + k >= lim) pr = 0.f;
                        }
                        ds[k] = pr * fmaf(ca, __uint_as_float(a[i + k]), -Dg);
                    }
                    pk[i / 2] = pack_p<F16>(ds[0], ds[1]);
                }
            };
            if (need_mask) elementwise(std::true_type{});
            else elementwise(std::false_type{});
            tmem_st32(tS + hf * 32, pk);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(hf == 0 ? &bars->ds_half[g] : &bars->ds_full[g]);
        }
    }
    // ---------------------------------------------------------------- epilogue: dQ_g rows
    // Read from TMEM with the 16x256b shape and stored straight from registers: per
    // instruction a warp writes 8 rows x 32 contiguous bytes (whole 32-byte sectors).
    if (ok) ok = mbar_wait_warp(&bars->dq_done, 0, abort_flag, p.err, 0xD2);
    tc_fence_after();
    {
        const float scale = p.scale;  // 1 / sqrt(d)
        const int tr = lane >> 2, tc = lane & 3;
        float* dst = (g ? p.dq2 : p.dq1) + ((int64_t)b * p.H + h) * p.N * kD;
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
            uint32_t v[2][16];
            if (ok) {  // TMEM is read by whole warps (ok is the same in every lane)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    tmem_ld_16x256b_x4(lane_base + ((uint32_t)(16 * hh) << 16) + kColQ + g * kD + c * 32, v[hh]);
                tmem_ld_wait();
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int ar = 0; ar < 2; ++ar) {
                    const int qr = q0 + lg * 32 + 16 * hh + 8 * ar + tr;
                    if (!ok || qr >= p.N) continue;
                    float* row = dst + (int64_t)qr * kD + c * 32 + 2 * tc;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int rg = 4 * i + 2 * ar;
                        *reinterpret_cast<float2*>(row + 8 * i) =
                            make_float2(__uint_as_float(v[hh][rg]) * scale, __uint_as_float(v[hh][rg + 1]) * scale);
                    }
                }
        }
    }
    tc_fence_before();
    named_bar_sync(2, kThreads);
}

// ============================================================================
// bwd_dkdv: one CTA per 128-key tile of one (b, h); query steps of 64 rows.
// ============================================================================
// TMEM (keys = lanes): S1^T [0,64), S2^T [64,128), dA^T [128,192) for one step's
// 64 queries; dV [192,320), dK1 [320,384), dK2 [384,448); A^T [448,480) and
// dS1^T [480,512) as 16-bit pairs. The elementwise warps write A^T = P1 - lambda P2
// and dS1^T (operand type) into those last columns and dS2^T to shared memory as a
// K-major 128-byte-swizzled tile: the left operands of
//   dV += A^T dO,  dK1 += dS1^T Q1  (A from TMEM),  dK2 += dS2^T Q2  (A from smem).
// Shared memory bandwidth bounds this kernel (the tensor core's operand reads, the
// TMA fills and the elementwise traffic), so what can live in TMEM does.
// The score columns are free as soon as the elementwise warps have loaded them,
// so the products of step t+1's scores run while step t's elementwise work does:
//   S/dA(0) ... [loads of S/dA(t)] S/dA(t+1) [elementwise t, stores] dV/dK(t) ...
// Warps 0..3 handle the step's queries 0..31, warps 4..7 queries 32..63 (every
// key row).
namespace dkdv {
constexpr int kSQ = 64;                        // queries per step
constexpr int kStages = 4;
constexpr int kKBytes = BM * kD * 2;           // K tile, 16 KB
constexpr int kVBytes = BM * kDV * 2;          // V tile, 32 KB
constexpr int kQBytes = kSQ * kD * 2;          // Q step, 8 KB
constexpr int kOBytes = kSQ * kDV * 2;         // dO step, 16 KB
constexpr int kSBytes = kSQ * 16;              // stats of the step, 1 KB
constexpr int kPBytes = BM * kSQ * 2;          // the dS2^T result tile, 16 KB
constexpr int kStageBytes = 2 * kQBytes + kOBytes + 1024;  // + stats, padded to keep tiles 1024-aligned
constexpr int kOffK1 = 0, kOffK2 = kKBytes, kOffV = 2 * kKBytes, kOffP = 2 * kKBytes + kVBytes;
constexpr int kOffStages = kOffP + kPBytes;
constexpr int kOffBar = kOffStages + kStages * kStageBytes;
constexpr size_t kSmem = 1024 + (size_t)kOffBar + 256;
static_assert(kSmem <= 232448, "shared memory budget");
static_assert(kOffP % 1024 == 0 && kOffStages % 1024 == 0 && kStageBytes % 1024 == 0, "swizzled tiles");
constexpr uint32_t kColS1 = 0, kColS2 = 64, kColA = 128, kColV = 192, kColK1 = 320, kColK2 = 384;
// A^T and dS1^T of the step as 16-bit pairs (the left operands of the dV and dK1 products)
constexpr uint32_t kColPA = 448, kColP1 = 480;
// Register split: the MMA warp's loop (two waits and two groups of products per step) needs
// more than 56 registers; the elementwise warps need far fewer than 216.
constexpr int kRegsMathKV = 216, kRegsOtherKV = 72;
static_assert(2 * 128 * kRegsMathKV + 128 * kRegsOtherKV <= kThreads * kRegsLaunch, "register split");

struct Bars {
    uint64_t kv_full;
    uint64_t q_full[kStages], q_empty[kStages];
    uint64_t s_full;      // S1^T, S2^T, dA^T of the step in TMEM
    uint64_t s_free;      // every elementwise warp has loaded them (8 warps)
    uint64_t p_full;      // A^T, dS1^T of the step in TMEM and dS2^T in shared memory (8 warps)
    uint64_t p_empty;     // the products that read them completed
    uint64_t acc_done;    // the last products completed
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block fits the 256 bytes past kOffBar");
}  // namespace dkdv

// D (+)= A[smem, K-major] * B[smem, MN-major]: one K=16 step advances 32 bytes in A's
// 128-byte rows and 16 rows of 128 bytes in B.
template <int KSTEPS>
__device__ __forceinline__ void mma_kmajor_mn(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk)
        umma_ss(d_tmem, a_desc + (uint64_t)(kk * 2), b_desc + (uint64_t)(kk * 128), idesc,
                (accumulate || kk > 0) ? 1u : 0u);
}

template <bool F16>
__global__ void __launch_bounds__(kThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdTcParams p) {
    using namespace dkdv;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
    volatile int* abort_flag = &bars->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = p.B * p.H;
    const int kt = (int)(blockIdx.x / BH);  // key tile; the first ones see the most queries
    const int bh = blockIdx.x % BH, b = bh / p.H, h = bh % p.H;
    const int k0 = kt * BM;
    const int qs0 = p.causal ? k0 : 0;                 // first query that can see these keys
    const int nsteps = (p.N - qs0 + kSQ - 1) / kSQ;    // query steps of 64 rows

    if (threadIdx.x == 0) {
        mbar_init(&bars->kv_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->q_full[s], 1);
            mbar_init(&bars->q_empty[s], 1);
        }
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->s_free, 8);
        mbar_init(&bars->p_full, 8);
        mbar_init(&bars->p_empty, 1);
        mbar_init(&bars->acc_done, 1);
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbarrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&bars->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    uint8_t* stages = smem + kOffStages;

    if (warp >= 8) {
        setmaxnreg_dec<kRegsOtherKV>();
        if (warp == kWarpProducer) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars->kv_full, 2 * kKBytes + kVBytes);
                index_ok(k0 < p.N && h < p.H && b < p.B, p.err, 0xE0);
                tma_load_4d(smem + kOffK1, &p.tm_k1, &bars->kv_full, 0, k0, h, b);
                tma_load_4d(smem + kOffK2, &p.tm_k2, &bars->kv_full, 0, k0, h, b);
                for (int x = 0; x < kDV / 64; ++x)
                    tma_load_4d(smem + kOffV + x * BM * 128, &p.tm_v, &bars->kv_full, x * 64, k0, h, b);
                const int row0 = (b * p.H + h) * p.N;  // first row of (b, h) in the stats matrix
                // dO and the statistics come from the preparation kernel launched before this one
                asm volatile("griddepcontrol.wait;" ::: "memory");
                int t = 0;
                for (; t < nsteps; ++t) {
                    const int s = t % kStages, q = qs0 + t * kSQ;
                    if (!mbar_wait(&bars->q_empty[s], ((t / kStages) & 1) ^ 1, abort_flag, p.err, 0xE1)) break;
                    uint8_t* st = stages + s * kStageBytes;
                    mbar_arrive_expect_tx(&bars->q_full[s], 2 * kQBytes + kOBytes + kSBytes);
                    index_ok(q < p.N, p.err, 0xE2);
                    tma_load_4d(st, &p.tm_q1s, &bars->q_full[s], 0, q, h, b);
                    tma_load_4d(st + kQBytes, &p.tm_q2s, &bars->q_full[s], 0, q, h, b);
                    for (int x = 0; x < kDV / 64; ++x)
                        tma_load_4d(st + 2 * kQBytes + x * kSQ * 128, &p.tm_dos, &bars->q_full[s], x * 64, q, h, b);
                    tma_load_2d(st + 2 * kQBytes + kOBytes, &p.tm_stats, &bars->q_full[s], 0, row0 + q);
                }
                mbar_wait(&bars->kv_full, 0, nullptr, p.err, 0xE3);
                for (int u = max(0, t - kStages); u < t; ++u)
                    mbar_wait(&bars->q_full[u % kStages], (u / kStages) & 1, nullptr, p.err, 0xE4);
            }
        } else if (warp == kWarpMma) {
            const bool lead = elect_one();
            // K-major descriptors differ only in the start address (bytes >> 4, far below the
            // field's 2^14 limit for shared memory): one base plus constant offsets.
            const uint64_t dk1 = sdesc_sw128(smem_u32(smem), 16, 1024);
            const uint64_t dk2 = dk1 + (kOffK2 >> 4), dv = dk1 + (kOffV >> 4);
            const uint64_t dp2 = dk1 + (kOffP >> 4);                                // dS2^T, K-major
            const uint64_t dst0 = dk1 + (kOffStages >> 4);                          // K-major step tiles
            const uint64_t dsn0 = sdesc_sw128(smem_u32(stages), kSQ * 128, 1024);   // MN-major step tiles
            constexpr uint64_t kStep = kStageBytes >> 4, kQ2 = kQBytes >> 4, kO = (2 * kQBytes) >> 4;
            constexpr uint32_t id_s = idesc_kind_f16(BM, kSQ, 0, 0, F16);    // S^T, dA^T: 128 x 64
            constexpr uint32_t id_v = idesc_kind_f16(BM, kDV, 0, 1, F16);    // dV: 128 x 128, B MN-major
            constexpr uint32_t id_k = idesc_kind_f16(BM, kD, 0, 1, F16);     // dK: 128 x 64, B MN-major
            auto issue_scores = [&](int s) {
                const uint64_t st = (uint64_t)s * kStep;
                mma_kmajor<kD / 16, F16>(tmem + kColS1, dk1, dst0 + st, 0, 0, id_s, false);
                mma_kmajor<kD / 16, F16>(tmem + kColS2, dk2, dst0 + st + kQ2, 0, 0, id_s, false);
                mma_kmajor<kDV / 16, F16>(tmem + kColA, dv, dst0 + st + kO, BM * 128, kSQ * 128, id_s, false);
                umma_commit(&bars->s_full);
            };
            bool ok = mbar_wait_warp(&bars->kv_full, 0, abort_flag, p.err, 0xE5) &&
                      (nsteps == 0 || mbar_wait_warp(&bars->q_full[0], 0, abort_flag, p.err, 0xE6));
            if (ok && nsteps > 0) {
                tc_fence_after();
                if (lead) issue_scores(0);
                __syncwarp();
            }
            for (int t = 0; ok && t < nsteps; ++t) {
                const int s = t % kStages, s1 = (t + 1) % kStages;
                const bool more = t + 1 < nsteps;
                const uint64_t st = (uint64_t)s * kStep;
                if (more) {
                    // step t+1's scores overwrite step t's once the elementwise warps hold them
                    ok = mbar_wait_warp(&bars->s_free, t & 1, abort_flag, p.err, 0xE7) &&
                         mbar_wait_warp(&bars->q_full[s1], ((t + 1) / kStages) & 1, abort_flag, p.err, 0xE8);
                    if (!ok) break;
                    tc_fence_after();
                    if (lead) issue_scores(s1);
                    __syncwarp();
                }
                ok = mbar_wait_warp(&bars->p_full, t & 1, abort_flag, p.err, 0xEA);
                if (!ok) break;
                tc_fence_after();
                if (lead) {
                    mma_tmem_a<kSQ / 16>(tmem + kColV, tmem + kColPA, dsn0 + st + kO, id_v, t > 0);
                    mma_tmem_a<kSQ / 16>(tmem + kColK1, tmem + kColP1, dsn0 + st, id_k, t > 0);
                    mma_kmajor_mn<kSQ / 16>(tmem + kColK2, dp2, dsn0 + st + kQ2, id_k, t > 0);
                    umma_commit(&bars->q_empty[s]);
                    umma_commit(&bars->p_empty);
                    if (!more) umma_commit(&bars->acc_done);
                }
                __syncwarp();
            }
            if (lead) umma_commit(&bars->drain);
            __syncwarp();
            mbar_wait(&bars->drain, 0, nullptr, p.err, 0xE9);
        }
        tc_fence_before();
        named_bar_sync(2, kThreads);
        if (warp == kWarpMma) {
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
        return;
    }

    // ---------------------------------------------------------------- elementwise
    setmaxnreg_inc<kRegsMathKV>();
    const int g = warp >> 2, lg = warp & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(lg * 32) << 16);
    const float sl2 = p.scale_log2, lam = p.lambda;
    constexpr int kHQ = kSQ / 2;  // queries per group and step
    // In the step loop a warp reads its 32 lanes x 32 query columns with the 16x256b shape:
    // thread (tr, tc) = (lane / 4, lane % 4) holds key rows lg*32 + 16h + 8a + tr (h, a in
    // {0, 1}) and the group's query columns 8i + 2tc + e (i in 0..3, e in {0, 1}), register
    // 4i + 2a + e of the load at lane offset 16h. It needs the statistics of 8 queries, where
    // a thread holding a whole key row would need all 32 (they are broadcast reads).
    const int tr = lane >> 2, tc = lane & 3;
    // Result tiles: row R at R*128 bytes, 16-byte chunk c at c ^ (R % 8); R % 8 = tr here.
    const uint32_t pbase = smem_u32(smem + kOffP) + (uint32_t)((lg * 32 + tr) * 128 + tc * 4);
    bool ok = true;
    for (int t = 0; ok && t < nsteps; ++t) {
        const int s = t % kStages;
        ok = mbar_wait_warp(&bars->s_full, t & 1, abort_flag, p.err, 0xF0);
        if (!ok) break;
        tc_fence_after();
        uint32_t s1[2][16], s2[2][16], ga[2][16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t lb = lane_base + ((uint32_t)(16 * h) << 16) + g * kHQ;
            tmem_ld_16x256b_x4(lb + kColS1, s1[h]);
            tmem_ld_16x256b_x4(lb + kColS2, s2[h]);
            tmem_ld_16x256b_x4(lb + kColA, ga[h]);
        }
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free);

        // L1, L2, D1, D2 of the thread's 8 queries
        const uint32_t stats = smem_u32(stages + s * kStageBytes + 2 * kQBytes + kOBytes) + (g * kHQ + 2 * tc) * 16;
        float4 st[4][2];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 2; ++e) st[i][e] = lds_f4(stats + (8 * i + e) * 16);
        const int qbase = qs0 + t * kSQ + g * kHQ;  // first query of this group's columns
        // Every (query, key) pair of the warp visible: no masks (warp-uniform).
        const bool full = (!p.causal || qbase >= k0 + lg * 32 + 31) && qbase + kHQ <= p.N;
        uint32_t pa[2][2][4], p1[2][2][4], p2[2][2][4];
        auto elementwise = [&](auto masked) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int ar = 0; ar < 2; ++ar)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float va[2], v1[2], v2[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int reg = 4 * i + 2 * ar + e;
                            const float4 q4 = st[i][e];
                            float e1 = fast_exp2(fmaf(__uint_as_float(s1[h][reg]), sl2, -q4.x));
                            float e2 = fast_exp2(fmaf(__uint_as_float(s2[h][reg]), sl2, -q4.y));
                            const float da = __uint_as_float(ga[h][reg]);
                            float d1 = da - q4.z, d2 = fmaf(-lam, da, -q4.w);
                            if constexpr (decltype(masked)::value) {
                                // a query past N reads another row's statistics: every result is zeroed
                                const int q = qbase + 8 * i + 2 * tc + e;
                                const int kr = k0 + lg * 32 + 16 * h + 8 * ar + tr;
                                const bool vis = q < p.N && (!p.causal || kr <= q);
                                e1 = vis ? e1 : 0.f;
                                e2 = vis ? e2 : 0.f;
                                d1 = vis ? d1 : 0.f;
                                d2 = vis ? d2 : 0.f;
                            }
                            va[e] = fmaf(-lam, e2, e1);
                            v1[e] = e1 * d1;
                            v2[e] = e2 * d2;
                        }
                        pa[h][ar][i] = pack_p<F16>(va[0], va[1]);
                        p1[h][ar][i] = pack_p<F16>(v1[0], v1[1]);
                        p2[h][ar][i] = pack_p<F16>(v2[0], v2[1]);
                    }
        };
        if (full) elementwise(std::false_type{});
        else elementwise(std::true_type{});

        // the previous step's products have read the tiles this step overwrites
        if (t > 0) ok = mbar_wait_warp(&bars->p_empty, (t - 1) & 1, abort_flag, p.err, 0xF2);
        if (!ok) break;
        // A^T and dS1^T go to TMEM with the 16x128b shape: register 2i + a of the store at
        // lane offset 16h is lane 16h + 8a + tr, column 4i + tc of the group's 16 (queries
        // 8i + 2tc, +1 as one pair), which is exactly where this thread's pair belongs.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t lb = lane_base + ((uint32_t)(16 * h) << 16) + g * (kHQ / 2);
            const uint32_t ra[8] = {pa[h][0][0], pa[h][1][0], pa[h][0][1], pa[h][1][1],
                                    pa[h][0][2], pa[h][1][2], pa[h][0][3], pa[h][1][3]};
            const uint32_t r1[8] = {p1[h][0][0], p1[h][1][0], p1[h][0][1], p1[h][1][1],
                                    p1[h][0][2], p1[h][1][2], p1[h][0][3], p1[h][1][3]};
            tmem_st_16x128b_x4(lb + kColPA, ra);
            tmem_st_16x128b_x4(lb + kColP1, r1);
        }
        // dS2^T to shared memory: per store instruction the warp writes 8 rows x 16 bytes
        // into 8 distinct chunk positions ((4g + i) ^ tr): one wavefront, no bank conflict.
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int ar = 0; ar < 2; ++ar)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t off = (uint32_t)((16 * h + 8 * ar) * 128 + (((4 * g + i) ^ tr) << 4));
                    sts_u32(pbase + off, p2[h][ar][i]);
                }
        tmem_st_wait();
        fence_proxy_async_shared();  // the tensor core reads the tile through the async proxy
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full);
    }
    // ---------------------------------------------------------------- epilogue: dV, dK rows
    // Group 0 writes dV columns 0..63 and dK1, group 1 dV columns 64..127 and dK2, read from
    // TMEM with the 16x256b shape and stored straight from registers: per instruction a warp
    // writes 8 rows x 32 contiguous bytes, whole 32-byte sectors (faster than staging the
    // rows for TMA stores, whose drain the CTA has to wait for before it exits).
    if (ok && nsteps > 0) ok = mbar_wait_warp(&bars->acc_done, 0, abort_flag, p.err, 0xF1);
    tc_fence_after();
    {
        const float scale = p.scale;
        const int64_t row0 = ((int64_t)b * p.H + h) * p.N;
        float* dkbase = g ? p.dk2 : p.dk1;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            uint32_t v[2][16], k[2][16];
            if (ok) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t lb = lane_base + ((uint32_t)(16 * hh) << 16) + c * 32;
                    tmem_ld_16x256b_x4(lb + kColV + g * 64, v[hh]);
                    tmem_ld_16x256b_x4(lb + (g ? kColK2 : kColK1), k[hh]);
                }
                tmem_ld_wait();
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int ar = 0; ar < 2; ++ar) {
                    const int key = k0 + lg * 32 + 16 * hh + 8 * ar + tr;
                    if (!ok || key >= p.N) continue;
                    float* dvr = p.dv + (row0 + key) * kDV + g * 64 + c * 32 + 2 * tc;
                    float* dkr = dkbase + (row0 + key) * kD + c * 32 + 2 * tc;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int rg = 4 * i + 2 * ar;
                        *reinterpret_cast<float2*>(dvr + 8 * i) =
                            make_float2(__uint_as_float(v[hh][rg]), __uint_as_float(v[hh][rg + 1]));
                        *reinterpret_cast<float2*>(dkr + 8 * i) =
                            make_float2(__uint_as_float(k[hh][rg]) * scale, __uint_as_float(k[hh][rg + 1]) * scale);
                    }
                }
        }
    }
    tc_fence_before();
    named_bar_sync(2, kThreads);
}

template <typename K>
cudaError_t setup(K kernel, size_t smem) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

}  // namespace

bool bwd_tc_supported(int d, int Dv, int in_dtype) { return d == kD && Dv == kDV && (in_dtype == 1 || in_dtype == 2); }

cudaError_t launch_bwd_tc(const BwdTcParams& p, cudaStream_t key_stream, cudaStream_t query_stream) {
    if (p.d != kD || p.Dv != kDV) return cudaErrorInvalidValue;
    const bool f16 = p.in_f16 != 0;
    cudaError_t e;
    if (f16) {
        if ((e = prepare_once<bwd_dkdv_kernel<true>>((int)dkdv::kSmem, kRegsLaunch)) != cudaSuccess ||
            (e = prepare_once<bwd_dq_kernel<true>>((int)dq::kSmem, kRegsLaunch)) != cudaSuccess)
            return e;
    } else {
        if ((e = prepare_once<bwd_dkdv_kernel<false>>((int)dkdv::kSmem, kRegsLaunch)) != cudaSuccess ||
            (e = prepare_once<bwd_dq_kernel<false>>((int)dq::kSmem, kRegsLaunch)) != cudaSuccess)
            return e;
    }
    const int n_tiles = (p.N + BM - 1) / BM;
    const int grid = n_tiles * p.B * p.H;
    // The key side follows the preparation in its stream as a programmatic dependent launch:
    // its CTAs may start while the preparation's last CTAs run, and its producer waits for
    // the preparation (griddepcontrol.wait) before loading dO and the statistics.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = dkdv::kSmem;
    cfg.stream = key_stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (f16) {
        if ((e = cudaLaunchKernelEx(&cfg, bwd_dkdv_kernel<true>, p)) != cudaSuccess) return e;
        bwd_dq_kernel<true><<<grid, kThreads, dq::kSmem, query_stream>>>(p);
    } else {
        if ((e = cudaLaunchKernelEx(&cfg, bwd_dkdv_kernel<false>, p)) != cudaSuccess) return e;
        bwd_dq_kernel<false><<<grid, kThreads, dq::kSmem, query_stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace da
