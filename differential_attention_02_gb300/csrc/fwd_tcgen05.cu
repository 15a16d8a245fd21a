// Fused causal prefill of differential attention on the 5th-generation
// tensor cores (tcgen05.mma with TMEM accumulators), fed by TMA.
//
// What it computes, per head: (softmax(Q1K1^T/sqrt d) - lambda
// softmax(Q2K2^T/sqrt d)) V — the DiffAttn formula of "Differential
// Transformer: Transformer que cancela ruído de atenção" (section "Como a
// atenção diferencial funciona") under the causal mask of the intoai.pub page
// ("A Deeper Dive Into Attention Calculations") — then each head's RMSNorm
// and the (1 - lambda_init) scale (section "Estrutura multi-head e
// arquitetura completa"). The output is written [B, N, H, Dv].
//
// The two maps only meet in the epilogue: map m keeps its own running max and
// sum and its own accumulator O_m = sum_j exp(S_m - max_m) V_j, and the
// epilogue forms O1/l1 - lambda O2/l2. (The pages' remark that FlashAttention
// can be reused is prior art only; nothing of it is followed here.)
//
// CTA = one 128-row query tile of one (b, h); 12 warps:
//   warp 8       TMA producer: Q1, Q2 once, then a 3-stage ring of (K1, K2, V)
//                tiles of 128 keys, all 128-byte swizzled.
//   warp 9       allocates 512 TMEM columns; the warp walks the MMA loop
//                converged and one elected lane issues every MMA:
//                S1 = Q1 K1^T, S2 = Q2 K2^T (fp32 in TMEM), O1 += P1 V,
//                O2 += P2 V (P read from TMEM, V from shared memory, fp32 O
//                in TMEM).
//   warps 0..3   softmax of map 1; warps 4..7 softmax of map 2 (warp w reads
//                TMEM lanes 32*(w%4)..+31). Thread r of a
//                group owns query row r (TMEM lane r): it reads its S row,
//                updates max and sum, writes its P row as bf16 back into the
//                first half of its S columns, and rescales its O row in TMEM
//                only when the running max grew by more than 2^8 (the stale
//                max is exact because the final division uses the same max).
// Keeping P in TMEM halves the shared-memory traffic of the PV products (only
// V is read from shared memory), which otherwise bounds the tensor pipe.
//   epilogue     both softmax groups: O1/l1 - lambda O2/l2, row RMSNorm,
//                (1 - lambda_init), norm weight, store.
// The MMA order PV1(j), S1(j+1), PV2(j), S2(j+1) lets one group's softmax run
// while the tensor core works for the other map. S_m(j+1) overwrites the TMEM
// columns PV_m(j) reads P from; tcgen05.mma operations issued by one thread
// execute in issue order, so the read completes before the overwrite.
//
// Two launch forms share these roles. The per-tile kernel (one CTA per query
// tile) serves long sequences, fp32 output and the backward preparation. The
// persistent kernel (one CTA per SM walking a list of query tiles) serves
// 16-bit output of short sequences, where each CTA's start and tail (first
// loads and scores, epilogue, store, the next CTA's launch) are a large share
// of a tile's time: it overlaps them with the neighbouring tiles' work.
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

constexpr int BM = kFwdBM, BN = kFwdBN;
// Warps 0..3: softmax of map 1, 4..7: softmax of map 2 (warp w reads TMEM lanes
// 32*(w%4)..+31), 8: TMA producer, 9: TMEM owner and MMA issuer, 10..11: idle
// (they complete the third warpgroup, which register reallocation works on).
constexpr int kThreads = 12 * 32;
constexpr int kWarpProducer = 8, kWarpMma = 9;
// Register split: the softmax warpgroups grow to kRegsSoftmax, the third
// warpgroup shrinks to kRegsOther. The launch provides kRegsLaunch per thread;
// 2*128*kRegsSoftmax + 128*kRegsOther must not exceed 384*kRegsLaunch, or the
// increase would wait forever. The launcher checks the compiled count.
constexpr int kRegsLaunch = 168, kRegsSoftmax = 224, kRegsOther = 56;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsOther <= kThreads * kRegsLaunch, "register split");
constexpr int kKvStages = 3;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D, int DV>
struct FwdCfg {
    static constexpr int kQBytes = BM * D * 2;       // one Q half tile
    static constexpr int kKBytes = BN * D * 2;       // one K half tile
    static constexpr int kVBytes = BN * DV * 2;
    static constexpr int kBoxBytes = 128 * 128;      // one [128 rows][64 bf16] box
    static constexpr int kStageBytes = 2 * kKBytes + kVBytes;
    static constexpr int kOffQ1 = 0;
    static constexpr int kOffQ2 = kQBytes;
    static constexpr int kOffStages = 2 * kQBytes;
    static constexpr int kOffBar = kOffStages + kKvStages * kStageBytes;
    static constexpr int kBarBytes = 256;
    // The epilogue's exchange buffer (4 x 128 floats) reuses the Q1 tile, which
    // is idle once the last MMA has completed.
    static constexpr int kOffEpi = kOffQ1;
    static_assert(8 * BM * 4 <= kQBytes, "epilogue buffer fits in the Q1 tile");
    static_assert(BM * DV * 4 <= kStageBytes && BM * DV * 2 <= kStageBytes, "gain-gradient terms and dy fit a stage");
    static constexpr size_t kSmem = 1024 + (size_t)kOffBar + kBarBytes;
    static_assert(kSmem <= 232448, "shared memory budget");
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;               // S1 at 0, S2 at BN; P_m in the first BN/2 columns of S_m
    static constexpr uint32_t kColO = 2 * BN;          // O1 at 2BN, O2 at 2BN + DV
    static_assert(2 * BN + 2 * DV <= 512, "TMEM budget");
};

struct Bars {
    uint64_t q_full;
    uint64_t kv_full[kKvStages];
    uint64_t kv_empty[kKvStages];
    uint64_t s_full[2];
    uint64_t p_half[2];  // P of keys 0..BN/2-1 is in TMEM
    uint64_t p_full[2];
    uint64_t o_done[2];
    uint64_t drain;
    uint64_t dy_full;  // backward preparation: this tile's dy rows in shared memory
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= FwdCfg<64, 128>::kBarBytes, "barrier block fits its reserve");

// The MMA issuer shares its SM sub-partition with two softmax warps, so each
// MMA costs as few instructions as possible: descriptors are built once and
// advanced by adding the (16-byte-unit) start-address offset to the low word.
template <int D, bool F16>
__device__ __forceinline__ void issue_qk(uint32_t s_tmem, uint64_t q_desc, uint64_t k_desc) {
    constexpr uint32_t idesc = idesc_kind_f16(BM, BN, 0, 0, F16);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = (uint64_t)(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
        umma_ss(s_tmem, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u);
    }
}

// O (+)= P V with P in TMEM: lane r holds row r, 16 keys (bf16 pairs) per 8 columns.
// V tile descriptor: boxes of [BN keys][64 columns]; the next 64 columns are the
// next box (leading offset), the next 8 keys +1024 bytes (stride offset), so one
// K=16 step advances 2048 bytes (128 in 16-byte units).
template <int DV, bool F16>
__device__ __forceinline__ void issue_pv_half(uint32_t o_tmem, uint32_t p_tmem, uint64_t v_desc, int half,
                                              uint32_t accumulate) {
    constexpr uint32_t idesc = idesc_kind_f16(BM, DV, 0, 1, F16);
#pragma unroll
    for (int k = 0; k < BN / 32; ++k) {
        const int kk = half * (BN / 32) + k;
        umma_ts(o_tmem, p_tmem + kk * 8, v_desc + (uint64_t)(kk * 128), idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
}

// One key tile of map g's online softmax, by the group's four warps (thread =
// query row = TMEM lane): waits for the scores, masks keys past the causal
// diagonal or past N, updates the running max (O is rescaled in TMEM only when
// the max grew by more than the threshold; the stale max is exact because the
// final division uses the same max), and writes P = exp2(S * scale - max) as
// 16-bit pairs (lower key in the low half) into the first BN/2 columns of S,
// row sum in fp32. The first half of the keys is handed to the MMA warp before
// the second half is exponentiated, so the first half of PV overlaps the rest.
// `ph` is the parity of this tile's phase of the map's barriers. Returns false
// if a wait gave up.
template <int DV, bool F16>
__device__ __forceinline__ bool softmax_tile(const FwdParams& p, int g, uint64_t* s_full, uint64_t* o_done,
                                             uint64_t* p_half, uint64_t* p_full, volatile int* abort_flag,
                                             uint32_t tS, uint32_t tO, int q0, int qrow, int kbase, bool first,
                                             uint32_t ph, float& m_used, float& l) {
    const int lane = threadIdx.x & 31;
    const float sl2 = p.scale_log2;
    if (!mbar_wait_warp(s_full, ph, abort_flag, p.err, 0x40 + g)) return false;
    tc_fence_after();
    uint32_t sr[BN];
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS + c * 32, sr + c * 32);
    tmem_ld_wait();

    const bool need_mask = (p.causal && kbase + BN - 1 > q0) || (kbase + BN > p.N);
    if (need_mask) {
        const int lim = p.causal ? min(qrow + 1, p.N) : p.N;  // visible keys: kbase + i < lim
#pragma unroll
        for (int i = 0; i < BN; ++i)
            if (kbase + i >= lim) sr[i] = __float_as_uint(-INFINITY);
    }
    float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
    for (int i = 0; i < BN; i += 8) {
        mx0 = fmax3(mx0, __uint_as_float(sr[i]), __uint_as_float(sr[i + 1]));
        mx1 = fmax3(mx1, __uint_as_float(sr[i + 2]), __uint_as_float(sr[i + 3]));
        mx2 = fmax3(mx2, __uint_as_float(sr[i + 4]), __uint_as_float(sr[i + 5]));
        mx3 = fmax3(mx3, __uint_as_float(sr[i + 6]), __uint_as_float(sr[i + 7]));
    }
    const float m_new = fmax3(fmaxf(mx0, mx1), mx2, mx3) * sl2;
    float alpha = 1.f;
    bool rescale = false;
    if (first) {
        m_used = m_new;
    } else if (m_new > m_used + kRescaleThreshold) {
        alpha = fast_exp2(m_used - m_new);
        m_used = m_new;
        rescale = true;
    }
    // O must hold the previous tile's PV before it is rescaled; S landing already
    // implies that (MMAs complete in issue order), so this wait returns at once.
    if (!first && __any_sync(0xffffffffu, rescale)) {
        if (!mbar_wait_warp(o_done, ph ^ 1u, abort_flag, p.err, 0x42 + g)) return false;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < DV / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + c * 32, o);
        }
    }
    float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        uint32_t pk[BN / 4];
#pragma unroll
        for (int i = 0; i < BN / 2; i += 2) {
            const int k = hf * (BN / 2) + i;
            const float e0 = fast_exp2(fmaf(__uint_as_float(sr[k]), sl2, -m_used));
            const float e1 = fast_exp2(fmaf(__uint_as_float(sr[k + 1]), sl2, -m_used));
            rs[(i >> 1) & 3] += e0 + e1;
            pk[i / 2] = pack_p<F16>(e0, e1);
        }
        tmem_st32(tS + hf * (BN / 4), pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(hf == 0 ? p_half : p_full);
    }
    l = l * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
    return true;
}

// Epilogue of the backward preparation (PREP): instead of storing y, the two
// softmax groups derive, per query row, what the tensor-core backward consumes.
// With n = O/r, r = sqrt(mean(O^2) + eps), c = 1 - lambda_init, g = dy w c:
//   dO = (g - n mean(g n)) / r          (gradient of the pre-norm output O)
//   D1 = dO . (P1 V),  D2 = -lambda dO . (P2 V)
//   L_m = max_m + log2(l_m)             (so that P_m = exp2(S_m log2(e)/sqrt(d) - L_m))
// and, summed over the CTA's rows in a fixed order, dlambda = -sum dO . (P2 V)
// and the gain's gradient sum_rows dy n c. Group g handles output columns
// [g Dv/2, (g+1) Dv/2); row sums cross between the groups through `xch`.
template <int DV, bool F16>
__device__ __forceinline__ void prep_epilogue(const FwdParams& p, bool ok, int g, int r, int qrow, int b, int h,
                                              uint32_t lane_base, uint32_t col_o, float l, float m_used, float* xch,
                                              const uint8_t* dybuf, float* dwbuf, float* dlbuf) {
    constexpr int kHalf = DV / 2;
    using T16 = typename std::conditional<F16, __half, __nv_bfloat16>::type;
    const bool live = ok && qrow < p.N;
    // Row statistics of both maps.
    xch[g * BM + r] = l;
    xch[(2 + g) * BM + r] = m_used;
    named_bar_sync(1, 256);
    const float l1 = xch[r], l2 = xch[BM + r], mx1 = xch[2 * BM + r], mx2 = xch[3 * BM + r];
    const float i1 = 1.0f / l1, i2 = 1.0f / l2, lam = p.lambda, cs = 1.0f - p.lambda_init;
    const uint32_t t1 = lane_base + col_o + g * kHalf, t2 = lane_base + col_o + DV + g * kHalf;
    // This row's slice of dy (kHalf 16-bit values) in fp32, from the tile the producer
    // staged: box g of [128 rows][64 values], 128-byte swizzled (rows past N are zeros).
    float dyv[kHalf];
    static_assert(kHalf == 64, "one 64-column box per group");
    if (ok) {
#pragma unroll
        for (int c = 0; c < kHalf / 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(dybuf + g * (128 * 128) + sw128_offset(r, c));
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if constexpr (F16) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
                    dyv[c * 8 + 2 * e] = f.x;
                    dyv[c * 8 + 2 * e + 1] = f.y;
                } else {
                    dyv[c * 8 + 2 * e] = bf16lo_to_f32(w4[e]);
                    dyv[c * 8 + 2 * e + 1] = bf16hi_to_f32(w4[e]);
                }
            }
        }
    } else {
#pragma unroll
        for (int c = 0; c < kHalf; ++c) dyv[c] = 0.f;
    }
    // Pass 1: sum of squares of O over the row.
    float ss = 0.f;
    if (ok) {
#pragma unroll
        for (int c = 0; c < kHalf / 32; ++c) {
            uint32_t a[32], e[32];
            tmem_ld32(t1 + c * 32, a);
            tmem_ld32(t2 + c * 32, e);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float x = __uint_as_float(a[i]) * i1 - lam * (__uint_as_float(e[i]) * i2);
                ss = fmaf(x, x, ss);
            }
        }
    }
    xch[(4 + g) * BM + r] = ss;
    named_bar_sync(1, 256);
    const float ir = 1.0f / sqrtf((xch[4 * BM + r] + xch[5 * BM + r]) / (float)DV + p.eps);
    // Pass 2: mean(g n) over the row.
    float gn = 0.f;
    if (ok) {
#pragma unroll
        for (int c = 0; c < kHalf / 32; ++c) {
            uint32_t a[32], e[32];
            tmem_ld32(t1 + c * 32, a);
            tmem_ld32(t2 + c * 32, e);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int col = g * kHalf + c * 32 + i;
                const float n = (__uint_as_float(a[i]) * i1 - lam * (__uint_as_float(e[i]) * i2)) * ir;
                const float gg = dyv[c * 32 + i] * (p.norm_w ? p.norm_w[col] : 1.f) * cs;
                gn = fmaf(gg, n, gn);
            }
        }
    }
    xch[(6 + g) * BM + r] = gn;
    named_bar_sync(1, 256);
    gn = (xch[6 * BM + r] + xch[7 * BM + r]) / (float)DV;
    // Pass 3: dO (stored in the operand type), D1/D2 partials, gain-gradient terms.
    float x1 = 0.f, x2 = 0.f, x2e = 0.f;
    T16* dorow = static_cast<T16*>(p.d_o) + (((int64_t)b * p.H + h) * p.N + qrow) * DV + g * kHalf;
    // [BM][DV] with column c of row r at c ^ (r % 32): row-per-thread writes and
    // column-per-thread reads both hit 32 distinct banks.
    float* dwrow = dwbuf + r * DV;
    const int swz = r & 31;
#pragma unroll
    for (int c = 0; c < kHalf / 32; ++c) {
        uint32_t a[32], e[32];
        if (ok) {
            tmem_ld32(t1 + c * 32, a);
            tmem_ld32(t2 + c * 32, e);
            tmem_ld_wait();
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            float d2[2], o1v[2], o2v[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int col = g * kHalf + c * 32 + i + k;
                const float o1 = ok ? __uint_as_float(a[i + k]) * i1 : 0.f;
                const float o2 = ok ? __uint_as_float(e[i + k]) * i2 : 0.f;
                const float n = (o1 - lam * o2) * ir;
                const float dyc = dyv[c * 32 + i + k];
                const float gg = dyc * (p.norm_w ? p.norm_w[col] : 1.f) * cs;
                d2[k] = (gg - n * gn) * ir;
                o1v[k] = o1;
                o2v[k] = o2;
                dwrow[(g * kHalf + c * 32 + i + k) ^ swz] = live ? dyc * n * cs : 0.f;
            }
            pk[i / 2] = pack_p<F16>(d2[0], d2[1]);
            // D1, D2 from the rounded dO the gradient products will use, so that
            // sum_j P_ij (dA_ij - D_i) stays zero for every row.
            float r0, r1;
            if constexpr (F16) {
                const float2 rr = __half22float2(*reinterpret_cast<const __half2*>(&pk[i / 2]));
                r0 = rr.x;
                r1 = rr.y;
            } else {
                r0 = bf16lo_to_f32(pk[i / 2]);
                r1 = bf16hi_to_f32(pk[i / 2]);
            }
            x1 = fmaf(r0, o1v[0], fmaf(r1, o1v[1], x1));
            x2 = fmaf(r0, o2v[0], fmaf(r1, o2v[1], x2));
            x2e = fmaf(d2[0], o2v[0], fmaf(d2[1], o2v[1], x2e));  // dlambda takes the unrounded dO
        }
        if (live) {
            uint4* dst = reinterpret_cast<uint4*>(dorow + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
    }
    named_bar_sync(1, 256);  // every read of the exchange slots above is done
    xch[g * BM + r] = x1;
    xch[(2 + g) * BM + r] = x2;
    xch[(4 + g) * BM + r] = x2e;
    named_bar_sync(1, 256);
    const float X1 = xch[r] + xch[BM + r], X2 = xch[2 * BM + r] + xch[3 * BM + r];
    const float X2e = xch[4 * BM + r] + xch[5 * BM + r];
    if (g == 0 && live) {
        float4* st = reinterpret_cast<float4*>(p.stats + (((int64_t)b * p.H + h) * p.N + qrow) * 4);
        *st = make_float4(mx1 + __log2f(l1), mx2 + __log2f(l2), X1, -lam * X2);
    }
    if (g == 0) dlbuf[r] = live ? -X2e : 0.f;  // this row's dlambda term
    named_bar_sync(1, 256);
    // Column sums over the CTA's rows in a fixed order: thread t sums column t % DV over
    // rows 64 (t / DV) .. +63, then the two halves are added (256 threads, DV = 128).
    static_assert(2 * DV == 256, "two threads per column");
    const int t = g * BM + r;  // 0..255
    const int col = t % DV, half = t / DV;
    float acc = 0.f;
#pragma unroll 8
    for (int row = half * 64; row < half * 64 + 64; ++row) acc += dwbuf[row * DV + (col ^ (row & 31))];
    float* hsum = xch;  // the exchange slots are free again
    named_bar_sync(1, 256);  // every read of the exchange slots above is done
    if (half == 1) hsum[col] = acc;
    named_bar_sync(1, 256);
    if (half == 0) p.part_w[(int64_t)blockIdx.x * DV + col] = acc + hsum[col];
    // dlambda over the rows: warp 0 (group 0's first warp) adds four rows per lane, then
    // a fixed butterfly.
    if (t < 32) {
        float s4 = ((dlbuf[4 * t] + dlbuf[4 * t + 1]) + dlbuf[4 * t + 2]) + dlbuf[4 * t + 3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s4 += __shfl_xor_sync(0xffffffffu, s4, o);
        if (t == 0) p.part_lam[blockIdx.x] = s4;
    }
}

// What the per-tile kernel's epilogue does: store the output (plain), derive the
// backward's inputs instead (prep), or store the output and save the state the
// backward starts from (save: the unnormalised O1, O2 and each map's max and sum).
constexpr int kModePlain = 0, kModePrep = 1, kModeSave = 2;
// Save mode stages O1, O2 (8 boxes of 16 KB) in the K/V ring after the output's
// staging (at most 64 KB, fp32 output).
constexpr int kSaveStageOff = 64 * 1024;                 // x boxes (4 x 16 KB) of the saved state
constexpr int kSaveA2Off = kSaveStageOff + 4 * 128 * 128;  // O2/l2 boxes (2 x 16 KB)

template <int D, int DV, bool F16, int MODE>
__global__ void __launch_bounds__(kThreads, 1) fwd_bf16_kernel(const __grid_constant__ FwdParams p) {
    using C = FwdCfg<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);
    float* epi = reinterpret_cast<float*>(smem + C::kOffEpi);  // [4][BM]: 1/l1, lambda/l2, ss1, ss2
    volatile int* abort_flag = &bars->abort;
    // As the backward's preparation: the key-side kernel that follows may start its setup
    // and K/V loads once every CTA of this grid has started (it waits for this grid before
    // reading dO and the statistics).
    if constexpr (MODE == kModePrep) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = (p.N + BM - 1) / BM;
    const int BH = p.B * p.H;
    const int qt = n_tiles - 1 - (int)(blockIdx.x / BH);  // heaviest causal tiles first
    const int bh = blockIdx.x % BH;
    const int b = bh / p.H, h = bh % p.H;
    const int q0 = qt * BM;
    const int nkv = p.causal ? min(qt + 1, n_tiles) : n_tiles;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int s = 0; s < kKvStages; ++s) {
            mbar_init(&bars->kv_full[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(&bars->s_full[g], 1);
            mbar_init(&bars->p_half[g], 4);  // one arrival per softmax warp
            mbar_init(&bars->p_full[g], 4);
            mbar_init(&bars->o_done[g], 1);
        }
        mbar_init(&bars->drain, 1);
        mbar_init(&bars->dy_full, 1);
        bars->abort = 0;
        fence_mbarrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&bars->tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    uint8_t* q1s = smem + C::kOffQ1;
    uint8_t* q2s = smem + C::kOffQ2;
    uint8_t* stages = smem + C::kOffStages;

    if (warp >= 8) {
        // Third warpgroup: producer, MMA issuer, two idle warps. Each warpgroup
        // reallocates registers at the top of its own branch, so the compiler
        // applies each limit to that branch's code.
        setmaxnreg_dec<kRegsOther>();
        if (warp == kWarpProducer) {
            // ------------------------------------------------------------ producer
            if (lane == 0) {
                tma_prefetch_desc(&p.tm_q1);
                tma_prefetch_desc(&p.tm_q2);
                tma_prefetch_desc(&p.tm_k1);
                tma_prefetch_desc(&p.tm_k2);
                tma_prefetch_desc(&p.tm_v);
                mbar_arrive_expect_tx(&bars->q_full, 2 * C::kQBytes);
                index_ok(q0 < p.N && h < p.H && b < p.B, p.err, 0x90);
#pragma unroll
                for (int x = 0; x < D / 64; ++x) {
                    tma_load_4d(q1s + x * C::kBoxBytes, &p.tm_q1, &bars->q_full, x * 64, q0, h, b);
                    tma_load_4d(q2s + x * C::kBoxBytes, &p.tm_q2, &bars->q_full, x * 64, q0, h, b);
                }
                int j = 0;
                for (; j < nkv; ++j) {
                    const int s = j % kKvStages;
                    if (!mbar_wait(&bars->kv_empty[s], ((j / kKvStages) & 1) ^ 1, abort_flag, p.err, 0x31)) break;
                    uint8_t* st = stages + s * C::kStageBytes;
                    mbar_arrive_expect_tx(&bars->kv_full[s], C::kStageBytes);
                    index_ok(j * BN < p.N, p.err, 0x91);
#pragma unroll
                    for (int x = 0; x < D / 64; ++x) {
                        tma_load_4d(st + x * C::kBoxBytes, &p.tm_k1, &bars->kv_full[s], x * 64, j * BN, h, b);
                        tma_load_4d(st + C::kKBytes + x * C::kBoxBytes, &p.tm_k2, &bars->kv_full[s], x * 64, j * BN, h,
                                    b);
                    }
#pragma unroll
                    for (int x = 0; x < DV / 64; ++x)
                        tma_load_4d(st + 2 * C::kKBytes + x * C::kBoxBytes, &p.tm_v, &bars->kv_full[s], x * 64, j * BN,
                                    h, b);
                }
                // Backward preparation: this tile's dy rows ([128 rows][DV], boxes of 64 columns)
                // into the stage the ring frees next, so they land during the last tiles' work
                // (the epilogue reads them; out-of-range rows read zeros).
                bool dy_loaded = false;
                if constexpr (MODE == kModePrep) {
                    const int s = nkv % kKvStages;
                    if (j == nkv &&
                        mbar_wait(&bars->kv_empty[s], ((nkv / kKvStages) & 1) ^ 1, abort_flag, p.err, 0x3e)) {
                        mbar_arrive_expect_tx(&bars->dy_full, BM * DV * 2);
#pragma unroll
                        for (int x = 0; x < DV / 64; ++x)
                            tma_load_3d(stages + s * C::kStageBytes + x * C::kBoxBytes, &p.tm_dy, &bars->dy_full,
                                        h * DV + x * 64, q0, b);
                        dy_loaded = true;
                    }
                }
                // Drain: no copy may still be landing in shared memory when the CTA exits.
                mbar_wait(&bars->q_full, 0, nullptr, p.err, 0x32);
                for (int u = max(0, j - kKvStages); u < j; ++u)
                    mbar_wait(&bars->kv_full[u % kKvStages], (u / kKvStages) & 1, nullptr, p.err, 0x33);
                if (dy_loaded) mbar_wait(&bars->dy_full, 0, nullptr, p.err, 0x3f);
            }
        } else if (warp == kWarpMma) {
            // ------------------------------------------------------------ MMA issuer
            // The whole warp walks the loop and waits; one elected lane issues each
            // group of MMAs together with the commits that track them.
            const uint32_t tS[2] = {tmem + C::kColS, tmem + C::kColS + BN};
            const uint32_t tO[2] = {tmem + C::kColO, tmem + C::kColO + DV};
            const uint64_t dq[2] = {sdesc_sw128(smem_u32(q1s), 16, 1024), sdesc_sw128(smem_u32(q2s), 16, 1024)};
            // Stage s descriptors = stage-0 descriptors + s * kStageBytes (in 16-byte units).
            const uint64_t dk0 = sdesc_sw128(smem_u32(stages), 16, 1024);
            const uint64_t dv0 = sdesc_sw128(smem_u32(stages) + 2 * C::kKBytes, BN * 128, 1024);
            constexpr uint64_t kStageStep = C::kStageBytes >> 4;
            constexpr uint64_t kK2Step = C::kKBytes >> 4;
            bool ok = mbar_wait_warp(&bars->q_full, 0, abort_flag, p.err, 0x34) &&
                      mbar_wait_warp(&bars->kv_full[0], 0, abort_flag, p.err, 0x35);
            if (ok) {
                tc_fence_after();
                if (elect_one()) {
                    issue_qk<D, F16>(tS[0], dq[0], dk0);
                    umma_commit(&bars->s_full[0]);
                    issue_qk<D, F16>(tS[1], dq[1], dk0 + kK2Step);
                    umma_commit(&bars->s_full[1]);
                }
                __syncwarp();
            }
            for (int j = 0; ok && j < nkv; ++j) {
                const int s = j % kKvStages;
                const uint64_t dv = dv0 + s * kStageStep;
                const bool more = j + 1 < nkv;
                const int s1 = (j + 1) % kKvStages;
                const uint64_t dk1 = dk0 + s1 * kStageStep;
                // Per map: the first half of PV(j) as soon as the softmax has written the
                // first half of P(j), then the second half and S(j+1).
                for (int m = 0; m < 2; ++m) {
                    if (!mbar_wait_warp(&bars->p_half[m], j & 1, abort_flag, p.err, 0x36 + m)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (elect_one()) issue_pv_half<DV, F16>(tO[m], tS[m], dv, 0, j > 0 ? 1u : 0u);
                    __syncwarp();
                    // The next K/V tile is checked while the softmax still works on the
                    // second half of P, off the path from p_full to the MMAs.
                    if (m == 0 && more &&
                        !mbar_wait_warp(&bars->kv_full[s1], ((j + 1) / kKvStages) & 1, abort_flag, p.err, 0x38)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait_warp(&bars->p_full[m], j & 1, abort_flag, p.err, 0x3b + m)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (elect_one()) {
                        issue_pv_half<DV, F16>(tO[m], tS[m], dv, 1, 1u);
                        umma_commit(&bars->o_done[m]);
                        if (m == 1) umma_commit(&bars->kv_empty[s]);
                        if (more) {
                            issue_qk<D, F16>(tS[m], dq[m], dk1 + m * kK2Step);
                            umma_commit(&bars->s_full[m]);
                        }
                    }
                    __syncwarp();
                }
            }
            // Every MMA issued (also before an abort) must finish before TMEM is freed.
            if (elect_one()) umma_commit(&bars->drain);  // the lane that issued the MMAs
            __syncwarp();
            mbar_wait(&bars->drain, 0, nullptr, p.err, 0x39);
        }
        // ---------------------------------------------------------------- teardown
        tc_fence_before();
        named_bar_sync(2, kThreads);  // every role is done with TMEM and shared memory
        if (warp == kWarpMma) {
            tc_fence_after();
            tmem_dealloc(tmem, C::kTmemCols);
        }
    } else {
        setmaxnreg_inc<kRegsSoftmax>();
        // ------------------------------------------------------------ softmax (map g)
        const int g = warp >> 2;
        const int lg = warp & 3;
        const int r = lg * 32 + lane;  // query row within the tile == TMEM lane
        const int qrow = q0 + r;
        const uint32_t lane_base = tmem + ((uint32_t)(lg * 32) << 16);
        const uint32_t tS = lane_base + C::kColS + g * BN;
        const uint32_t tO = lane_base + C::kColO + g * DV;
        const float sl2 = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;

        for (int j = 0; j < nkv; ++j) {
            if (!mbar_wait_warp(&bars->s_full[g], j & 1, abort_flag, p.err, 0x40 + g)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS + c * 32, sr + c * 32);
            tmem_ld_wait();

            const int kbase = j * BN;
            const bool need_mask = (p.causal && kbase + BN - 1 > q0) || (kbase + BN > p.N);
            if (need_mask) {
                const int lim = p.causal ? min(qrow + 1, p.N) : p.N;  // visible keys: kbase + i < lim
#pragma unroll
                for (int i = 0; i < BN; ++i)
                    if (kbase + i >= lim) sr[i] = __float_as_uint(-INFINITY);
            }
            float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
            for (int i = 0; i < BN; i += 8) {
                mx0 = fmax3(mx0, __uint_as_float(sr[i]), __uint_as_float(sr[i + 1]));
                mx1 = fmax3(mx1, __uint_as_float(sr[i + 2]), __uint_as_float(sr[i + 3]));
                mx2 = fmax3(mx2, __uint_as_float(sr[i + 4]), __uint_as_float(sr[i + 5]));
                mx3 = fmax3(mx3, __uint_as_float(sr[i + 6]), __uint_as_float(sr[i + 7]));
            }
            const float m_new = fmax3(fmaxf(mx0, mx1), mx2, mx3) * sl2;
            float alpha = 1.f;
            bool rescale = false;
            if (j == 0) {
                m_used = m_new;
            } else if (m_new > m_used + kRescaleThreshold) {
                alpha = fast_exp2(m_used - m_new);
                m_used = m_new;
                rescale = true;
            }
            // O must hold PV(j-1) before it is rescaled; S(j) landing already implies
            // that (MMAs complete in issue order), so this wait returns at once.
            if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                if (!mbar_wait_warp(&bars->o_done[g], (j - 1) & 1, abort_flag, p.err, 0x42 + g)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < DV / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + c * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(tO + c * 32, o);
                }
            }
            // P = exp2(S * scale - max) as 16-bit pairs (lower key in the low half) into
            // the first BN/2 columns of S, row sum in fp32. The first half of the keys is
            // handed to the MMA warp before the second half is exponentiated, so the
            // first half of PV(j) overlaps the rest of the softmax.
            float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t pk[BN / 4];
#pragma unroll
                for (int i = 0; i < BN / 2; i += 2) {
                    const int k = hf * (BN / 2) + i;
                    const float e0 = fast_exp2(fmaf(__uint_as_float(sr[k]), sl2, -m_used));
                    const float e1 = fast_exp2(fmaf(__uint_as_float(sr[k + 1]), sl2, -m_used));
                    rs[(i >> 1) & 3] += e0 + e1;
                    pk[i / 2] = pack_p<F16>(e0, e1);
                }
                tmem_st32(tS + hf * (BN / 4), pk);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(hf == 0 ? &bars->p_half[g] : &bars->p_full[g]);
            }
            l = l * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
        }

        // ------------------------------------------------------------ epilogue
        if (ok && nkv > 0) {
            ok = mbar_wait_warp(&bars->o_done[0], (nkv - 1) & 1, abort_flag, p.err, 0x44) &&
                 mbar_wait_warp(&bars->o_done[1], (nkv - 1) & 1, abort_flag, p.err, 0x45);
        }
        tc_fence_after();
        named_bar_sync(1, 256);  // both groups past their last PV: the Q1 tile is free
        if constexpr (MODE == kModePrep) {
            // The exchange slots take 8 x BM floats of the Q1 tile; the gain-gradient
            // terms [BM][DV + 1] take the idle K/V ring.
            // dy is in stage nkv % 3 (the producer's last load); the gain-gradient terms take the
            // next stage and the dlambda terms the idle Q2 tile.
            const int sdy = nkv % kKvStages;
            const bool dy_ok = ok && mbar_wait_warp(&bars->dy_full, 0, abort_flag, p.err, 0x47);
            prep_epilogue<DV, F16>(p, dy_ok, g, r, qrow, b, h, lane_base, C::kColO, l, m_used, epi,
                                   stages + sdy * C::kStageBytes,
                                   reinterpret_cast<float*>(stages + ((sdy + 1) % kKvStages) * C::kStageBytes),
                                   reinterpret_cast<float*>(q2s));
            tc_fence_before();
            named_bar_sync(2, kThreads);
            return;
        }
        epi[g * BM + r] = (g == 0) ? 1.0f / l : p.lambda / l;
        named_bar_sync(1, 256);
        const float inv1 = epi[r], inv2 = epi[BM + r];
        constexpr int kHalf = DV / 2;  // columns handled by this group
        float oh[kHalf];
        float ss = 0.f;
        if (ok) {
#pragma unroll
            for (int c = 0; c < kHalf / 32; ++c) {
                uint32_t o1[32], o2[32];
                tmem_ld32(lane_base + C::kColO + g * kHalf + c * 32, o1);
                tmem_ld32(lane_base + C::kColO + DV + g * kHalf + c * 32, o2);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float x = __uint_as_float(o1[i]) * inv1 - __uint_as_float(o2[i]) * inv2;
                    oh[c * 32 + i] = x;
                    ss = fmaf(x, x, ss);
                }
                if constexpr (MODE == kModeSave) {
                    // x = O1/l1 - lambda O2/l2 (the output before the norm, fp32), this group's
                    // columns, staged for TMA stores behind the output's staging in the idle K/V
                    // ring as boxes of [128 rows][32 fp32]: box j (columns 32 j..) at j * 16 KB.
                    static_assert(kSaveA2Off + 2 * BM * 128 <= kKvStages * C::kStageBytes, "staging fits");
                    uint8_t* box = smem + C::kOffStages + kSaveStageOff + (g * (kHalf / 32) + c) * (BM * 128);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<float4*>(box + sw128_offset(r, i)) =
                            make_float4(oh[c * 32 + 4 * i], oh[c * 32 + 4 * i + 1], oh[c * 32 + 4 * i + 2],
                                        oh[c * 32 + 4 * i + 3]);
                }
            }
        }
        if constexpr (MODE == kModeSave) {
            // Map 2's own output O2 / l2 (its attention output), rounded to the operand type, by
            // group 1 (which holds l2), staged behind the x boxes as boxes of [128 rows][64
            // 16-bit values]; then the row's log-sum-exp of map g in base 2 of the scaled
            // scores, L_g = max_g + log2(l_g).
            if (ok && g == 1) {
                const float inv = 1.0f / l;
#pragma unroll
                for (int c = 0; c < DV / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(lane_base + C::kColO + DV + c * 32, o);
                    tmem_ld_wait();
                    uint8_t* box = smem + C::kOffStages + kSaveA2Off + (c / 2) * (BM * 128);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            pk[e] = pack_p<F16>(__uint_as_float(o[8 * i + 2 * e]) * inv,
                                                __uint_as_float(o[8 * i + 2 * e + 1]) * inv);
                        *reinterpret_cast<uint4*>(box + sw128_offset(r, (c % 2) * 4 + i)) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
            }
            if (ok && qrow < p.N) p.lse_save[(((int64_t)b * p.H + h) * p.N + qrow) * 2 + g] = m_used + log2f(l);
        }
        epi[(2 + g) * BM + r] = ss;
        named_bar_sync(1, 256);
        // Stage this group's DV/2 output columns in shared memory as 128-byte-swizzled
        // boxes of 128 rows (row-per-thread writes hit distinct banks) and write the
        // tile with TMA stores, which clip the rows past N. Row-per-thread global
        // stores would touch one 4 KB-strided row per lane and cost ~3.5K cycles a
        // tile. The K/V ring is idle after the last PV.
        uint8_t* stage = smem + C::kOffStages;
        if (ok) {
            const float tot = epi[2 * BM + r] + epi[3 * BM + r];
            const float rsc = (1.0f - p.lambda_init) / sqrtf(tot / (float)DV + p.eps);
            const float* w = p.norm_w ? p.norm_w + g * kHalf : nullptr;
            if (p.out_bf16 || p.out_f16) {
                const bool f16 = p.out_f16 != 0;
#pragma unroll
                for (int bx = 0; bx < kHalf / 64; ++bx) {
                    uint8_t* box = stage + (g * (kHalf / 64) + bx) * (BM * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int i = bx * 64 + c * 8 + e;
                            y[e] = oh[i] * rsc * (w ? w[i] : 1.f);
                        }
                        *reinterpret_cast<uint4*>(box + sw128_offset(r, c)) =
                            make_uint4(pack_16x2(y[0], y[1], f16), pack_16x2(y[2], y[3], f16),
                                       pack_16x2(y[4], y[5], f16), pack_16x2(y[6], y[7], f16));
                    }
                }
            } else {
#pragma unroll
                for (int bx = 0; bx < kHalf / 32; ++bx) {
                    uint8_t* box = stage + (g * (kHalf / 32) + bx) * (BM * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        float y[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = bx * 32 + c * 4 + e;
                            y[e] = oh[i] * rsc * (w ? w[i] : 1.f);
                        }
                        *reinterpret_cast<float4*>(box + sw128_offset(r, c)) = make_float4(y[0], y[1], y[2], y[3]);
                    }
                }
            }
        }
        fence_proxy_async_shared();
        named_bar_sync(1, 256);
        if (threadIdx.x == 0 && !*abort_flag) {
            const int bw = p.out_bf16 || p.out_f16 ? 64 : 32;  // elements per 128-byte box row
            index_ok(q0 < p.N, p.err, 0x92);
            for (int i = 0; i < DV / bw; ++i) tma_store_3d(&p.tm_out, stage + i * (BM * 128), h * DV + i * bw, q0, b);
            if constexpr (MODE == kModeSave) {
                // x (fp32) and O2/l2 (16-bit) of the tile: rows [q0, q0 + 128) of head (b, h);
                // rows past N are clipped.
                static_assert(DV == 128, "four 32-column fp32 boxes, two 64-column 16-bit boxes");
                for (int jb = 0; jb < 4; ++jb)
                    tma_store_3d(&p.tm_xsave, stage + kSaveStageOff + jb * (BM * 128), jb * 32, q0, b * p.H + h);
                for (int jb = 0; jb < 2; ++jb)
                    tma_store_3d(&p.tm_a2save, stage + kSaveA2Off + jb * (BM * 128), jb * 64, q0, b * p.H + h);
            }
            tma_store_commit();
            tma_store_wait_read();
        }
        tc_fence_before();
        named_bar_sync(2, kThreads);  // releases the MMA warp to free TMEM
    }
}

template <int D, int DV, bool F16, int MODE>
cudaError_t launch_t(const FwdParams& p, cudaStream_t stream) {
    using C = FwdCfg<D, DV>;
    auto k = fwd_bf16_kernel<D, DV, F16, MODE>;
    // The register split assumes the compiled per-thread count (see kRegsLaunch).
    cudaError_t e = prepare_once<fwd_bf16_kernel<D, DV, F16, MODE>>((int)C::kSmem, kRegsLaunch);
    if (e != cudaSuccess) return e;
    const int n_tiles = (p.N + BM - 1) / BM;
    k<<<n_tiles * p.B * p.H, kThreads, C::kSmem, stream>>>(p);
    return cudaGetLastError();
}

// Persistent form, 16-bit output. One CTA per SM walks a static list of query
// tiles (heaviest causal tiles first, dealt to the CTAs round by round in a
// snake order: c, then G-1-c, ...), with the per-tile kernel's warp roles,
// shared-memory ring and inner loops. What it saves is the start and the tail
// of every tile: the next tile's Q tiles and first K/V stages load during the
// current tile's last key tiles, its first score tiles are computed as soon as
// the current tile's last PV products have consumed P (so they are ready when
// the epilogue ends), the output tile's store drains while the next tile runs,
// and there is no CTA launch, barrier setup or TMEM allocation between tiles.
//
// The epilogue stages the output tile in the ring stage that held the tile's
// last (K1, K2, V) tiles. The producer, before it refills that stage, issues
// the tile's TMA store from it and waits until the store has read it.
constexpr int kPStages = 3;
// Dispatch: the persistent form runs when a query tile has at most this many key
// tiles on average (measured on B*H*N = 2^17 rows: 14%, 9% and 7% faster than the
// per-tile kernel at N = 512, 1024, 2048 causal, even at 4096, 5% slower at 8192).
constexpr double kPersistMaxMeanKv = 12.0;

template <int D, int DV>
struct PersistCfg {
    static constexpr int kQBytes = BM * D * 2;
    static constexpr int kKBytes = BN * D * 2;
    static constexpr int kVBytes = BN * DV * 2;
    static constexpr int kBoxBytes = 128 * 128;
    static constexpr int kStageBytes = 2 * kKBytes + kVBytes;
    static constexpr int kOffQ1 = 0;
    static constexpr int kOffQ2 = kQBytes;
    static constexpr int kOffStages = 2 * kQBytes;
    static constexpr int kOffX = kOffStages + kPStages * kStageBytes;  // [2][BM] floats
    static constexpr int kOffBar = kOffX + 2 * BM * 4;
    static constexpr int kBarBytes = 256;
    static constexpr size_t kSmem = 1024 + (size_t)kOffBar + kBarBytes;
    static_assert(kSmem <= 232448, "shared memory budget");
    static_assert(BM * DV * 2 <= kStageBytes, "a 16-bit output tile fits a stage");
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColO = 2 * BN;
    static_assert(2 * BN + 2 * DV <= 512, "TMEM budget");
};

struct PersistBars {
    uint64_t q_full, q_empty;
    uint64_t kv_full[kPStages], kv_empty[kPStages];
    uint64_t out_full[kPStages];  // a query tile's output is staged in this stage
    uint64_t s_full[2], p_half[2], p_full[2], o_done[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(PersistBars) <= PersistCfg<64, 128>::kBarBytes, "barrier block fits its reserve");

struct QTile {
    int q0, b, h, nkv;
};

template <int D, int DV, bool F16>
__global__ void __launch_bounds__(kThreads, 1) fwd_persist_kernel(const __grid_constant__ FwdParams p) {
    using C = PersistCfg<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PersistBars* bars = reinterpret_cast<PersistBars*>(smem + C::kOffBar);
    float* xch = reinterpret_cast<float*>(smem + C::kOffX);
    volatile int* abort_flag = &bars->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = (p.N + BM - 1) / BM;
    const int BH = p.B * p.H;
    const int total = n_tiles * BH;
    const int G = (int)gridDim.x, cta = (int)blockIdx.x;
    // k-th query tile of this CTA, or -1.
    auto tile_at = [&](int k) -> int {
        const int i = k * G + ((k & 1) ? (G - 1 - cta) : cta);
        return i < total ? i : -1;
    };
    auto decode = [&](int i) -> QTile {
        const int qt = n_tiles - 1 - i / BH;
        const int bh = i % BH;
        return QTile{qt * BM, bh / p.H, bh % p.H, p.causal ? min(qt + 1, n_tiles) : n_tiles};
    };

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(&bars->kv_full[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
            mbar_init(&bars->out_full[s], 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(&bars->s_full[g], 1);
            mbar_init(&bars->p_half[g], 4);  // one arrival per softmax warp
            mbar_init(&bars->p_full[g], 4);
            mbar_init(&bars->o_done[g], 1);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbarrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&bars->tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    uint8_t* q1s = smem + C::kOffQ1;
    uint8_t* q2s = smem + C::kOffQ2;
    uint8_t* stages = smem + C::kOffStages;

    if (warp >= 8) {
        setmaxnreg_dec<kRegsOther>();
        if (warp == kWarpProducer) {
            // ------------------------------------------------------------ producer
            if (lane == 0) {
                tma_prefetch_desc(&p.tm_q1);
                tma_prefetch_desc(&p.tm_q2);
                tma_prefetch_desc(&p.tm_k1);
                tma_prefetch_desc(&p.tm_k2);
                tma_prefetch_desc(&p.tm_v);
                tma_prefetch_desc(&p.tm_out);
                int it = 0, nq = 0;                 // stages filled, Q tiles loaded
                int pend[kPStages];                 // query tile whose output is staged in stage s, or -1
                for (int s = 0; s < kPStages; ++s) pend[s] = -1;
                uint32_t oph = 0;                   // parity of each stage's next out_full phase
                bool go = true;
                // Writes the output tile staged in stage s (if any) and waits until the
                // store has read it, so that the stage can be refilled.
                auto flush = [&](int s) -> bool {
                    if (pend[s] < 0) return true;
                    const QTile t = decode(pend[s]);
                    pend[s] = -1;
                    if (!mbar_wait(&bars->out_full[s], (oph >> s) & 1u, abort_flag, p.err, 0x78)) return false;
                    oph ^= 1u << s;
                    if (!*abort_flag) {
                        index_ok(t.q0 < p.N, p.err, 0x98);
                        for (int x = 0; x < DV / 64; ++x)
                            tma_store_3d(&p.tm_out, stages + s * C::kStageBytes + x * (BM * 128), t.h * DV + x * 64,
                                         t.q0, t.b);
                        tma_store_commit();
                    }
                    tma_store_wait_read();
                    return true;
                };
                for (int k = 0; go; ++k) {
                    const int ti = tile_at(k);
                    if (ti < 0) break;
                    const QTile t = decode(ti);
                    // Q of tile k replaces Q of tile k-1 once its last score tiles are done.
                    if (k > 0 && !(go = mbar_wait(&bars->q_empty, (k - 1) & 1, abort_flag, p.err, 0x70))) break;
                    mbar_arrive_expect_tx(&bars->q_full, 2 * C::kQBytes);
                    index_ok(t.q0 < p.N && t.h < p.H && t.b < p.B, p.err, 0x96);
#pragma unroll
                    for (int x = 0; x < D / 64; ++x) {
                        tma_load_4d(q1s + x * C::kBoxBytes, &p.tm_q1, &bars->q_full, x * 64, t.q0, t.h, t.b);
                        tma_load_4d(q2s + x * C::kBoxBytes, &p.tm_q2, &bars->q_full, x * 64, t.q0, t.h, t.b);
                    }
                    nq = k + 1;
                    for (int j = 0; j < t.nkv; ++j, ++it) {
                        const int s = it % kPStages;
                        if (!(go = mbar_wait(&bars->kv_empty[s], ((it / kPStages) & 1) ^ 1, abort_flag, p.err, 0x71)))
                            break;
                        if (!(go = flush(s))) break;
                        uint8_t* st = stages + s * C::kStageBytes;
                        mbar_arrive_expect_tx(&bars->kv_full[s], C::kStageBytes);
                        index_ok(j * BN < p.N, p.err, 0x97);
#pragma unroll
                        for (int x = 0; x < D / 64; ++x) {
                            tma_load_4d(st + x * C::kBoxBytes, &p.tm_k1, &bars->kv_full[s], x * 64, j * BN, t.h, t.b);
                            tma_load_4d(st + C::kKBytes + x * C::kBoxBytes, &p.tm_k2, &bars->kv_full[s], x * 64,
                                        j * BN, t.h, t.b);
                        }
#pragma unroll
                        for (int x = 0; x < DV / 64; ++x)
                            tma_load_4d(st + 2 * C::kKBytes + x * C::kBoxBytes, &p.tm_v, &bars->kv_full[s], x * 64,
                                        j * BN, t.h, t.b);
                        if (j + 1 == t.nkv) pend[s] = ti;  // this stage will hold the tile's output
                    }
                }
                // The last tiles' outputs, in the order the tiles ended.
                for (int u = 0; u < kPStages; ++u)
                    if (go) go = flush((it + u) % kPStages);
                // Drain: no copy may still be landing in shared memory when the CTA exits.
                if (nq > 0) mbar_wait(&bars->q_full, (nq - 1) & 1, nullptr, p.err, 0x73);
                for (int u = max(0, it - kPStages); u < it; ++u)
                    mbar_wait(&bars->kv_full[u % kPStages], (u / kPStages) & 1, nullptr, p.err, 0x73);
            }
        } else if (warp == kWarpMma) {
            // ------------------------------------------------------------ MMA issuer
            const uint32_t tS[2] = {tmem + C::kColS, tmem + C::kColS + BN};
            const uint32_t tO[2] = {tmem + C::kColO, tmem + C::kColO + DV};
            const uint64_t dq[2] = {sdesc_sw128(smem_u32(q1s), 16, 1024), sdesc_sw128(smem_u32(q2s), 16, 1024)};
            const uint64_t dk0 = sdesc_sw128(smem_u32(stages), 16, 1024);
            const uint64_t dv0 = sdesc_sw128(smem_u32(stages) + 2 * C::kKBytes, BN * 128, 1024);
            constexpr uint64_t kStageStep = C::kStageBytes >> 4, kK2Step = C::kKBytes >> 4;
            uint32_t J = 0;  // key tiles done over all query tiles (= ring stages consumed)
            int k = 0, ti = tile_at(0);
            bool ok = true;
            if (ti >= 0) {
                // Score tiles of the first query tile's first key tile.
                ok = mbar_wait_warp(&bars->q_full, 0, abort_flag, p.err, 0x74) &&
                     mbar_wait_warp(&bars->kv_full[0], 0, abort_flag, p.err, 0x75);
                if (ok) {
                    tc_fence_after();
                    if (elect_one()) {
                        issue_qk<D, F16>(tS[0], dq[0], dk0);
                        umma_commit(&bars->s_full[0]);
                        issue_qk<D, F16>(tS[1], dq[1], dk0 + kK2Step);
                        umma_commit(&bars->s_full[1]);
                        if (decode(ti).nkv == 1) umma_commit(&bars->q_empty);
                    }
                    __syncwarp();
                }
            }
            while (ok && ti >= 0) {
                const int nkv = decode(ti).nkv;
                const int tn = tile_at(k + 1);
                const int nkv_next = tn >= 0 ? decode(tn).nkv : 0;
                for (int j = 0; ok && j < nkv; ++j, ++J) {
                    const bool last = j + 1 == nkv;
                    const bool more = !last || tn >= 0;  // a next score tile exists
                    const bool new_q = last && tn >= 0;  // ... and it belongs to the next query tile
                    // The next score tile is the last one of its query tile: its completion frees Q.
                    const bool last_s = last ? nkv_next == 1 : j + 2 == nkv;
                    const int s = (int)(J % kPStages), s1 = (int)((J + 1) % kPStages);
                    const uint64_t dv = dv0 + s * kStageStep, dk1 = dk0 + s1 * kStageStep;
                    for (int m = 0; m < 2; ++m) {
                        if (!mbar_wait_warp(&bars->p_half[m], J & 1, abort_flag, p.err, 0x77 + m)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (elect_one()) issue_pv_half<DV, F16>(tO[m], tS[m], dv, 0, j > 0 ? 1u : 0u);
                        __syncwarp();
                        // The next Q and K/V tiles are checked while the softmax still works on
                        // the second half of P, off the path from p_full to the MMAs.
                        if (m == 0 && more) {
                            if (new_q && !mbar_wait_warp(&bars->q_full, (k + 1) & 1, abort_flag, p.err, 0x79)) {
                                ok = false;
                                break;
                            }
                            if (!mbar_wait_warp(&bars->kv_full[s1], ((J + 1) / kPStages) & 1, abort_flag, p.err,
                                                0x7a)) {
                                ok = false;
                                break;
                            }
                        }
                        if (!mbar_wait_warp(&bars->p_full[m], J & 1, abort_flag, p.err, 0x7b + m)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (elect_one()) {
                            issue_pv_half<DV, F16>(tO[m], tS[m], dv, 1, 1u);
                            umma_commit(&bars->o_done[m]);
                            if (m == 1) umma_commit(&bars->kv_empty[s]);
                            if (more) {
                                issue_qk<D, F16>(tS[m], dq[m], dk1 + m * kK2Step);
                                umma_commit(&bars->s_full[m]);
                                if (m == 1 && last_s) umma_commit(&bars->q_empty);
                            }
                        }
                        __syncwarp();
                    }
                }
                ++k;
                ti = tn;
            }
            // Every MMA issued (also before an abort) must finish before TMEM is freed.
            if (elect_one()) umma_commit(&bars->drain);
            __syncwarp();
            mbar_wait(&bars->drain, 0, nullptr, p.err, 0x7d);
        }
        tc_fence_before();
        named_bar_sync(2, kThreads);
        if (warp == kWarpMma) {
            tc_fence_after();
            tmem_dealloc(tmem, C::kTmemCols);
        }
    } else {
        setmaxnreg_inc<kRegsSoftmax>();
        // ------------------------------------------------------------ softmax (map g) and epilogue
        const int g = warp >> 2;
        const int lg = warp & 3;
        const int r = lg * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(lg * 32) << 16);
        const uint32_t tS = lane_base + C::kColS + g * BN;
        const uint32_t tO = lane_base + C::kColO + g * DV;
        constexpr int kHalf = DV / 2;  // output columns handled by this group
        const bool f16 = p.out_f16 != 0;
        uint32_t J = 0;
        bool ok = true;
        // Every softmax thread walks the same tile list and takes every named barrier,
        // also after a failed wait (then without waiting or computing).
        for (int k = 0;; ++k) {
            const int ti = tile_at(k);
            if (ti < 0) break;
            const QTile t = decode(ti);
            const int q0 = t.q0, nkv = t.nkv;
            const int qrow = q0 + r;
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; ok && j < nkv; ++j, ++J)
                ok = softmax_tile<DV, F16>(p, g, &bars->s_full[g], &bars->o_done[g], &bars->p_half[g],
                                           &bars->p_full[g], abort_flag, tS, tO, q0, qrow, j * BN, j == 0, J & 1u,
                                           m_used, l);
            // Epilogue: O1/l1 - lambda O2/l2, row RMSNorm, (1 - lambda_init), norm weight.
            if (ok) {
                ok = mbar_wait_warp(&bars->o_done[0], (J - 1) & 1u, abort_flag, p.err, 0x44) &&
                     mbar_wait_warp(&bars->o_done[1], (J - 1) & 1u, abort_flag, p.err, 0x45);
            }
            tc_fence_after();
            // Exchange slot X[g][r] is written by group g and read by the other group,
            // which then reuses it for its own sum of squares.
            const float own = (g == 0) ? 1.0f / l : p.lambda / l;
            xch[g * BM + r] = own;
            named_bar_sync(1, 256);
            const float par = xch[(1 - g) * BM + r];
            const float inv1 = g == 0 ? own : par, inv2 = g == 0 ? par : own;
            // Two passes over O (sum of squares, then the scaled output), so that no
            // output row is held in registers across the exchange.
            float ss = 0.f;
            if (ok) {
#pragma unroll
                for (int c = 0; c < kHalf / 32; ++c) {
                    uint32_t o1[32], o2[32];
                    tmem_ld32(lane_base + C::kColO + g * kHalf + c * 32, o1);
                    tmem_ld32(lane_base + C::kColO + DV + g * kHalf + c * 32, o2);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float x = __uint_as_float(o1[i]) * inv1 - __uint_as_float(o2[i]) * inv2;
                        ss = fmaf(x, x, ss);
                    }
                }
            }
            xch[(1 - g) * BM + r] = ss;
            named_bar_sync(1, 256);
            // Stage this group's DV/2 columns as 128-byte-swizzled boxes of 128 rows in the
            // stage that held the tile's last K/V tiles (idle since the last PV); the
            // producer stores the tile from there.
            uint8_t* stage = stages + (int)((J - 1) % kPStages) * C::kStageBytes;
            if (ok) {
                const float tot = ss + xch[g * BM + r];
                const float rsc = (1.0f - p.lambda_init) / sqrtf(tot / (float)DV + p.eps);
                const float* w = p.norm_w ? p.norm_w + g * kHalf : nullptr;
#pragma unroll
                for (int c = 0; c < kHalf / 32; ++c) {
                    uint32_t o1[32], o2[32];
                    tmem_ld32(lane_base + C::kColO + g * kHalf + c * 32, o1);
                    tmem_ld32(lane_base + C::kColO + DV + g * kHalf + c * 32, o2);
                    tmem_ld_wait();
                    // 32 columns = half a box row: box (g DV/2 + 32 c) / 64, 16-byte chunks (c % 2) * 4 ..
                    uint8_t* box = stage + ((g * kHalf + c * 32) / 64) * (BM * 128);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int i = q * 8 + e;
                            const float x = __uint_as_float(o1[i]) * inv1 - __uint_as_float(o2[i]) * inv2;
                            y[e] = x * rsc * (w ? w[c * 32 + i] : 1.f);
                        }
                        *reinterpret_cast<uint4*>(box + sw128_offset(r, (c & 1) * 4 + q)) =
                            make_uint4(pack_16x2(y[0], y[1], f16), pack_16x2(y[2], y[3], f16),
                                       pack_16x2(y[4], y[5], f16), pack_16x2(y[6], y[7], f16));
                    }
                }
            }
            // Both groups' reads of O precede this barrier; the next tile's first PV products
            // (which overwrite O) follow it through the P hand-off.
            tc_fence_before();
            fence_proxy_async_shared();
            named_bar_sync(1, 256);
            if (threadIdx.x == 0) mbar_arrive(&bars->out_full[(J - 1) % kPStages]);
        }
        tc_fence_before();
        named_bar_sync(2, kThreads);
    }
}

template <int D, int DV, bool F16>
cudaError_t launch_persist_t(const FwdParams& p, cudaStream_t stream) {
    using C = PersistCfg<D, DV>;
    auto k = fwd_persist_kernel<D, DV, F16>;
    cudaError_t e = prepare_once<fwd_persist_kernel<D, DV, F16>>((int)C::kSmem, kRegsLaunch);
    if (e != cudaSuccess) return e;
    int sms = 0;
    if ((e = device_sm_count(&sms)) != cudaSuccess) return e;
    const int total = ((p.N + BM - 1) / BM) * p.B * p.H;
    k<<<min(total, sms), kThreads, C::kSmem, stream>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Backward preparation from the state a training forward saved, on the CUDA
// cores: per query row, the quantities prep_epilogue derives in the forward
// (dO rounded to the operand type, L1, L2, D1, D2, and the row's dlambda and
// gain-gradient terms), from O1, O2 and each map's max and sum instead of TMEM.
// HBM-bound (~1.3 KB per row): one warp per row, four columns per lane, warp
// butterflies for the row sums; one CTA (8 warps) per 128-row query tile, whose
// rows its warps take in a fixed order, so the per-CTA partials of dlambda and
// of the gain's gradient are indexed and summed like the forward's. At most 64
// registers, so four CTAs share an SM (45 us vs 48 us at three).
constexpr int kSavedThreads = 256;

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <bool F16>
__global__ void __launch_bounds__(kSavedThreads, 4) bwd_prep_saved_kernel(const __grid_constant__ FwdParams p) {
    // the key-side kernel that follows may start its setup and K/V loads once every CTA of
    // this grid has started (it waits for this grid before reading dO and the statistics)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int DV = 128, kWarps = kSavedThreads / 32;
    using T16x2 = typename std::conditional<F16, __half2, __nv_bfloat162>::type;
    __shared__ float wsum[kWarps][DV];
    __shared__ float lsum[kWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = (p.N + BM - 1) / BM;
    const int BH = p.B * p.H;
    const int qt = n_tiles - 1 - (int)(blockIdx.x / BH);  // the forward's CTA order
    const int bh = blockIdx.x % BH;
    const int b = bh / p.H, h = bh % p.H;
    const int q0 = qt * BM;
    const float lam = p.lambda, cs = 1.0f - p.lambda_init;
    const int c0 = 4 * lane;
    const float4 w = p.norm_w ? *reinterpret_cast<const float4*>(p.norm_w + c0) : make_float4(1.f, 1.f, 1.f, 1.f);
    float dw[4] = {0.f, 0.f, 0.f, 0.f}, dl = 0.f;
    // The warp's rows, in order; each row's operands are loaded one row ahead.
    const int rbeg = q0 + warp * (BM / kWarps), rend = min(rbeg + BM / kWarps, p.N);
    struct RowIn {
        float2 lse;  // L1, L2
        float4 x;    // this lane's four columns of x = O1/l1 - lambda O2/l2
        uint2 a2;    // and of O2/l2 (16-bit)
        uint2 dy;
    };
    auto load_row = [&](int qrow) {
        const int64_t row = ((int64_t)b * p.H + h) * p.N + qrow;
        RowIn in;
        in.lse = *reinterpret_cast<const float2*>(p.lse_save + row * 2);
        in.x = *reinterpret_cast<const float4*>(p.x_save + row * DV + c0);
        in.a2 = *reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(p.a2_save) + (row * DV + c0) * 2);
        in.dy = *reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(p.dy) +
                                                ((((int64_t)b * p.N + qrow) * p.H + h) * DV + c0) * 2);
        return in;
    };
    RowIn next{};
    if (rbeg < rend) next = load_row(rbeg);
    for (int qrow = rbeg; qrow < rend; ++qrow) {  // warp-uniform bounds
        const int64_t row = ((int64_t)b * p.H + h) * p.N + qrow;
        const RowIn cur = next;
        if (qrow + 1 < rend) next = load_row(qrow + 1);
        const float2 lse = cur.lse;
        // four 16-bit values of the operand type as floats
        auto unpack4 = [](uint2 u, float* o) {
            if constexpr (F16) {
                const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
                const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
                o[0] = a.x; o[1] = a.y; o[2] = c.x; o[3] = c.y;
            } else {
                o[0] = bf16lo_to_f32(u.x); o[1] = bf16hi_to_f32(u.x);
                o[2] = bf16lo_to_f32(u.y); o[3] = bf16hi_to_f32(u.y);
            }
        };
        float a2[4], dyv[4];
        unpack4(cur.a2, a2);
        unpack4(cur.dy, dyv);
        const float xv[4] = {cur.x.x, cur.x.y, cur.x.z, cur.x.w};
        float a1[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) a1[k] = fmaf(lam, a2[k], xv[k]);  // O1/l1
        const float wv[4] = {w.x, w.y, w.z, w.w};
        float x[4], ss = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[k] = xv[k];  // the forward's own fp32 value
            ss = fmaf(x[k], x[k], ss);
        }
        const float ir = 1.0f / sqrtf(warp_allsum(ss) / (float)DV + p.eps);
        float n[4], gg[4], gn = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            n[k] = x[k] * ir;
            gg[k] = dyv[k] * wv[k] * cs;
            gn = fmaf(gg[k], n[k], gn);
        }
        gn = warp_allsum(gn) / (float)DV;
        float d[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) d[k] = (gg[k] - n[k] * gn) * ir;
        // dO in the operand type; D1, D2 from the rounded dO the gradient products use (so
        // that sum_j P_ij (dA_ij - D_i) stays zero for every row), dlambda from the unrounded one.
        T16x2 lo, hi;
        float r[4];
        if constexpr (F16) {
            lo = __floats2half2_rn(d[0], d[1]);
            hi = __floats2half2_rn(d[2], d[3]);
            const float2 u = __half22float2(lo), v = __half22float2(hi);
            r[0] = u.x; r[1] = u.y; r[2] = v.x; r[3] = v.y;
        } else {
            lo = __floats2bfloat162_rn(d[0], d[1]);
            hi = __floats2bfloat162_rn(d[2], d[3]);
            const float2 u = __bfloat1622float2(lo), v = __bfloat1622float2(hi);
            r[0] = u.x; r[1] = u.y; r[2] = v.x; r[3] = v.y;
        }
        uint2 packed;
        packed.x = *reinterpret_cast<const uint32_t*>(&lo);
        packed.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.d_o) + (row * DV + c0) * 2) = packed;
        float x1 = 0.f, x2 = 0.f, x2e = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x1 = fmaf(r[k], a1[k], x1);
            x2 = fmaf(r[k], a2[k], x2);
            x2e = fmaf(d[k], a2[k], x2e);
            dw[k] = fmaf(dyv[k] * n[k], cs, dw[k]);
        }
        x1 = warp_allsum(x1);
        x2 = warp_allsum(x2);
        x2e = warp_allsum(x2e);
        if (lane == 0)
            *reinterpret_cast<float4*>(p.stats + row * 4) =
                make_float4(lse.x, lse.y, x1, -lam * x2);
        dl -= x2e;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) wsum[warp][c0 + k] = dw[k];
    if (lane == 0) lsum[warp] = dl;
    __syncthreads();
    if (threadIdx.x < DV) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < kWarps; ++k) acc += wsum[k][threadIdx.x];
        p.part_w[(int64_t)blockIdx.x * DV + threadIdx.x] = acc;
    }
    if (threadIdx.x == 0) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < kWarps; ++k) acc += lsum[k];
        p.part_lam[blockIdx.x] = acc;
    }
}

template <bool F16>
cudaError_t launch_prep_saved_t(const FwdParams& p, cudaStream_t stream) {
    const int n_tiles = (p.N + BM - 1) / BM;
    bwd_prep_saved_kernel<F16><<<n_tiles * p.B * p.H, kSavedThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdParams& p, cudaStream_t stream) {
    if (p.d == 64 && p.Dv == 128) {
        // Short sequences: the persistent form (its saving per query tile outweighs its
        // slower key-tile loop while a query tile has few key tiles; measured crossover
        // near 16 key tiles on average, i.e. causal N = 4096).
        const int n_tiles = (p.N + BM - 1) / BM;
        const double mean_kv = p.causal ? 0.5 * (n_tiles + 1) : (double)n_tiles;
        if ((p.out_bf16 || p.out_f16) && mean_kv <= kPersistMaxMeanKv)
            return p.in_f16 ? launch_persist_t<64, 128, true>(p, stream) : launch_persist_t<64, 128, false>(p, stream);
        return p.in_f16 ? launch_t<64, 128, true, kModePlain>(p, stream) : launch_t<64, 128, false, kModePlain>(p, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_train(const FwdParams& p, cudaStream_t stream) {
    if (p.d == 64 && p.Dv == 128 && p.x_save && p.a2_save && p.lse_save)
        return p.in_f16 ? launch_t<64, 128, true, kModeSave>(p, stream) : launch_t<64, 128, false, kModeSave>(p, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_prep_saved(const FwdParams& p, cudaStream_t stream) {
    if (p.d == 64 && p.Dv == 128 && p.dy && p.d_o && p.stats && p.part_lam && p.part_w && p.x_save && p.a2_save && p.lse_save)
        return p.in_f16 ? launch_prep_saved_t<true>(p, stream) : launch_prep_saved_t<false>(p, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_prep(const FwdParams& p, cudaStream_t stream) {
    if (p.d == 64 && p.Dv == 128 && p.dy && p.d_o && p.stats && p.part_lam && p.part_w)
        return p.in_f16 ? launch_t<64, 128, true, kModePrep>(p, stream) : launch_t<64, 128, false, kModePrep>(p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace da
