// Fused causal prefill of differential attention for wide heads on a pair of
// CTAs (a 2-CTA thread-block cluster), tcgen05 MMAs with TMEM accumulators.
//
// Same computation as fwd_tcgen05.cu — the DiffAttn formula of "Differential
// Transformer: Transformer que cancela ruído de atenção" (section "Como a
// atenção diferencial funciona") under the causal mask of the intoai.pub page
// ("A Deeper Dive Into Attention Calculations"), then the per-head RMSNorm and
// (1 - lambda_init) scale (section "Estrutura multi-head e arquitetura
// completa"), output [B, N, H, Dv] — for head widths whose two accumulators do
// not fit one CTA's tensor memory together with the score tiles
// (d = 128, Dv = 256: S1 + S2 + O1 + O2 would need 768 of 512 TMEM columns).
//
// The two maps are independent until the final combination, so CTA rank m of
// the pair computes map m alone: S = Q_m K_m^T into a double-buffered score
// tile (2 x 128 columns), its online softmax, O_m += P V (Dv columns). While
// the softmax warps work on S(j+1), the tensor core runs PV(j) and S(j+2).
// The epilogue forms O1/l1 - lambda O2/l2 across the pair through distributed
// shared memory: each CTA finishes half of the Dv columns, the two halves'
// sums of squares are exchanged for the row RMSNorm, and each CTA stores its
// half of the output.
//
// Warps: 0 TMA producer (Q_m once, then rings of K_m and V tiles), 1 TMEM owner
// and MMA issuer, 2..5 softmax and epilogue (warp w reads TMEM lanes
// 32*(w%4)..+31, i.e. query rows of the tile).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace da {
namespace {

constexpr int BM = 128, BN = 128;
constexpr int kThreads = 6 * 32;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D, int DV>
struct PairCfg {
    static constexpr int kQBytes = BM * D * 2;
    static constexpr int kKBytes = BN * D * 2;
    static constexpr int kVBytes = BN * DV * 2;
    static constexpr int kVHBytes = kVBytes / 2;      // half a V tile: 64 keys
    static constexpr int kBoxBytes = 128 * 128;  // one [128 rows][64 bf16] box
    // Separate K and V rings: S(j+2) needs K two tiles ahead, PV(j) needs V(j).
    static constexpr int kKStages = (D == 128) ? 2 : 4;
    static constexpr int kVStages = (D == 128) ? 2 : 4;
    static constexpr int kVHStages = 2 * kVStages;   // the V ring holds half tiles
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kQBytes;
    static constexpr int kOffV = kOffK + kKStages * kKBytes;
    static constexpr int kOffStages = kOffK;
    static constexpr int kOffBar = kOffV + kVStages * kVBytes;
    static constexpr int kBarBytes = 320;             // PairBars, rounded up
    static constexpr size_t kSmem = 1024 + (size_t)kOffBar + kBarBytes;
    static constexpr int kHalf = DV / 2;              // output columns finished by each CTA
    static constexpr int kXStride = kHalf + 4;        // padded row of the exchange buffer (floats)
    static constexpr int kOffX = kOffStages;          // exchange buffer reuses the K/V rings
    static constexpr int kOffSS = kOffX + BM * kXStride * 4;
    static_assert(kOffSS + BM * 4 <= kOffBar, "epilogue buffers fit in the K/V rings");
    // Output staging (128-byte-swizzled boxes of 128 rows, up to 64 KB) in the
    // second half of the V ring, clear of the exchange buffers.
    static constexpr int kOffOut = kOffV + kVStages * kVBytes / 2;
    static_assert(kOffOut >= kOffSS + BM * 4 && kOffOut % 1024 == 0, "staging after the exchange buffers");
    static_assert(kOffOut + BM * 128 * (kHalf / 32) <= kOffBar, "fp32 staging fits");
    static_assert(kSmem <= 232448, "shared memory budget");
    static_assert(kKStages <= 4 && kVHStages <= 8 && kVHStages % 2 == 0, "barrier arrays");
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColO = 2 * BN;
    static_assert(2 * BN + DV <= 512, "TMEM budget");
};

struct PairBars {
    uint64_t q_full;
    uint64_t k_full[4];  // kKStages <= 4
    uint64_t k_empty[4];
    uint64_t v_full[8];
    uint64_t v_empty[8];
    uint64_t s_full[2];
    uint64_t p_half[2];  // P of keys 0..BN/2-1 of score buffer b is in TMEM
    uint64_t p_full[2];
    uint64_t o_done;
    uint64_t drain;
    uint64_t xsync;  // epilogue rendezvous of the pair: one local and one remote arrival per phase
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(PairBars) <= PairCfg<128, 256>::kBarBytes, "barrier block");

template <int D, bool F16>
__device__ __forceinline__ void issue_qk(uint32_t s_tmem, uint64_t q_desc, uint64_t k_desc) {
    constexpr uint32_t idesc = idesc_kind_f16(BM, BN, 0, 0, F16);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = (uint64_t)(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
        umma_ss(s_tmem, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u);
    }
}

// O (+)= P V with P in TMEM (lane r = row r, 16 keys per 8 columns) and the V
// tile's descriptor advancing 2048 bytes (16 keys) per step.
// O (+)= P V for one half of the keys: P from TMEM (keys half*BN/2 .. +BN/2, 16
// keys per 8 columns), V from a half-tile stage: boxes of [BN/2 keys][64 columns]
// (leading offset to the next 64 columns), 8 keys per 1024 bytes, so one K=16 step
// advances 2048 bytes (128 in 16-byte units).
template <int DV, bool F16>
__device__ __forceinline__ void issue_pv_half(uint32_t o_tmem, uint32_t p_tmem, uint64_t vh_desc, int half,
                                              uint32_t accumulate) {
    constexpr uint32_t idesc = idesc_kind_f16(BM, DV, 0, 1, F16);
#pragma unroll
    for (int k = 0; k < BN / 32; ++k) {
        const int kk = half * (BN / 32) + k;
        umma_ts(o_tmem, p_tmem + kk * 8, vh_desc + (uint64_t)(k * 128), idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
}

template <int D, int DV, bool F16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    fwd_pair_kernel(const __grid_constant__ FwdParams p) {
    using C = PairCfg<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PairBars* bars = reinterpret_cast<PairBars*>(smem + C::kOffBar);
    volatile int* abort_flag = &bars->abort;

    const uint32_t rank = cluster_ctarank();  // which map this CTA computes
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = (p.N + BM - 1) / BM;
    const int BH = p.B * p.H;
    const int tile = (int)(blockIdx.x >> 1);
    const int qt = n_tiles - 1 - tile / BH;  // heaviest causal tiles first
    const int bh = tile % BH;
    const int b = bh / p.H, h = bh % p.H;
    const int q0 = qt * BM;
    const int nkv = p.causal ? min(qt + 1, n_tiles) : n_tiles;
    const CUtensorMap* tm_q = rank ? &p.tm_q2 : &p.tm_q1;
    const CUtensorMap* tm_k = rank ? &p.tm_k2 : &p.tm_k1;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
        }
        for (int s = 0; s < C::kVHStages; ++s) {
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->p_half[i], 4);  // one arrival per softmax warp
            mbar_init(&bars->p_full[i], 4);
        }
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->drain, 1);
        mbar_init(&bars->xsync, 2);
        bars->abort = 0;
        fence_mbarrier_init();
    }
    // The peer arrives on xsync later, so its initialisation must be visible
    // cluster-wide first. Both CTAs of a cluster are co-scheduled, so this
    // barrier waits only for the peer to start (it precedes every other wait).
    cluster_sync_start();
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // The setup above may overlap the previous kernel's tail (the projection GEMM that wrote
    // Q, K and V).
    pdl_trigger();
    pdl_wait();
    const uint32_t tmem = bars->tmem_base;
    uint8_t* qs = smem + C::kOffQ;
    uint8_t* ks = smem + C::kOffK;
    uint8_t* vs = smem + C::kOffV;

    bool ok = true;
    float l = 0.f;
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(tm_q);
            tma_prefetch_desc(tm_k);
            tma_prefetch_desc(&p.tm_v);
            mbar_arrive_expect_tx(&bars->q_full, C::kQBytes);
            index_ok(q0 < p.N && h < p.H && b < p.B, p.err, 0x93);
#pragma unroll
            for (int x = 0; x < D / 64; ++x) tma_load_4d(qs + x * C::kBoxBytes, tm_q, &bars->q_full, x * 64, q0, h, b);
            // Issue order K(j), V(j): K tiles run ahead as soon as S frees them, V tiles
            // follow the PV products.
            int jk = 0, jv = 0;
            bool go = true;
            for (int j = 0; go && j < nkv; ++j) {
                const int sk = j % C::kKStages;
                go = mbar_wait(&bars->k_empty[sk], ((j / C::kKStages) & 1) ^ 1, abort_flag, p.err, 0x51);
                if (!go) break;
                mbar_arrive_expect_tx(&bars->k_full[sk], C::kKBytes);
                index_ok(j * BN < p.N, p.err, 0x94);
#pragma unroll
                for (int x = 0; x < D / 64; ++x)
                    tma_load_4d(ks + sk * C::kKBytes + x * C::kBoxBytes, tm_k, &bars->k_full[sk], x * 64, j * BN, h,
                                b);
                jk = j + 1;
                // V(j) as two half tiles of BN/2 keys, each in its own stage of the V ring.
                for (int hh = 0; go && hh < 2; ++hh) {
                    const int u = 2 * j + hh, su = u % C::kVHStages;
                    go = mbar_wait(&bars->v_empty[su], ((u / C::kVHStages) & 1) ^ 1, abort_flag, p.err, 0x52);
                    if (!go) break;
                    mbar_arrive_expect_tx(&bars->v_full[su], C::kVHBytes);
#pragma unroll
                    for (int x = 0; x < DV / 64; ++x)
                        tma_load_4d(vs + su * C::kVHBytes + x * (BN / 2) * 128, &p.tm_v, &bars->v_full[su], x * 64,
                                    j * BN + hh * (BN / 2), h, b);
                    jv = u + 1;
                }
            }
            // Drain: no copy may still be landing in shared memory when the CTA exits.
            mbar_wait(&bars->q_full, 0, nullptr, p.err, 0x53);
            for (int u = max(0, jk - C::kKStages); u < jk; ++u)
                mbar_wait(&bars->k_full[u % C::kKStages], (u / C::kKStages) & 1, nullptr, p.err, 0x53);
            for (int u = max(0, jv - C::kVHStages); u < jv; ++u)
                mbar_wait(&bars->v_full[u % C::kVHStages], (u / C::kVHStages) & 1, nullptr, p.err, 0x53);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp walks the loop and waits; one elected lane issues each
        // group of MMAs together with the commits that track them.
        const uint32_t tS[2] = {tmem, tmem + BN};
        const uint32_t tO = tmem + C::kColO;
        const uint64_t dq = sdesc_sw128(smem_u32(qs), 16, 1024);
        const uint64_t dk0 = sdesc_sw128(smem_u32(ks), 16, 1024);
        const uint64_t dv0 = sdesc_sw128(smem_u32(vs), (BN / 2) * 128, 1024);
        constexpr uint64_t kKStep = C::kKBytes >> 4, kVHStep = C::kVHBytes >> 4;
        // S(j) = Q K(j)^T into score buffer j % 2, then K(j) is released.
        auto issue_s = [&](int j) -> bool {
            const int sk = j % C::kKStages;
            if (!mbar_wait_warp(&bars->k_full[sk], (j / C::kKStages) & 1, abort_flag, p.err, 0x55)) return false;
            tc_fence_after();
            if (elect_one()) {
                issue_qk<D, F16>(tS[j & 1], dq, dk0 + sk * kKStep);
                umma_commit(&bars->s_full[j & 1]);
                umma_commit(&bars->k_empty[sk]);
            }
            __syncwarp();
            return true;
        };
        bool go = mbar_wait_warp(&bars->q_full, 0, abort_flag, p.err, 0x54) && issue_s(0) && (nkv < 2 || issue_s(1));
        for (int j = 0; go && j < nkv; ++j) {
            const int bf = j & 1;
            // Half h of PV(j) reads V half tile u = 2j + h and the h-th half of P(j); the
            // first starts as soon as the softmax has written the first half of P(j).
            const int u0 = (2 * j) % C::kVHStages, u1 = (2 * j + 1) % C::kVHStages;
            const uint32_t pu = (uint32_t)((2 * j) / C::kVHStages) & 1;  // same phase for both halves
            if (!mbar_wait_warp(&bars->v_full[u0], pu, abort_flag, p.err, 0x58)) break;
            if (!mbar_wait_warp(&bars->p_half[bf], (j >> 1) & 1, abort_flag, p.err, 0x56)) break;
            tc_fence_after();
            if (elect_one()) {
                issue_pv_half<DV, F16>(tO, tS[bf], dv0 + u0 * kVHStep, 0, j > 0 ? 1u : 0u);
                umma_commit(&bars->v_empty[u0]);
            }
            __syncwarp();
            if (!mbar_wait_warp(&bars->v_full[u1], pu, abort_flag, p.err, 0x5a)) break;
            if (!mbar_wait_warp(&bars->p_full[bf], (j >> 1) & 1, abort_flag, p.err, 0x57)) break;
            tc_fence_after();
            if (elect_one()) {
                issue_pv_half<DV, F16>(tO, tS[bf], dv0 + u1 * kVHStep, 1, 1u);
                umma_commit(&bars->o_done);
                umma_commit(&bars->v_empty[u1]);
            }
            __syncwarp();
            // S(j+2) reuses buffer bf: it is issued after PV(j), which reads P(j)
            // there, and tcgen05 MMAs of one thread execute in issue order.
            if (j + 2 < nkv && !issue_s(j + 2)) break;
        }
        // Every MMA issued (also before an abort) must finish before TMEM is freed.
        if (elect_one()) umma_commit(&bars->drain);
        __syncwarp();
        mbar_wait(&bars->drain, 0, nullptr, p.err, 0x59);
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int lg = warp & 3;
        const int r = lg * 32 + lane;  // query row within the tile == TMEM lane
        const int qrow = q0 + r;
        const uint32_t lane_base = tmem + ((uint32_t)(lg * 32) << 16);
        const uint32_t tO = lane_base + C::kColO;
        const float sl2 = p.scale_log2;
        float m_used = -INFINITY;
        for (int j = 0; j < nkv; ++j) {
            const int bf = j & 1;
            const uint32_t tS = lane_base + bf * BN;
            if (!mbar_wait_warp(&bars->s_full[bf], (j >> 1) & 1, abort_flag, p.err, 0x60)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS + c * 32, sr + c * 32);
            tmem_ld_wait();
            const int kbase = j * BN;
            if ((p.causal && kbase + BN - 1 > q0) || (kbase + BN > p.N)) {
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
            // Only a rescale of O has to wait for PV(j-1); P(j) goes to the other
            // score buffer. S(j) was issued after PV(j-2), so once it has landed
            // o_done is at most one phase behind and the parity wait is exact.
            if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                if (!mbar_wait_warp(&bars->o_done, (j - 1) & 1, abort_flag, p.err, 0x61)) {
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
            // P row (16-bit pairs, lower key in the low half) -> the first BN/2 columns of
            // S, in two halves: the first is handed to the MMA warp before the second is
            // exponentiated, so the first half of PV(j) overlaps the rest of the softmax.
            float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t pk[BN / 4];
#pragma unroll
                for (int i = 0; i < BN / 2; i += 2) {
                    const int kx = hf * (BN / 2) + i;
                    const float e0 = fast_exp2(fmaf(__uint_as_float(sr[kx]), sl2, -m_used));
                    const float e1 = fast_exp2(fmaf(__uint_as_float(sr[kx + 1]), sl2, -m_used));
                    rs[(i >> 1) & 3] += e0 + e1;
                    pk[i / 2] = pack_p<F16>(e0, e1);
                }
                tmem_st32(tS + hf * (BN / 4), pk);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(hf == 0 ? &bars->p_half[bf] : &bars->p_full[bf]);
            }
            l = l * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
        }
        if (ok && nkv > 0) ok = mbar_wait_warp(&bars->o_done, (nkv - 1) & 1, abort_flag, p.err, 0x62);
        tc_fence_after();
    }

    // ---------------------------------------------------------------- epilogue
    // Every thread of both CTAs takes part in the three pair_sync calls below.
    // TMEM reads are done by whole warps (tcgen05.ld is warp-collective); only
    // the global stores depend on the row being < N. The pair exchanges data by
    // pushing it into the peer's shared memory (remote stores), then reads its
    // own shared memory.
    constexpr int H2 = C::kHalf;
    float* xbuf = reinterpret_cast<float*>(smem + C::kOffX);  // [BM][kXStride]: the peer's part of my half
    float* ssbuf = reinterpret_cast<float*>(smem + C::kOffSS);  // the peer's sums of squares
    const bool epi = warp >= 2;
    const int lg = warp & 3;
    const int r = lg * 32 + lane;
    const uint32_t tO = tmem + ((uint32_t)(lg * 32) << 16) + C::kColO;
    const uint32_t peer = rank ^ 1u;
    const float coef = (rank == 0) ? 1.0f / l : -p.lambda / l;  // this map's weight in O1/l1 - lambda O2/l2
    const uint32_t own0 = rank * H2, other0 = peer * H2;
    // The exchange buffers live in the K/V rings: both CTAs must be past their
    // last MMA before either writes into the other's.
    ok = pair_sync(&bars->xsync, peer, 0, abort_flag, p.err, 0x63) && ok;
    ok = __all_sync(0xffffffffu, ok);
    if (epi && ok) {
        // Phase A: the half of this map's row the peer finishes -> the peer's buffer.
        const uint32_t peer_x = mapa_shared(smem_u32(xbuf + r * C::kXStride), peer);
#pragma unroll 1
        for (int c = 0; c < H2 / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + other0 + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i)
                st_dsmem_f4(peer_x + (uint32_t)(c * 32 + 4 * i) * 4u,
                            make_float4(__uint_as_float(o[4 * i]) * coef, __uint_as_float(o[4 * i + 1]) * coef,
                                        __uint_as_float(o[4 * i + 2]) * coef, __uint_as_float(o[4 * i + 3]) * coef));
        }
    }
    ok = pair_sync(&bars->xsync, peer, 1, abort_flag, p.err, 0x64) && ok;
    ok = __all_sync(0xffffffffu, ok);
    const float* xrow = xbuf + r * C::kXStride;
    float ss = 0.f;
    if (epi && ok) {
        // Phase B: this CTA's half of O1/l1 - lambda O2/l2 and its sum of squares,
        // which goes to the peer as well.
#pragma unroll 1
        for (int c = 0; c < H2 / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + own0 + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 q = *reinterpret_cast<const float4*>(xrow + c * 32 + 4 * i);
                const float x0 = fmaf(__uint_as_float(o[4 * i]), coef, q.x);
                const float x1 = fmaf(__uint_as_float(o[4 * i + 1]), coef, q.y);
                const float x2 = fmaf(__uint_as_float(o[4 * i + 2]), coef, q.z);
                const float x3 = fmaf(__uint_as_float(o[4 * i + 3]), coef, q.w);
                ss = fmaf(x0, x0, fmaf(x1, x1, fmaf(x2, x2, fmaf(x3, x3, ss))));
            }
        }
        st_dsmem_f32(mapa_shared(smem_u32(ssbuf + r), peer), ss);
    }
    ok = pair_sync(&bars->xsync, peer, 2, abort_flag, p.err, 0x65) && ok;
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    if (epi && ok) {
        // Phase C: normalise and store this CTA's half of the row.
        const float tot = ss + ssbuf[r];
        const float rsc = (1.0f - p.lambda_init) / sqrtf(tot / (float)DV + p.eps);
        // Stage the half row in 128-byte-swizzled boxes of 128 rows; one TMA store per
        // box writes the tile and clips the rows past N.
        uint8_t* stage = smem + C::kOffOut;
#pragma unroll 1
        for (int c = 0; c < H2 / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + own0 + c * 32, o);
            tmem_ld_wait();
            float y[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 q = *reinterpret_cast<const float4*>(xrow + c * 32 + 4 * i);
                y[4 * i] = fmaf(__uint_as_float(o[4 * i]), coef, q.x) * rsc;
                y[4 * i + 1] = fmaf(__uint_as_float(o[4 * i + 1]), coef, q.y) * rsc;
                y[4 * i + 2] = fmaf(__uint_as_float(o[4 * i + 2]), coef, q.z) * rsc;
                y[4 * i + 3] = fmaf(__uint_as_float(o[4 * i + 3]), coef, q.w) * rsc;
            }
            if (p.norm_w) {
#pragma unroll
                for (int i = 0; i < 32; ++i) y[i] *= p.norm_w[own0 + c * 32 + i];
            }
            if (p.out_bf16 || p.out_f16) {
                const bool f16 = p.out_f16 != 0;
                // 32 columns = half a box row: box c/2, 16-byte chunks (c%2)*4 .. +3.
                uint8_t* box = stage + (c >> 1) * (BM * 128);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    *reinterpret_cast<uint4*>(box + sw128_offset(r, (c & 1) * 4 + i)) =
                        make_uint4(pack_16x2(y[8 * i], y[8 * i + 1], f16), pack_16x2(y[8 * i + 2], y[8 * i + 3], f16),
                                   pack_16x2(y[8 * i + 4], y[8 * i + 5], f16),
                                   pack_16x2(y[8 * i + 6], y[8 * i + 7], f16));
            } else {
                uint8_t* box = stage + c * (BM * 128);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    *reinterpret_cast<float4*>(box + sw128_offset(r, i)) =
                        make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
            }
        }
    }
    if (epi) {
        fence_proxy_async_shared();
        named_bar_sync(1, 128);  // all four epilogue warps, on every path
        if (warp == 2 && lane == 0 && !*abort_flag) {
            const int bw = p.out_bf16 || p.out_f16 ? 64 : 32;  // elements per 128-byte box row
            index_ok(q0 < p.N && own0 + H2 <= DV, p.err, 0x95);
            for (int i = 0; i < H2 / bw; ++i)
                tma_store_3d(&p.tm_out, smem + C::kOffOut + i * (BM * 128), h * DV + own0 + i * bw, q0, b);
            tma_store_commit();
            tma_store_wait_read();
        }
    }
    // No remote access follows the third rendezvous: each CTA's pushes into the
    // other landed before it, so either may exit.

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, int DV, bool F16>
cudaError_t launch_t(const FwdParams& p, cudaStream_t stream) {
    using C = PairCfg<D, DV>;
    auto k = fwd_pair_kernel<D, DV, F16>;
    cudaError_t e = prepare_once<fwd_pair_kernel<D, DV, F16>>((int)C::kSmem);
    if (e != cudaSuccess) return e;
    const int n_tiles = (p.N + BM - 1) / BM;
    return launch_pdl(k, dim3(2 * n_tiles * p.B * p.H), dim3(kThreads), C::kSmem, stream, p);
}

}  // namespace

cudaError_t launch_fwd_pair_bf16(const FwdParams& p, cudaStream_t stream) {
    if (p.d == 128 && p.Dv == 256)
        return p.in_f16 ? launch_t<128, 256, true>(p, stream) : launch_t<128, 256, false>(p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace da
