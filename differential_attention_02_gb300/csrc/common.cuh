// Device-side building blocks shared by the kernels of libdiffattn.so:
// error reporting, bounded mbarrier waits, TMA loads, and tcgen05 (UMMA / TMEM)
// wrappers written as inline PTX for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace da {

// ----------------------------------------------------------------------------
// Workspace control block and device error word
// ----------------------------------------------------------------------------
// Every workspace starts with a 256-byte control block; word 0 is the error word.
// A device code is (site << 8) | kind; kind 1 = a bounded wait gave up.
constexpr size_t kControlBytes = 256;
constexpr int32_t kErrWaitTimeout = 1;

// Upper bound for one barrier wait. No legitimate wait in these kernels comes
// within orders of magnitude of it; reaching it means a lost arrival.
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // 1 s
// Outer polling rounds of one wait: a backstop should %globaltimer not advance. A failed
// try_wait without a suspend hint can return within tens of nanoseconds, so the cap is set
// for eight of them per round to outlast the 1 s time bound.
constexpr uint32_t kWaitMaxIters = 1u << 23;

__device__ __forceinline__ void report_error(int32_t* err, int32_t site, int32_t kind) {
    if (err != nullptr) atomicCAS(err, 0, (site << 8) | kind);
}

// Device-side index checks of a debug build (compiled with DIFFATTN_DEBUG_CHECKS;
// build(debug=True) makes libdiffattn_debug.so). A failed check records
// (site << 8) | kErrIndex in the error word; it never traps. The checked accesses
// are TMA coordinates, paged block-table entries and split ranges, all of which
// the hardware or the kernel already makes safe (an out-of-range TMA load reads
// zeros, a store past the tensor's end is clipped), so a failure is reported
// rather than skipped. In a release build index_ok compiles to `true`.
constexpr int32_t kErrIndex = 2;
#ifdef DIFFATTN_DEBUG_CHECKS
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif
__device__ __forceinline__ bool index_ok(bool cond, int32_t* err, int32_t site) {
    if constexpr (kDebugChecks) {
        if (!cond) {
            report_error(err, site, kErrIndex);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------------------------------
// mbarrier
// ----------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

constexpr uint32_t kSleepHintNs = 1000000;  // suspend hint of the cluster waits: 1 ms per attempt, bounded below

// Waits for the phase of `bar` with the given parity to complete.
// Gives up when *abort becomes non-zero (another role of the CTA failed) or
// after kWaitTimeoutNs; on a timeout it records `site` in the error word and
// raises *abort so the rest of the CTA stops too. Returns true on completion.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* err,
                                          int32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        // try_wait without a suspend-time hint: the hardware still suspends the thread
        // for a short while, and wakes it sooner than with a long hint (about 1% on the
        // prefill and backward kernels, whose critical paths are chains of these waits).
        for (int i = 0; i < 8; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (abort != nullptr && *abort) return false;
        // Time bound, with an iteration cap as a backstop should the timer not advance.
        if (globaltimer_ns() - t0 > kWaitTimeoutNs || it > kWaitMaxIters) {
            report_error(err, site, kErrWaitTimeout);
            if (abort != nullptr) *abort = 1;
            return false;
        }
    }
}

// ----------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), completion signalled on an mbarrier
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
        "[%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z,
                                            int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, "
        "%6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}

// TMA store of a shared-memory box to a 3-D / 2-D tensor (out-of-range rows are
// clipped by the hardware). The generic-proxy writes that filled the box must
// be fenced (fence_proxy_async_shared) and synchronised before the issuing
// thread calls this.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(map),
                 "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed store of this thread has finished reading shared memory.
__device__ __forceinline__ void tma_store_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Offset of 16-byte chunk c of row r in a 128-byte-swizzled [rows][128 B] box.
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// ----------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA
// ----------------------------------------------------------------------------
// Must be executed by one full warp; writes the TMEM base address to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Instruction descriptor for kind::f16 with an fp32 accumulator; A and B are
// both bf16 (ab_f16 = 0) or both fp16 (ab_f16 = 1). Bits: [4,6) D format
// (1 = f32), [7,10) A format, [10,13) B format (0 = f16, 1 = bf16), 15 A major
// (1 = MN-major), 16 B major, [17,23) N/8, [24,29) M/16.
__host__ __device__ constexpr uint32_t idesc_kind_f16(int M, int N, int a_mn_major, int b_mn_major, int ab_f16) {
    return (1u << 4) | (static_cast<uint32_t>(ab_f16 ? 0 : 1) << 7) | (static_cast<uint32_t>(ab_f16 ? 0 : 1) << 10) |
           (static_cast<uint32_t>(a_mn_major) << 15) | (static_cast<uint32_t>(b_mn_major) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn_major, int b_mn_major) {
    return idesc_kind_f16(M, N, a_mn_major, b_mn_major, 0);
}

// Shared-memory matrix descriptor, 128-byte swizzle. Fields: [0,14) start
// address >> 4, [16,30) leading byte offset >> 4, [32,46) stride byte offset
// >> 4, [46,48) descriptor version (1), [61,64) layout (2 = 128-byte swizzle).
// The swizzle pattern repeats every 1024 bytes, so tile bases are 1024-aligned.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// D[tmem] (+)= A[smem] * B[smem]; one thread issues.
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]; A is M lanes x K (16-bit values, two per column).
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on `bar` when all previously issued MMAs of this thread are done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Each thread of the warp reads 16 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Each thread of the warp writes 16 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Each thread of the warp writes 32 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Programmatic dependent launch (kernels started with launch_pdl). pdl_trigger lets the
// next kernel in the stream start its CTAs once every CTA of this grid has triggered or
// exited (so no CTA of this grid is still waiting for resources); pdl_wait blocks until
// the previous kernel in the stream has completed and its writes are visible (it returns
// at once without a programmatic predecessor). A kernel calls pdl_wait in every thread
// before it reads what an earlier kernel wrote and before it can exit, which keeps
// completion transitive along a chain of such launches.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Named barrier over `count` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Register reallocation between warpgroups (all 128 threads of a warpgroup
// execute it). An increase waits until other warpgroups have released enough
// registers of the block's launch allotment.
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// True in exactly one lane of the (fully converged) calling warp; the same
// lane each time for the same member mask. MMAs and the commits that track
// them are issued by that lane: a commit covers only its own thread's MMAs.
// Issuing from a converged warp this way is measurably cheaper than from a
// lone lane of a diverged warp (about 36 vs 63 cycles per tcgen05.mma).
__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred P1;\n\t"
        "elect.sync _|P1, %1;\n\t"
        "selp.b32 %0, 1, 0, P1;\n\t}"
        : "=r"(pred)
        : "r"(0xffffffffu));
    return pred != 0;
}

// mbar_wait whose result is the same in every lane of the warp: if any lane
// gave up, all lanes report failure (needed before warp-collective tcgen05 ops).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* err,
                                               int32_t site) {
    const bool ok = mbar_wait(bar, parity, abort, err, site);
    return __all_sync(0xffffffffu, ok);
}

// ----------------------------------------------------------------------------
// Thread-block clusters: rank, distributed shared memory, cluster barrier
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address (shared::cluster window) of the same offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t caddr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(caddr)
                 : "memory");
    return v;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t caddr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(caddr) : "memory");
    return v;
}
// Stores into a peer CTA's shared memory. Unlike remote loads they need no
// round trip, so a CTA pair exchanges data by pushing it (measured: pulling
// 64 KB with remote loads took ~12K cycles per pass).
__device__ __forceinline__ void st_dsmem_f4(uint32_t caddr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(caddr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_dsmem_f32(uint32_t caddr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(caddr), "f"(v) : "memory");
}
// Hardware cluster barrier. It has no bounded form, so it is used only where
// it depends on nothing but every CTA of the cluster having started (right
// after barrier initialisation, before any other wait).
__device__ __forceinline__ void cluster_sync_start() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster_local(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Arrive on the barrier at shared::cluster address `caddr` (another CTA's barrier).
__device__ __forceinline__ void mbar_arrive_cluster_remote(uint32_t caddr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded two-CTA rendezvous. `bar` (count 2) receives, per phase, one arrival
// from this CTA and one from the peer. Each thread's earlier shared-memory
// writes are released at cluster scope, so after it returns true the peer's
// writes before its matching call are visible. Returns false (error recorded,
// *abort raised) if the peer does not arrive within kWaitTimeoutNs.
__device__ __forceinline__ bool pair_sync(uint64_t* bar, uint32_t peer, uint32_t phase, volatile int* abort,
                                          int32_t* err, int32_t site) {
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_cluster_local(bar);
        mbar_arrive_cluster_remote(mapa_shared(smem_u32(bar), peer));
    }
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; !mbar_try_wait_cluster(bar, phase & 1, kSleepHintNs); ++it) {
        if (globaltimer_ns() - t0 > kWaitTimeoutNs || it > 8 * kWaitMaxIters) {
            report_error(err, site, kErrWaitTimeout);
            if (abort != nullptr) *abort = 1;
            return false;
        }
    }
    return true;
}

// ----------------------------------------------------------------------------
// Numeric helpers
// ----------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo_to_f32(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }

// Packs two floats as bf16 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Packs two floats as fp16 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Packs two floats as fp16 when `f16`, else as bf16 (16-bit outputs chosen at run time).
__device__ __forceinline__ uint32_t pack_16x2(float lo, float hi, bool f16) {
    return f16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
}

// P tile packing for an MMA operand of 16-bit type F16 ? fp16 : bf16.
template <bool F16>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
    if constexpr (F16) return pack_f16x2(lo, hi);
    else return pack_bf16x2(lo, hi);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

}  // namespace da
