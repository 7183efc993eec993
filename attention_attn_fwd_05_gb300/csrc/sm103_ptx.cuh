// sm103_ptx.cuh -- inline-PTX wrappers for the Blackwell (sm_103a) features the
// attention kernels use: mbarriers, TMA tensor copies, tcgen05 tensor-core
// MMAs with TMEM accumulators, and a bounded barrier wait.
//
// Every wait in the kernels goes through bounded_wait(): if a barrier does not
// complete within the launch's time limit, the waiting thread records a
// timeout bit in the device status word, raises the CTA's abort flag and
// returns false, so the kernel can wind down and exit instead of hanging.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace attn {

// ------------------------------------------------------------ addresses ---

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------- mbarrier ---

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Non-blocking probe: has the phase with parity `parity` completed?
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Per-CTA control block for bounded waits.
struct WaitCtl {
    volatile uint32_t *abort;  // shared-memory flag, non-zero once any thread gave up
    uint32_t *status;          // device status word (global)
    uint64_t timeout_ns;       // limit for one wait
};

// Status bits recorded in the device status word.
enum : uint32_t {
    STATUS_TIMEOUT = 1u << 0,
    STATUS_BOUNDS = 1u << 1,  // debug build only: an index or TMA coordinate out of range
};

// Bounds checks of the debug build (compiled with -DATTN_DEBUG_BOUNDS): before
// a global access or a TMA copy the kernels test its index or coordinates
// against the tensor's extent (B*H, N, d).  A failed test records
// STATUS_BOUNDS in the status word and the access is skipped (a skipped TMA
// load then leaves its barrier incomplete, and the bounded wait on it reports
// a timeout as well); nothing traps.  In the normal build every check is the
// constant true and costs nothing.
#ifdef ATTN_DEBUG_BOUNDS
static __device__ __noinline__ bool bounds_fail(uint32_t *status) {
    atomicOr(status, STATUS_BOUNDS);
    __threadfence();
    return false;
}
#define ATTN_IN_BOUNDS(cond, status) ((cond) ? true : ::attn::bounds_fail(status))
#else
#define ATTN_IN_BOUNDS(cond, status) true
#endif

// Slow path of bounded_wait (kept out of line so the fast path stays a
// single try_wait): keep polling; every 64 polls look at the abort flag, the
// status word and the clock.
static __device__ __noinline__ bool bounded_wait_slow(uint32_t bar, uint32_t parity, const WaitCtl ctl) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63u) == 0u) {
            if (*ctl.abort) return false;
            // A timeout recorded by any CTA (this launch or an earlier one whose
            // status has not been read yet) makes every later wait give up at
            // once, so a broken launch winds down in one time limit, not one
            // per CTA.
            if (*reinterpret_cast<volatile uint32_t *>(ctl.status) & STATUS_TIMEOUT) {
                *ctl.abort = 1u;
                return false;
            }
            if (globaltimer_ns() - t0 > ctl.timeout_ns) {
                *ctl.abort = 1u;
                atomicOr(ctl.status, STATUS_TIMEOUT);
                __threadfence();
                return false;
            }
        }
    }
}

// Wait for the phase with parity `parity` of barrier `bar` to complete.
// Returns true when it did; false if the wait ran out of time (the timeout is
// recorded) or another thread of the CTA already gave up.  A phase that is
// already complete costs one try_wait.
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, const WaitCtl &ctl) {
    if (mbar_try_wait(bar, parity)) return true;
    return bounded_wait_slow(bar, parity, ctl);
}

// A bounded wait that never suspends: polls with the non-blocking
// mbarrier.test_wait, and every 256 polls looks at the abort flag, the status
// word and the clock like bounded_wait_slow.  For the single MMA-issuing
// thread, whose reaction to a completed phase is on the critical path:
// mbarrier.try_wait may suspend the thread, and measured on GB300 it took the
// issuer a few hundred cycles to notice that the softmax warps had arrived.
__device__ __forceinline__ bool spin_wait(uint32_t bar, uint32_t parity, const WaitCtl &ctl) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((n & 255u) == 0u) {
            if (*ctl.abort) return false;
            if (*reinterpret_cast<volatile uint32_t *>(ctl.status) & STATUS_TIMEOUT) {
                *ctl.abort = 1u;
                return false;
            }
            if (globaltimer_ns() - t0 > ctl.timeout_ns) {
                *ctl.abort = 1u;
                atomicOr(ctl.status, STATUS_TIMEOUT);
                __threadfence();
                return false;
            }
        }
    }
}

// The same wait for a whole warp: lane 0 polls, the others wait at the
// shuffle, and every lane gets lane 0's answer.  Call from all 32 lanes.
__device__ __forceinline__ bool bounded_wait_warp(uint32_t bar, uint32_t parity,
                                                  const WaitCtl &ctl) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = bounded_wait(bar, parity, ctl);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// ------------------------------------------------ clusters and DSMEM ---
//
// Distributed shared memory between the CTAs of a thread-block cluster on
// this GPU: a CTA maps an address of its own shared memory to the same
// address in cluster CTA `rank` (mapa), stores there, and arrives on an
// mbarrier there; the owner waits on its own barrier with cluster-scope
// acquire, which makes the stores that came before the arrivals visible.

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t map_shared_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f32x2(uint32_t addr, float a, float b) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b)
                 : "memory");
}
__device__ __forceinline__ void st_cluster_f32x4(uint32_t addr, float a, float b, float c,
                                                 float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}
// Arrive on an mbarrier of a cluster CTA (address from map_shared_to_rank),
// releasing this thread's earlier stores at cluster scope.
__device__ __forceinline__ void arrive_remote(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ bool try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Every thread of every CTA of the cluster (unbounded: only where every path
// of every CTA reaches it).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}
// Bounded wait on a barrier that other CTAs of the cluster arrive on: gives up
// after `timeout_ns`, or at once when a timeout is already recorded.
static __device__ __noinline__ bool wait_cluster_bounded(uint32_t bar, uint32_t parity,
                                                         uint32_t *status, uint64_t timeout_ns) {
    if (try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (try_wait_cluster(bar, parity)) return true;
        if ((n & 63u) == 0u) {
            if (*reinterpret_cast<volatile uint32_t *>(status) & STATUS_TIMEOUT) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                atomicOr(status, STATUS_TIMEOUT);
                __threadfence();
                return false;
            }
        }
    }
}

// ------------------------------------------------------------------ TMA ---

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Same, with an L2 cache-policy hint (K/V tiles are re-read by other CTAs).
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const void *tmap, int x, int y,
                                                 int z, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Bring one box of a tensor map into L2 (no shared memory, no barrier).
// Untiled bulk copy of `bytes` (a multiple of 16) from global memory to this
// CTA's shared memory, completing on mbarrier `bar` (both addresses 16-byte
// aligned).
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_l2_3d(const void *tmap, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void tma_store_3d(const void *tmap, uint32_t src, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_store_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk store has finished reading shared memory.
__device__ __forceinline__ void tma_store_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy reads of them (TMA stores, tcgen05 MMAs).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------- tcgen05 ---

// Allocate `ncols` TMEM columns (power of two >= 32); the base address is
// written to shared memory at `dst`.  Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 operands, fp32 accumulator).
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One 128 x N x (16*KSTEPS) GEMM as KSTEPS back-to-back tcgen05.mma (kind::f16)
// from shared-memory descriptors.  Step k uses a_desc + a_off[k] and
// b_desc + b_off[k] (16-byte units added to the start-address field).  The
// first step overwrites D unless `accumulate`; later steps accumulate.
#define ATTN_MMA_SS_STEP(K, AOFF, BOFF)                                               \
    "add.s64 a, %1, " #AOFF ";\n\tadd.s64 b, %2, " #BOFF ";\n\t"                        \
    "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, " K ";\n\t"
__device__ __forceinline__ void gemm_ss_k8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    // K-major 128-byte-swizzled operands: steps 0-3 walk 32 B within the first
    // 64-column block, steps 4-7 the same in the block 16 KB further on.
    asm volatile(
        "{\n\t.reg .pred pf, pt;\n\t.reg .b64 a, b;\n\t"
        "setp.ne.b32 pf, %4, 0;\n\tsetp.eq.b32 pt, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
        ATTN_MMA_SS_STEP("pt", 2, 2) ATTN_MMA_SS_STEP("pt", 4, 4) ATTN_MMA_SS_STEP("pt", 6, 6)
        ATTN_MMA_SS_STEP("pt", 1024, 1024) ATTN_MMA_SS_STEP("pt", 1026, 1026)
        ATTN_MMA_SS_STEP("pt", 1028, 1028) ATTN_MMA_SS_STEP("pt", 1030, 1030)
        "}\n" ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void gemm_ss_k4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred pf, pt;\n\t.reg .b64 a, b;\n\t"
        "setp.ne.b32 pf, %4, 0;\n\tsetp.eq.b32 pt, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
        ATTN_MMA_SS_STEP("pt", 2, 2) ATTN_MMA_SS_STEP("pt", 4, 4) ATTN_MMA_SS_STEP("pt", 6, 6)
        "}\n" ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
#undef ATTN_MMA_SS_STEP

// 128 x N x 128 GEMM with A in TMEM (bf16 pairs, 8 columns per 16-wide step)
// and B an MN-major shared-memory operand advancing 2048 B (16 rows of 128 B)
// per step.
#define ATTN_MMA_TS_STEP(ACOL, BOFF)                                                  \
    "add.u32 ta, %1, " #ACOL ";\n\tadd.s64 b, %2, " #BOFF ";\n\t"                       \
    "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %3, pt;\n\t"
__device__ __forceinline__ void gemm_ts_k8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred pf, pt;\n\t.reg .b64 b;\n\t.reg .b32 ta;\n\t"
        "setp.ne.b32 pf, %4, 0;\n\tsetp.eq.b32 pt, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pf;\n\t"
        ATTN_MMA_TS_STEP(8, 128) ATTN_MMA_TS_STEP(16, 256) ATTN_MMA_TS_STEP(24, 384)
        ATTN_MMA_TS_STEP(32, 512) ATTN_MMA_TS_STEP(40, 640) ATTN_MMA_TS_STEP(48, 768)
        ATTN_MMA_TS_STEP(56, 896)
        "}\n" ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
#undef ATTN_MMA_TS_STEP

// Arrive (once) on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Instruction descriptor for kind::f16 with bf16 A/B and an fp32 accumulator
// (bit layout of the tcgen05 instruction descriptor: D format at bit 4,
// A/B formats at bits 7 and 10, A/B major-ness at bits 15/16, N>>3 at bit 17,
// M>>4 at bit 24).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major,
                                                      bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (16-byte units), descriptor version 1, layout 2.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld_x32(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]) :: "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]) : "memory");
}
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld_x16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]) :: "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]) : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// --------------------------------------------------------------- math ---

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Pack two floats into a bf16x2 word (round to nearest even), lo in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Packed fp32 pair arithmetic (Blackwell f32x2 instructions): two lanes of
// work per instruction issue.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// a * b + c on both halves.
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace attn
