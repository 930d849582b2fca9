// ptx.cuh — sm_103a device primitives written as inline PTX: mbarriers with
// bounded waits, TMA tile loads, tcgen05 tensor-memory allocation, MMA, loads
// and stores, and the shared-memory / instruction descriptors the MMA reads.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace gbattn {

// Device-side wait limit.  A wait that has not completed after this many
// nanoseconds of %globaltimer gives up, so a broken pipeline returns an error
// status instead of hanging the GPU.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Nanoseconds since t0, signed.  The timer follows a clock the driver may
// step: after a step backwards the difference is negative (the wait goes on
// for the size of the step) instead of wrapping to a huge unsigned value that
// would end every wait in flight at once.  Kept to one subtraction: extra
// code in these waits (re-basing t0, a poll counter) made the kernels 1-4%
// slower.
__device__ __forceinline__ long long elapsed_ns(unsigned long long t0) {
    return static_cast<long long>(globaltimer() - t0);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One arrival on behalf of the whole warp, counting 32: the warp barrier
// orders every lane's prior work (and its tcgen05 fences) before lane 0's
// arrival, which has release semantics.  The barrier's 32 arrivals then cost
// one shared-memory operation instead of 32.  Used for the forward's P
// barriers (C3 -0.9%, N = 16384 at d = 64 -2.1%); in the backward's compute
// and dQ warps it measured 0.6% (d = 128) and 3% (d = 256) slower.
__device__ __forceinline__ void mbar_arrive_warp(uint64_t* bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], 32;" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Single-thread bounded wait for the phase of `bar` with the given parity.
// Returns false (and raises *abort) when the limit expires or another role has
// already raised *abort.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (*abort) return false;
            if (elapsed_ns(t0) > static_cast<long long>(limit_ns)) {
                *abort = 1;
                return false;
            }
        }
    }
}

// Warp-collective bounded wait: every lane polls, and all lanes return the
// same answer, so the warp stays converged for the .sync.aligned tcgen05
// instructions that follow.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity,
                                               volatile int* abort,
                                               unsigned long long limit_ns = kWaitLimitNs) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 0;; ++it) {
        const bool ok = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        if ((it & 31u) == 31u) {
            int give_up = (*abort != 0) || (elapsed_ns(t0) > static_cast<long long>(limit_ns));
            give_up = __shfl_sync(0xffffffffu, give_up, 0);
            if (give_up) {
                *abort = 1;
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box into shared memory; completion is counted on `bar`
// in bytes.  c0 (innermost) must be a multiple of 16 bytes' worth of elements.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// 3-D tiled store of one box from shared memory (same box and swizzle as the
// map's loads).  Rows past the tensor's extent are not written.  Completion
// is tracked per thread with bulk groups: commit, then wait before the
// shared-memory source is reused or the CTA exits.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0,
                                             int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until every committed bulk store of this thread has finished reading
// shared memory.
__device__ __forceinline__ void bulk_wait_group_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the kernel before it in the stream is still
// running (once that one has signalled launch_dependents); grid_dep_wait()
// then blocks the calling thread until the preceding grid has completed and
// its memory operations are visible.  Every kernel here calls it before its
// first access to memory a preceding kernel may still write or read.  Only
// the backward's main kernel reads anything (its inputs) before that wait, so
// the preprocess launched just before it signals its dependents after its own
// wait; the main and dQ-conversion kernels signal at their start, the forward
// not at all.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Barrier over `nthreads` threads (a multiple of 32) on hardware barrier `id`
// (1-15; 0 is the one __syncthreads uses).
__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Untiled bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Fire-and-forget adds into global memory (no value comes back, so the issuing
// warp never waits on them).  red_add_v4 needs a 16-byte aligned address.
__device__ __forceinline__ void red_add_v4(float* gptr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(gptr), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void red_add_f32(float* gptr, float a) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(gptr), "f"(a) : "memory");
}

// Make generic-proxy writes to shared memory visible to the async proxy (MMA
// operand reads, TMA stores).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
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

// Arrive once on `bar` when every tcgen05 operation this thread has issued so
// far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T  (both operands through descriptors)
template <bool kTF32>
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    if constexpr (kTF32) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
    }
}

// D[tmem] (+)= A[tmem] * B[smem]^T  (A read from tensor memory)
template <bool kTF32>
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    if constexpr (kTF32) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
            "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate));
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
            "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate));
    }
}

// Runs of kind::f16 MMAs into one accumulator, each run issued from one PTX
// block.  The MMA warp shares its SM sub-partition with busy softmax / compute
// warps, so every instruction it issues costs several cycles; the products
// themselves are queued in order.  The descriptors advance by adding to their
// low 32 bits only (the 14-bit start-address field cannot carry out of them,
// see sdesc_adv): before MMA k (k >= 1) the A and B descriptors advance by
// A<k> and B<k> 16-byte units.  The first MMA accumulates into D when
// first_accumulates is non-zero, every later one does.
#define GBATTN_MMA_SS_HEAD                                                         \
    "{\n\t.reg .pred p, pt;\n\t.reg .b32 al, ah, bl, bh;\n\t.reg .b64 a, b;\n\t" \
    "setp.ne.b32 p, %4, 0;\n\tsetp.eq.u32 pt, 0, 0;\n\t"                           \
    "mov.b64 {al, ah}, %1;\n\tmov.b64 {bl, bh}, %2;\n\t"                          \
    "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
#define GBATTN_MMA_SS_STEP(ia, ib)                                                      \
    "add.u32 al, al, %" #ia ";\n\tadd.u32 bl, bl, %" #ib ";\n\t"                        \
    "mov.b64 a, {al, ah};\n\tmov.b64 b, {bl, bh};\n\t"                                   \
    "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"

template <uint32_t A1, uint32_t A2, uint32_t A3, uint32_t A4, uint32_t A5, uint32_t A6, uint32_t A7,
          uint32_t B1, uint32_t B2, uint32_t B3, uint32_t B4, uint32_t B5, uint32_t B6, uint32_t B7>
__device__ __forceinline__ void mma8_ss_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t first_accumulates) {
    asm volatile(GBATTN_MMA_SS_HEAD GBATTN_MMA_SS_STEP(5, 12) GBATTN_MMA_SS_STEP(6, 13)
                     GBATTN_MMA_SS_STEP(7, 14) GBATTN_MMA_SS_STEP(8, 15) GBATTN_MMA_SS_STEP(9, 16)
                         GBATTN_MMA_SS_STEP(10, 17) GBATTN_MMA_SS_STEP(11, 18) "}"
                 ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(first_accumulates),
                 "n"(A1), "n"(A2), "n"(A3), "n"(A4), "n"(A5), "n"(A6), "n"(A7),
                 "n"(B1), "n"(B2), "n"(B3), "n"(B4), "n"(B5), "n"(B6), "n"(B7));
}

template <uint32_t A1, uint32_t A2, uint32_t A3, uint32_t B1, uint32_t B2, uint32_t B3>
__device__ __forceinline__ void mma4_ss_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t first_accumulates) {
    asm volatile(GBATTN_MMA_SS_HEAD GBATTN_MMA_SS_STEP(5, 8) GBATTN_MMA_SS_STEP(6, 9)
                     GBATTN_MMA_SS_STEP(7, 10) "}"
                 ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(first_accumulates),
                 "n"(A1), "n"(A2), "n"(A3), "n"(B1), "n"(B2), "n"(B3));
}

// The TS form (A read from tensor memory): A advances by A_STEP columns and
// the B descriptor by B_STEP 16-byte units per MMA; kN MMAs (4 or 8).
#define GBATTN_MMA_TS_HEAD                                                         \
    "{\n\t.reg .pred p, pt;\n\t.reg .b32 at, bl, bh;\n\t.reg .b64 b;\n\t"        \
    "setp.ne.b32 p, %4, 0;\n\tsetp.eq.u32 pt, 0, 0;\n\t"                           \
    "mov.b32 at, %1;\n\tmov.b64 {bl, bh}, %2;\n\t"                                \
    "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
#define GBATTN_MMA_TS_STEP                                                             \
    "add.u32 at, at, %5;\n\tadd.u32 bl, bl, %6;\n\tmov.b64 b, {bl, bh};\n\t"          \
    "tcgen05.mma.cta_group::1.kind::f16 [%0], [at], b, %3, pt;\n\t"

template <int kN, uint32_t A_STEP, uint32_t B_STEP>
__device__ __forceinline__ void mma_run_ts_f16(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                               uint32_t idesc, uint32_t first_accumulates) {
    static_assert(kN == 4 || kN == 8, "runs of 4 or 8 MMAs");
    if constexpr (kN == 8)
        asm volatile(GBATTN_MMA_TS_HEAD GBATTN_MMA_TS_STEP GBATTN_MMA_TS_STEP GBATTN_MMA_TS_STEP
                         GBATTN_MMA_TS_STEP GBATTN_MMA_TS_STEP GBATTN_MMA_TS_STEP GBATTN_MMA_TS_STEP "}"
                     ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(first_accumulates),
                     "n"(A_STEP), "n"(B_STEP));
    else
        asm volatile(GBATTN_MMA_TS_HEAD GBATTN_MMA_TS_STEP GBATTN_MMA_TS_STEP GBATTN_MMA_TS_STEP "}"
                     ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(first_accumulates),
                     "n"(A_STEP), "n"(B_STEP));
}

// The same two products with 8-bit floating-point operands (kind::f8f6f4; the
// operand formats are in the instruction descriptor).
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Each lane of the warp reads 32 consecutive 32-bit columns of its own lane
// (lane = warp's 32-lane quarter + laneid).  Results are valid after
// tmem_ld_wait() followed by reg_fence().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Ties registers to the point after a tcgen05.wait::ld so the compiler cannot
// read them earlier.
template <int n>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[n]) {
#pragma unroll
    for (int i = 0; i < n; ++i) asm volatile("" : "+r"(r[i])::"memory");
}

// ---------------------------------------------------------------------------
// Descriptors
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile whose
// 1024-byte swizzle atoms start 1024-byte aligned.
//   K-major (rows of 128 bytes along K): sbo = byte distance between
//     consecutive groups of 8 rows; lbo unused (encoded as 16 bytes).
//   MN-major (128 bytes along M/N per K row): lbo = byte distance between
//     consecutive 128-byte column blocks along M/N; sbo = byte distance
//     between consecutive groups of 8 K rows.
// Fields: start address >> 4 in bits 0-13, lbo >> 4 in bits 16-29,
// sbo >> 4 in bits 32-45, descriptor version 1 in bits 46-47, base offset 0,
// swizzle mode "128B" (2) in bits 61-63.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// The same descriptor moved `bytes` (a multiple of 16) further into shared
// memory: only the start-address field changes, and it cannot carry out of its
// 14 bits for addresses inside the 228 KB window.
__device__ __forceinline__ uint64_t sdesc_adv(uint64_t desc, uint32_t bytes) {
    return desc + static_cast<uint64_t>(bytes >> 4);
}

// Operand format codes of the instruction descriptor (A and B always share
// one).  kind::f16 and kind::tf32 use the first three; under kind::f8f6f4
// code 0 means e4m3.
constexpr uint32_t kFmtF16 = 0, kFmtBF16 = 1, kFmtTF32 = 2, kFmtE4M3 = 0;

// Instruction descriptor for kind::f16 (f16 or bf16 operands) and kind::tf32,
// fp32 accumulator, dense: D format (bits 4-5) = f32, A and B formats (bits
// 7-9, 10-12) = fmt, A/B major bits 15/16 (0 = K-major, 1 = MN-major), N >> 3
// in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f32acc(int M, int N, uint32_t fmt, bool a_mn_major,
                                                    bool b_mn_major) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(a_mn_major) << 15) |
           (static_cast<uint32_t>(b_mn_major) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// CTA schedule
// ---------------------------------------------------------------------------
// Maps a linear CTA index over (heads x blocks) to (head, rank) so that the
// CTAs resident at one time work on a group of at most kHeadGroup heads
// (their tiles and accumulators stay in L2) and, inside a group, CTAs of rank
// 0 (the caller makes rank 0 the heaviest block) start first.
constexpr int kHeadGroup = 16;
__device__ __forceinline__ void grouped_schedule(int x, int BH, int nblk, int& bh, int& rank) {
    const int grp = x / (kHeadGroup * nblk);
    const int g0 = grp * kHeadGroup;
    const int gsize = min(kHeadGroup, BH - g0);
    const int r = x - grp * kHeadGroup * nblk;
    rank = r / gsize;
    bh = g0 + r % gsize;
}

// ---------------------------------------------------------------------------
// Small numeric helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Three-input maximum (sm_100+).
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Packed pairs of fp32 in one 64-bit register and the sm_100 paired
// arithmetic on them (one instruction for both lanes of the pair).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Two floats -> packed bf16x2 (round to nearest even); `lo` in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) {
    return __uint_as_float(v & 0xFFFF0000u);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float f16lo_to_f32(uint32_t v) {
    float r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}" : "=f"(r) : "r"(v));
    return r;
}
__device__ __forceinline__ float f16hi_to_f32(uint32_t v) {
    float r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, hi;\n\t}" : "=f"(r) : "r"(v));
    return r;
}

// The 16-bit storage types (bf16 or f16, chosen by kF16): two floats packed
// with round-to-nearest-even, the low / high half widened back to float, and
// the tcgen05 operand format code.
template <bool kF16>
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    if constexpr (kF16) return pack_f16x2(lo, hi);
    else return pack_bf16x2(lo, hi);
}
template <bool kF16>
__device__ __forceinline__ float h2lo_to_f32(uint32_t v) {
    if constexpr (kF16) return f16lo_to_f32(v);
    else return bf16lo_to_f32(v);
}
template <bool kF16>
__device__ __forceinline__ float h2hi_to_f32(uint32_t v) {
    if constexpr (kF16) return f16hi_to_f32(v);
    else return bf16hi_to_f32(v);
}
template <bool kF16>
constexpr uint32_t fmt16() { return kF16 ? kFmtF16 : kFmtBF16; }

// Four floats rounded to e4m3 (round to nearest even, saturating to +-448)
// packed into one word, a in the low byte: the layout in which an 8-bit A
// operand is read from tensor memory (consecutive K elements from the low
// byte up).
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

}  // namespace gbattn
