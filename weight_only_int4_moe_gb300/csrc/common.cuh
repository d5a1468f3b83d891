// Device helpers shared by the kernels of the INT4 MoE library: inline-PTX
// wrappers for mbarriers, bulk/tensor async copies (TMA) and the tcgen05
// tensor-memory / MMA instructions of sm_100-family GPUs (built for sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#define MOE_DEV __device__ __forceinline__

namespace moe {

// Error word layout inside the workspace (uint32[2]): flags, dropped-pair count.
constexpr uint32_t kErrBadExpert = 0x1u;
constexpr uint32_t kErrTimeout = 0x2u;
constexpr uint32_t kErrBounds = 0x4u;
// A value left fp16's finite range on its way to an fp16 tensor-core operand
// (an x element or a SwiGLU intermediate beyond +-65504, infinite or NaN): it
// was saturated and the result is not valid.
constexpr uint32_t kErrRange = 0x8u;

// Records kErrRange once per warp if any lane saw an out-of-range value
// (whole-warp call).
MOE_DEV void report_range(bool bad, uint32_t *err) {
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0 && err) atomicOr(err, kErrRange);
}

// Two bf16 -> two fp16 (exact for magnitudes in [2^-14, 65504]; fp16
// subnormals below, within 2^-25); `bad` records a value beyond +-65504,
// infinite or NaN, which is saturated.
MOE_DEV uint32_t bf16x2_to_f16x2_sat(uint32_t v, bool &bad) {
    float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xFFFF0000u);
    bad |= !(fabsf(lo) <= 65504.0f) || !(fabsf(hi) <= 65504.0f);
    lo = fminf(fmaxf(lo, -65504.0f), 65504.0f);
    hi = fminf(fmaxf(hi, -65504.0f), 65504.0f);
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

MOE_DEV uint4 bf16x8_to_f16x8_sat(uint4 v, bool &bad) {
    v.x = bf16x2_to_f16x2_sat(v.x, bad);
    v.y = bf16x2_to_f16x2_sat(v.y, bad);
    v.z = bf16x2_to_f16x2_sat(v.z, bad);
    v.w = bf16x2_to_f16x2_sat(v.w, bad);
    return v;
}

// One row of H bf16 values to fp16 (the gate/up GEMM's B operand), copied by
// one warp with U 16-byte loads in flight per lane: a row takes
// ceil(H / (256 U)) dependent memory round trips.
template <int U>
MOE_DEV void gather_row(const uint16_t *src_row, uint16_t *dst_row, int H, bool &bad) {
    const uint4 *src = reinterpret_cast<const uint4 *>(src_row);
    uint4 *dst = reinterpret_cast<uint4 *>(dst_row);
    const int n8 = H / 8, lane = threadIdx.x & 31;
    for (int c0 = lane; c0 < n8; c0 += 32 * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (c0 + 32 * u < n8) v[u] = src[c0 + 32 * u];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (c0 + 32 * u < n8) dst[c0 + 32 * u] = bf16x8_to_f16x8_sat(v[u], bad);
    }
}

// ------------------------------------------------- hand-offs between CTAs --
// Acquire load at GPU scope (a counter that other CTAs release).
MOE_DEV int ld_acquire_gpu(const int32_t *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Release add at GPU scope.
MOE_DEV void red_release_gpu(int32_t *p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Orders this thread's generic-proxy global accesses with the async proxy's
// (TMA) accesses to global memory.
MOE_DEV void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Debug-bounds builds (-DMOE_DEBUG_BOUNDS) check the indices that kernels read
// back from the routing buffers (block count, expert ids, pair ids) before using
// them: a failed check records kErrBounds and the caller substitutes an
// in-range index, so no access leaves its buffer and no pipeline wait is left
// unanswered.  Other builds compile the checks away (bounds_ok is true).
#ifdef MOE_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif

// A pipeline wait that takes longer than this many SM cycles (about 2 s at the
// GB300's 2.07 GHz maximum clock) is treated as a kernel bug: the waiting role
// records kErrTimeout and the CTA winds down.  Debug-bounds builds give up
// after about 50 ms, so that their timeout test (a stage whose copy is never
// issued) ends quickly.
#ifdef MOE_DEBUG_BOUNDS
constexpr long long kWaitTimeoutCycles = 100000000ll;
#else
constexpr long long kWaitTimeoutCycles = 4000000000ll;
#endif

MOE_DEV bool bounds_ok(bool in_range, uint32_t *err) {
    if (!kDebugBounds) return true;
    if (!in_range && err) atomicOr(err, kErrBounds);
    return in_range;
}

MOE_DEV uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier --
MOE_DEV void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
MOE_DEV void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
MOE_DEV void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
MOE_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}
// try_wait with a suspend-time hint suspends the thread until the phase
// completes or kSuspendHintNs passes, so a waiting warp does not spin on the
// issue slots; but each call costs ~50 cycles alone and ~180 cycles on an SM
// sub-partition busy with other warps, even when the phase is already complete.
// Waits therefore test first without the hint and suspend only after that.
constexpr uint32_t kSuspendHintNs = 20000;

MOE_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}
MOE_DEV bool mbar_try_wait_nohint(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on the phase with the given parity: one test without the
// suspend hint (the common, already-complete case), then a few suspending
// polls; after that it sleeps `backoff_ns` between polls (0: keep polling, for
// waits on the critical path) and only then starts reading the cycle counter.
// Returns false (and records the timeout) if the wait gives up or another role
// of the CTA already aborted.
MOE_DEV bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, uint32_t *err,
                       uint32_t backoff_ns = 0, long long limit = kWaitTimeoutCycles) {
    if (mbar_try_wait_nohint(bar, parity)) return true;
#pragma unroll 1
    for (int it = 0; it < 8; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
#pragma unroll 1
    for (uint32_t round = 0; round < (1u << 24); ++round) {
#pragma unroll 1
        for (int it = 0; it < 16; ++it) {
            if (mbar_try_wait(bar, parity)) return true;
            if (backoff_ns) __nanosleep(backoff_ns);
        }
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) break;
    }
    *abort_flag = 1;
    if (err) atomicOr(err, kErrTimeout);
    return false;
}

// Shared-memory loads by 32-bit shared address (ld.shared: the short-latency
// path; a load through a generic pointer may be issued as a generic load).
// volatile: they must stay after the mbarrier wait that publishes the data.
MOE_DEV uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
MOE_DEV uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel of the stream still runs;
// it must call pdl_wait() before touching anything that kernel writes.
// pdl_launch_dependents() lets the next such kernel start its own set-up.
MOE_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Producer/consumer named barrier: arrive without waiting / wait for `threads`.
MOE_DEV void named_bar_arrive(uint32_t id, uint32_t threads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Position in a ring of n stages: index and the parity of the current lap.
struct Ring {
    uint32_t idx, ph, n;
    MOE_DEV explicit Ring(uint32_t n_) : idx(0), ph(0), n(n_) {}
    MOE_DEV void next() {
        if (++idx == n) {
            idx = 0;
            ph ^= 1u;
        }
    }
    // Moves k positions ahead (k >= 0; any number of laps).
    MOE_DEV void advance(uint32_t k) {
        idx += k;
        while (idx >= n) {
            idx -= n;
            ph ^= 1u;
        }
    }
};

// ------------------------------------------------------------- async copies --
MOE_DEV uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> shared through the TMA unit, completing on `bar`.
MOE_DEV void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                      uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// 2-D tiled tensor copy global -> shared (TMA), completing on `bar`.
MOE_DEV void tma_load_2d(uint32_t dst, const void *tmap, int32_t c0, int32_t c1,
                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

MOE_DEV void named_bar_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also returns the OR of `pred` over the participating
// threads (the same value in every thread).
MOE_DEV bool named_bar_or(uint32_t id, uint32_t threads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------------------ tcgen05 --
MOE_DEV void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     slot_smem),
                 "r"(ncols)
                 : "memory");
}
MOE_DEV void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}
MOE_DEV void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
MOE_DEV void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Warp-collective forms: every lane of the warp executes them with the same
// operands and elect.sync picks the one lane that issues.  (Issuing from
// warp-uniform code keeps the operands in uniform registers.)
// Arrive on `bar` once every tcgen05 async operation issued so far by the
// elected thread has completed.
MOE_DEV void tc_commit_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            bar)
        : "memory");
}

// Four kind::f16 MMAs along K (K = 16 each: A columns +8, B descriptor start
// +32 bytes) from one elected thread, then commits to bar1 and bar2 (each only
// if non-zero).  One elect and one instruction block per 64-wide k step keeps
// the issuing warp's instruction stream short while it shares its SM
// sub-partition with busy dequantising warps.  The first MMA accumulates iff
// `accumulate`.
MOE_DEV void mma_ts_f16_k64_commit(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                   uint32_t idesc, uint32_t accumulate, uint32_t bar1,
                                   uint32_t bar2) {
    asm volatile(
        "{\n\t.reg .pred p, t, e, c;\n\t.reg .b32 a1, a2, a3;\n\t.reg .b64 b1, b2, b3;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 t, %4, %4;\n\t"
        "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
        "add.u64 b1, %2, 2;\n\tadd.u64 b2, %2, 4;\n\tadd.u64 b3, %2, 6;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, t;\n\t"
        "setp.ne.and.b32 c, %5, 0, e;\n\t"
        "@c tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t"
        "setp.ne.and.b32 c, %6, 0, e;\n\t"
        "@c tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t}" ::"r"(
            d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(bar1), "r"(bar2)
        : "memory");
}

// Commits to bar1 and bar2 (each only if non-zero) from one elected thread.
MOE_DEV void tc_commit2_elect(uint32_t bar1, uint32_t bar2) {
    asm volatile(
        "{\n\t.reg .pred e, c;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.and.b32 c, %0, 0, e;\n\t"
        "@c tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t"
        "setp.ne.and.b32 c, %1, 0, e;\n\t"
        "@c tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%1];\n\t}" ::"r"(
            bar1),
        "r"(bar2)
        : "memory");
}

// Instruction descriptor of kind::f16: fp16 A and B (format code 0), fp32 D,
// both K-major, M = 128, N = n (multiple of 16, 16..256).
MOE_DEV uint32_t idesc_f16_m128(uint32_t n) {
    return (1u << 4)            // D format: f32
           | (0u << 7)          // A format: f16
           | (0u << 10)         // B format: f16
           | ((n >> 3) << 17)   // N / 8
           | ((128u >> 4) << 24);  // M / 16
}

// Shared-memory matrix descriptor: K-major operand with the 128-byte swizzle;
// rows of 128 bytes, 8-row atoms of 1024 bytes (stride byte offset 1024).
MOE_DEV uint64_t smem_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu)   // start address
           | ((uint64_t)1u << 16)               // leading byte offset (unused)
           | ((uint64_t)(1024u >> 4) << 32)     // stride byte offset
           | ((uint64_t)1u << 46)               // descriptor version
           | ((uint64_t)2u << 61);              // swizzle: 128 B
}

// 32 lanes x 32 consecutive 32-bit columns: each thread stores its lane's row,
// then waits for the store to complete.
MOE_DEV void tmem_st_32x32b_x32_wait(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
        "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
        "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]),
        "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]),
        "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// The same store without the wait (tmem_wait_st waits for all of a thread's).
MOE_DEV void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
        "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
        "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]),
        "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]),
        "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
MOE_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 16 consecutive 32-bit columns from one address, waited for inside
// the same asm statement so no use of the registers can precede the wait.
MOE_DEV void tmem_ld_32x32b_x16_wait(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, "
        "%9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Two 32x32b.x16 loads (two accumulators of the same lanes), one wait.
MOE_DEV void tmem_ld2_32x32b_x16_wait(uint32_t ta, uint32_t tb, float (&va)[16],
                                      float (&vb)[16]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, "
        "%9, %10, %11, %12, %13, %14, %15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, "
        "%24, %25, %26, %27, %28, %29, %30, %31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
          "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(ta), "r"(tb)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(r[16 + i]);
    }
}

}  // namespace moe
