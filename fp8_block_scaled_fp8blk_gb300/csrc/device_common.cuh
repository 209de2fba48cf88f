// device_common.cuh -- sm_103a device primitives shared by the libfp8blk
// kernels: mbarrier + 1-D bulk-copy (TMA) pipeline pieces with bounded waits,
// programmatic-dependent-launch controls, and in-register format decoders.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8blk {

// Longest a kernel thread waits for a weight tile before giving up (ns).  A
// healthy tile lands in microseconds; on expiry the kernel records
// FP8BLK_STATUS_WAIT_TIMEOUT and returns instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes freshly initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

// Test-and-sleep: returns true once phase `parity` has completed; otherwise
// the thread sleeps up to kSuspendHintNs (or less, at the hardware's choice)
// without occupying issue slots, then returns false.
constexpr uint32_t kSuspendHintNs = 100000;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "n"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// try_wait without a suspend hint: returns after a short hardware-chosen
// interval; for a thread on the critical path that must react at once.
__device__ __forceinline__ bool mbar_try_wait_short(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of the barrier to complete, for at most
// kWaitLimitNs.  Returns false on expiry.  SLEEP = false polls without the
// suspend hint.
template <bool SLEEP = true>
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    auto poll = [&]() { return SLEEP ? mbar_try_wait(bar, parity) : mbar_try_wait_short(bar, parity); };
    if (poll()) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (poll()) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Non-blocking test of phase `parity` (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// A consumer's wait for a weight tile with a process-wide limit (set on the
// host, fp8blk_set_wait_limit).  At the default limit this is
// mbar_wait_bounded; a shorter limit polls without sleeping, so a limit of 0
// gives up unless the phase has already completed.  Drains of copies still in
// flight never use this: they keep the fixed kWaitLimitNs bound, so a CTA
// never exits with a copy landing in its shared memory.
template <bool SLEEP = true>
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (limit_ns >= kWaitLimitNs) return mbar_wait_bounded<SLEEP>(bar, parity);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_test_wait(bar, parity))
        if (global_timer_ns() - t0 >= limit_ns) return false;
    return true;
}

// Plain arrive (release) on a barrier, e.g. "this warp is done with a stage".
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// ---------------------------------------------------------------- bulk copy
// L2 policy for data read exactly once (weights): evict first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> shared, completing `bytes` of transaction count on
// `bar`.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Hint: bring `bytes` (multiple of 16, src 16-byte aligned) into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- PDL
// Programmatic dependent launch: wait for the preceding grid's memory to be
// visible / allow the next grid to start launching.  No-ops when the launch
// did not enable programmatic serialization.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- decoders
// Four e4m3 codes (bytes of `word`, lowest byte = lowest column) -> two f32
// pairs.  The hardware conversion e4m3 -> f16 is exact (every e4m3 value is an
// f16 value) and f16 -> f32 is exact, so each float equals e4m3(code).
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t word, float2 &lo, float2 &hi) {
    uint32_t h01, h23;
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(h01), "=r"(h23)
        : "r"(word));
    lo = __half22float2(*reinterpret_cast<const __half2 *>(&h01));
    hi = __half22float2(*reinterpret_cast<const __half2 *>(&h23));
}

// Two bf16 bit patterns (low half = lower column) -> f32 pair, exactly.
__device__ __forceinline__ float2 bf16x2_to_f32(uint32_t word) {
    return make_float2(__uint_as_float(word << 16), __uint_as_float(word & 0xFFFF0000u));
}

// Two e4m3 codes (low byte first) -> f32 pair, exactly.
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t pair16) {
    uint32_t h;
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t}"
        : "=r"(h)
        : "r"(pair16));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// Eight e2m1 codes (two per byte, low nibble = lower column) -> four f16x2
// words, exactly (every e2m1 value is an f16 value).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t word, uint32_t out[4]) {
    asm("{\n\t.reg .b8 a, b, c, d;\n\t"
        "mov.b32 {a, b, c, d}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, a;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, c;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, d;\n\t}"
        : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
        : "r"(word));
}

// Round two f32 to bf16 (nearest even) and pack, `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
    return r;
}

}  // namespace fp8blk
