// Device helpers shared by the librapid kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#define RAPID_DEVICE __device__ __forceinline__

namespace rapid {

// Bits of the sticky per-device error word (defined in capi.cu; kernels get
// its address as a parameter and only ever OR bits into it; the host reads
// and clears it through rapid_device_error()).
enum : unsigned int { kErrWaitTimeout = 1u, kErrBadInput = 2u };

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

RAPID_DEVICE float to_float(float x) { return x; }
RAPID_DEVICE float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> RAPID_DEVICE T from_float(float x);
template <> RAPID_DEVICE float from_float<float>(float x) { return x; }
template <> RAPID_DEVICE __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

RAPID_DEVICE float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
RAPID_DEVICE float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------------------
// Packed fp32 pairs (f32x2 arithmetic: one instruction for two lanes of work).
// ---------------------------------------------------------------------------
RAPID_DEVICE uint64_t pack2(float2 v) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
    return r;
}
RAPID_DEVICE float2 unpack2(uint64_t r) {
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
RAPID_DEVICE float2 mul2(float2 a, float2 b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack2(a)), "l"(pack2(b)));
    return unpack2(d);
}
RAPID_DEVICE float2 add2(float2 a, float2 b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack2(a)), "l"(pack2(b)));
    return unpack2(d);
}
RAPID_DEVICE float2 fma2(float2 a, float2 b, float2 c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pack2(a)), "l"(pack2(b)), "l"(pack2(c)));
    return unpack2(d);
}

// ---------------------------------------------------------------------------
// Philox4x32-10 counter-based generator (Salmon, Moraes, Dror, Shaw, "Parallel
// Random Numbers: As Easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64-bit
// multiplies and xors, key advanced by two Weyl constants per round.
// ---------------------------------------------------------------------------
struct Philox4 {
    uint32_t w[4];
};

RAPID_DEVICE Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                   uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t a0 = 0xD2511F53u * c0;            // low half of M0 * c0
        const uint32_t b0 = __umulhi(0xD2511F53u, c0);   // high half
        const uint32_t a1 = 0xCD9E8D57u * c2;
        const uint32_t b1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = b1 ^ c1 ^ k0;
        const uint32_t n2 = b0 ^ c3 ^ k1;
        c0 = n0;
        c1 = a1;
        c2 = n2;
        c3 = a0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    Philox4 r;
    r.w[0] = c0; r.w[1] = c1; r.w[2] = c2; r.w[3] = c3;
    return r;
}

// Uniform in [0, 1) from the top 24 bits of a word (exact in float).
RAPID_DEVICE float word_uniform(uint32_t w) { return (float)(w >> 8) * (1.0f / 16777216.0f); }

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start while its predecessor in the stream is finishing;
// griddep_wait() blocks until that predecessor has completed and its memory
// is visible, so every kernel calls it before its first read of an input.
// griddep_launch_dependents() lets the next kernel be scheduled early.
// ---------------------------------------------------------------------------
RAPID_DEVICE void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
RAPID_DEVICE void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// mbarrier + bulk-copy (TMA) primitives, inline PTX.
// ---------------------------------------------------------------------------
RAPID_DEVICE uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

RAPID_DEVICE void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

RAPID_DEVICE void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

RAPID_DEVICE void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

RAPID_DEVICE void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

RAPID_DEVICE void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Non-blocking test of phase `parity` (mbarrier.test_wait never suspends the
// thread, so a caller's own time limit really bounds the wait).
RAPID_DEVICE bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

RAPID_DEVICE uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Default wall-clock bound of one wait.  Legitimate waits last microseconds;
// one second means the producer of the phase is gone.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Bounded wait on phase `parity` of an mbarrier: gives up after `limit_ns` of
// wall-clock time (globaltimer), records kErrWaitTimeout in err[0] and, if it
// is the first failure, `code` in err[1], and returns false.  Every wait on an
// mbarrier in this library goes through it.
RAPID_DEVICE bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* err,
                            unsigned int code = 0, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) break;
    }
    if (err) {
        atomicOr(err, kErrWaitTimeout);
        atomicCAS(err + 1, 0u, code | 0x80000000u);
    }
    return false;
}

// Blocking test of phase `parity` that suspends the thread for at most
// `hint_ns` (mbarrier.try_wait with an explicit suspend-time hint), so a
// waiting warp does not spin on issue slots.
RAPID_DEVICE bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait like mbar_wait, but sleeping between polls.
RAPID_DEVICE bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, unsigned int* err,
                                  unsigned int code = 0, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (global_timer_ns() - t0 > limit_ns) break;
    }
    if (err) {
        atomicOr(err, kErrWaitTimeout);
        atomicCAS(err + 1, 0u, code | 0x80000000u);
    }
    return false;
}

// 1-D bulk copy global -> shared memory of this CTA, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
RAPID_DEVICE void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// bulk_g2s with an L2 cache policy (for example evict-first for data that is
// read once, so that its stream does not push other data and code out of L2).
RAPID_DEVICE void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// L2 policy for data read once: its lines are the first to be evicted.
RAPID_DEVICE uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk prefetch of global memory into L2 (no completion to wait for).
// src 16-byte aligned; bytes a multiple of 16.
RAPID_DEVICE void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

}  // namespace rapid
