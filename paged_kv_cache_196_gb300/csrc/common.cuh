// Device-side helpers shared by the kernels: mbarriers, bulk (TMA) copies,
// bfloat16 packing, bounded waits.  Inline PTX written for sm_100-family
// parts (built for sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "paged_kv.h"

#define KV_DEVICE __device__ __forceinline__

namespace pkv {

// A pipeline wait gives up after this many nanoseconds by default (then the
// kernel records KV_DEVERR_TIMEOUT and winds down instead of spinning forever).
constexpr unsigned long long kWaitLimitNs = KV_WAIT_LIMIT_DEFAULT_NS;

// The limit pipeline waits use: kWaitLimitNs unless a test shortened it
// (kv_debug_set_wait_limit_ns).  One copy per translation unit and device.
static __device__ unsigned long long g_wait_limit_ns = kWaitLimitNs;

// Host: sets this translation unit's copy of the limit on the current device.
static inline cudaError_t set_wait_limit_here(unsigned long long ns) {
    return cudaMemcpyToSymbol(g_wait_limit_ns, &ns, sizeof(ns));
}

KV_DEVICE uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

KV_DEVICE unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
KV_DEVICE void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

// Makes barrier initialisation visible to the async (TMA / tensor) proxy.
KV_DEVICE void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

KV_DEVICE void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

KV_DEVICE void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

KV_DEVICE bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false
// (after setting KV_DEVERR_TIMEOUT in *err) if it has not completed by the
// end of the first round of 64 polls that ends after limit_ns have passed
// since the first poll failed; with limit_ns = 0 the first failed poll gives
// up.  The clock is read only between rounds of polls.
KV_DEVICE bool mbar_wait_for(uint64_t *bar, uint32_t parity, int *err,
                             unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    if (limit_ns == 0) {
        if (err) atomicOr(err, KV_DEVERR_TIMEOUT);
        return false;
    }
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 >= limit_ns) {
            if (err) atomicOr(err, KV_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// A pipeline wait: data a producer has to deliver, a stage a consumer has to
// release.  TW = false (the kernels' ordinary instantiations): the limit is
// the compile-time kWaitLimitNs.  TW = true (the instantiations launched
// while a test has shortened the limit, kv_debug_set_wait_limit_ns): the
// limit is read from g_wait_limit_ns.  A run-time limit in every wait costs
// the register-bound kernels a few per cent, so it stays out of the
// ordinary instantiations.
template <bool TW = false>
KV_DEVICE bool mbar_wait(uint64_t *bar, uint32_t parity, int *err) {
    if constexpr (TW)
        return mbar_wait_for(bar, parity, err, g_wait_limit_ns);
    else
        return mbar_wait_for(bar, parity, err, kWaitLimitNs);
}

// A warp's wait for its own copies or tensor-core operations before it exits
// or its CTA frees what they write (shared or tensor memory): always the full
// default limit, whatever a test set for pipeline waits, so that nothing is
// still in flight when the CTA ends.
KV_DEVICE bool mbar_wait_drain(uint64_t *bar, uint32_t parity, int *err) {
    return mbar_wait_for(bar, parity, err, kWaitLimitNs);
}

// ------------------------------------------------------------ bulk copies
// One-dimensional bulk copy global -> shared, completion signalled on an
// mbarrier as transaction bytes.  dst, src 16-byte aligned; bytes % 16 == 0.
KV_DEVICE void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                        uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// L2 policy for data read exactly once (streamed KV).
KV_DEVICE uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Named barrier over a subset of warps.
KV_DEVICE void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also returns the OR of a flag over the participating
// threads, so that they all take the same decision.
KV_DEVICE bool named_bar_or(int id, int threads, bool flag) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)flag), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------- bf16
// A 32-bit word holding two bfloat16 values (low half = lower index).
// Widening bf16 -> fp32 is exact: the bf16 bits are the top half of fp32.
KV_DEVICE float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

KV_DEVICE float bf16_to_float(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

KV_DEVICE uint16_t float_to_bf16_rn(float f) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

KV_DEVICE float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// ---------------------------------------------------------------- fp16
// Two IEEE half-precision values (a 32-bit word, low half = lower index) as fp32
// (exact).
KV_DEVICE float2 f16x2_to_float2(uint32_t w) {
    float lo, hi;
    asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(w));
    return make_float2(lo, hi);
}

KV_DEVICE uint16_t float_to_f16_rn(float f) {
    uint16_t r;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

// One output element, stored as the call's output type (KV_F32, KV_BF16 or
// KV_F16; 16-bit outputs rounded to nearest even).
KV_DEVICE void store_out(void *out, size_t idx, float v, int out_type) {
    if (out_type == KV_F32)
        reinterpret_cast<float *>(out)[idx] = v;
    else if (out_type == KV_BF16)
        reinterpret_cast<uint16_t *>(out)[idx] = float_to_bf16_rn(v);
    else
        reinterpret_cast<uint16_t *>(out)[idx] = float_to_f16_rn(v);
}

}  // namespace pkv
