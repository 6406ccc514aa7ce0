// Device-side helpers shared by the cq kernels: block-format constants,
// binary16 loads, and thin inline-PTX wrappers for mbarriers and the bulk
// (TMA, one-dimensional) global->shared copy engine of sm_90+/sm_100+.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "cq.h"

namespace cq {

// Bytes per 256-element chunk (eight 32-blocks or one superblock).
constexpr int CHUNK_ELEMS = 256;
constexpr int WCHUNK_Q4_0 = 8 * 18;   // 144
constexpr int WCHUNK_Q4_1 = 8 * 20;   // 160
constexpr int WCHUNK_Q8_0 = 8 * 34;   // 272
constexpr int WCHUNK_Q4_K = 144;
constexpr int WCHUNK_Q5_K = 176;
constexpr int WCHUNK_Q6_K = 210;
constexpr int ACHUNK_Q8_0 = 8 * 34;   // 272
constexpr int ACHUNK_Q8_1 = 8 * 36;   // 288
constexpr int ACHUNK_Q8_K = 292;

__host__ __device__ constexpr int wchunk_bytes(int fmt) {
    return fmt == CQ_Q4_0 ? WCHUNK_Q4_0 : fmt == CQ_Q4_1 ? WCHUNK_Q4_1 : fmt == CQ_Q8_0 ? WCHUNK_Q8_0
         : fmt == CQ_Q4_K ? WCHUNK_Q4_K : fmt == CQ_Q5_K ? WCHUNK_Q5_K : fmt == CQ_Q6_K ? WCHUNK_Q6_K : 0;
}
__host__ __device__ constexpr int act_fmt_for(int wfmt) {
    return wfmt == CQ_Q4_0 || wfmt == CQ_Q8_0 ? CQ_Q8_0 : wfmt == CQ_Q4_1 ? CQ_Q8_1
         : wfmt == CQ_Q4_K || wfmt == CQ_Q5_K || wfmt == CQ_Q6_K ? CQ_Q8_K : -1;
}
__host__ __device__ constexpr int achunk_bytes(int afmt) {
    return afmt == CQ_Q8_0 ? ACHUNK_Q8_0 : afmt == CQ_Q8_1 ? ACHUNK_Q8_1 : afmt == CQ_Q8_K ? ACHUNK_Q8_K : 0;
}

// One int8 quant of a Q8 block: round(v * id) to nearest, ties away from
// zero, clamped to [-127, 127]; id = 1/d, d = amax / 127, all fp32 RN.
__device__ __forceinline__ int quant_q8(float v, float id) {
    float r = roundf(__fmul_rn(v, id));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return static_cast<int>(r);
}
__device__ __forceinline__ float q8_scale(float amax) { return __fdiv_rn(amax, 127.0f); }
__device__ __forceinline__ float q8_inv(float d) { return d != 0.0f ? __frcp_rn(d) : 0.0f; }

__device__ __forceinline__ float h2f(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xffffu)));
}

// Four signed bytes (q - 8) from four nibbles 0..15 held one per byte:
// q + 0x78 stays below 0x100, and flipping bit 7 maps it to (q - 8) mod 256.
__device__ __forceinline__ int nib_minus8(uint32_t nibs) {
    return static_cast<int>((nibs + 0x78787878u) ^ 0x80808080u);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch. pdl_trigger lets the next grid in the stream
// begin launching (its CTAs take SM resources as this grid's CTAs leave; its
// own griddepcontrol.wait still waits for this grid to complete). pdl_wait
// returns once the grids this one depends on have completed and their writes
// are visible (at once for a grid launched without such a dependency): no
// kernel reads or writes global memory before it, except the GEMV's weight
// prefetches -- into L2 always (L2 is coherent, so nothing stale can reach
// shared memory through it), into shared memory only under the
// weights-constant option.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
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
// A flag word in this CTA's shared memory, read and written with explicit
// shared-space instructions: a pointer rebuilt from an aligned integer address
// would otherwise be accessed as generic memory, a long-latency load on every
// check.
struct SmemFlag {
    uint32_t addr;
    __device__ __forceinline__ int get() const {
        int v;
        asm volatile("ld.volatile.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
        return v;
    }
    __device__ __forceinline__ void set(int v) const {
        asm volatile("st.volatile.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
    }
};

// try_wait with a suspend-time hint: a thread whose phase is not complete is
// parked by the hardware until it completes or about hint_ns pass, instead of
// returning at once -- waiting warps then take no issue slots from the warps
// doing work on the same scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
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

// Bounded wait that parks between checks (see mbar_try_wait_sleep): gives up
// after `limit_ns` of wall time and returns false.
__device__ __forceinline__ bool mbar_wait_bounded_sleep(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Bounded wait for a phase to complete: gives up after `limit_ns` of wall
// time (checked every 256 polls) and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// One-dimensional bulk copy global -> this CTA's shared memory, completing
// `bytes` transactions on `bar`. Addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
// 4-byte asynchronous copy global -> shared, zero-filled when src_bytes is 0
// (src must still be a valid address). Complete once the issuing thread has
// passed cp_async_wait_all; only that thread's own copies are covered.
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Prefetch [gsrc, gsrc + bytes) from global memory into L2 (no completion to
// wait for). Address 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// L2 policy for data many CTAs re-read (kept ahead of streamed weights).
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Wall-time limit of any copy-completion wait (a copy that has not landed by
// then never will): the kernel flags CQ_DEV_WAIT_TIMEOUT and stops.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

}  // namespace cq
