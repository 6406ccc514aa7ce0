// Thin inline-PTX wrappers for the sm_100-family tensor-core path: TMEM
// allocation, tcgen05.mma (kind::f16) issue and commit, TMEM loads/stores,
// 2-D TMA tile loads, and the shared-memory matrix descriptors.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>

#include "cq_device.cuh"

namespace cq {
namespace tc {

// ------------------------------------------------------------------ TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Byte offset of element (r, k) in a K-major, no-swizzle operand tile whose
// rows hold kt fp16 elements: 8-row x 16-byte core matrices, adjacent along K
// 128 bytes apart, 8-row groups kt * 16 bytes apart (the smem_desc below with
// lbo = 128, sbo = kt * 16).
__host__ __device__ constexpr int tile_off(int r, int k, int kt) {
    return (r >> 3) * (kt * 16) + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

// Byte offset of element (r, k) in a K-major operand tile with the 128-byte
// swizzle, rows of kt fp16 elements (kt a multiple of 64) for nr rows: the
// tile is kt / 64 column blocks of nr 128-byte rows (64 elements each), block
// b at b * nr * 128; inside a block the 16-byte chunk c of row r sits at
// chunk position c ^ (r % 8) (the smem_desc_sw128 below, sbo = 1024, on a
// 1024-byte aligned base).
__host__ __device__ constexpr int tile_off_sw128(int r, int k, int nr) {
    return (k >> 6) * (nr * 128) + r * 128 + ((((k >> 3) & 7) ^ (r & 7)) << 4) + (k & 7) * 2;
}

// Four signed bytes -> two half2 holding the same integers, in byte order
// (bytes 0, 1 | bytes 2, 3): the sign bits flipped (b + 128 as an unsigned
// byte), each byte placed under a 0x64 high byte (binary16 1024 + (b + 128),
// exact), then 1152 subtracted. The operand conversion of int8 quants.
__device__ __forceinline__ void s8x4_half(uint32_t w, uint32_t& o0, uint32_t& o1) {
    const __half2 k1152 = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const uint32_t u = w ^ 0x80808080u;
    uint32_t p01 = __byte_perm(u, 0x64646464u, 0x4140), p23 = __byte_perm(u, 0x64646464u, 0x4342);
    __half2 r01 = __hsub2(*reinterpret_cast<const __half2*>(&p01), k1152);
    __half2 r23 = __hsub2(*reinterpret_cast<const __half2*>(&p23), k1152);
    o0 = *reinterpret_cast<const uint32_t*>(&r01);
    o1 = *reinterpret_cast<const uint32_t*>(&r23);
}

// A role's bounded wait: on timeout it raises the CTA's abort flag and the
// library status bit, so the other roles leave their loops too.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, SmemFlag flag, int* status) {
    if (mbar_wait_bounded(bar, parity, WAIT_LIMIT_NS)) return true;
    flag.set(1);
    atomicOr(status, CQ_DEV_WAIT_TIMEOUT);
    return false;
}
// The same, parked between checks (mbar_wait_bounded_sleep): for roles that
// share their schedulers with busy warps.
__device__ __forceinline__ bool wait_or_abort_sleep(uint64_t* bar, uint32_t parity, SmemFlag flag, int* status) {
    if (mbar_wait_bounded_sleep(bar, parity, WAIT_LIMIT_NS)) return true;
    flag.set(1);
    atomicOr(status, CQ_DEV_WAIT_TIMEOUT);
    return false;
}

// ---------------------------------------------------------------- cluster
// This CTA's rank in its cluster.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of `local` (a shared::cta address) in the CTA
// of rank `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local), "r"(rank));
    return a;
}
// Every thread of every CTA of the cluster: arrive (release) and wait
// (acquire). Orders barrier initialisation before peers' remote operations,
// and keeps a CTA's shared memory alive until its peers are done with it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// this CTA's shared memory to a peer's (dst and its barrier as
// shared::cluster addresses), completing `bytes` transactions on that barrier.
__device__ __forceinline__ void bulk_s2peer(uint32_t dst, const void* src, uint32_t bytes, uint32_t peer_bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "r"(smem_u32(src)), "r"(bytes), "r"(peer_bar)
                 : "memory");
}
// Raise the expected transaction count of the barrier's current phase
// without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------- MMA
// D[tmem] (+)= A[smem] * B[smem]^T, fp16 operands, fp32 accumulator.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// The same, arriving on the barrier at this offset in every CTA of the
// cluster whose rank bit is set in `mask`.
__device__ __forceinline__ void commit_multicast(uint64_t* bar, uint16_t mask) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                 ::"r"(smem_u32(bar)), "h"(mask)
                 : "memory");
}

// Instruction descriptor, kind::f16: A, B fp16 K-major, D fp32, shape M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4)                                  // D format: f32
           | (0u << 7) | (0u << 10)                   // A, B: f16
           | (0u << 15) | (0u << 16)                  // A, B: K-major
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// Shared-memory matrix descriptor, no swizzle, K-major: 8-row x 16-byte core
// matrices; lbo = byte distance between core matrices adjacent along K,
// sbo = byte distance between 8-row groups.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu)
           | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16)
           | (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32)
           | (1ull << 46);                            // descriptor version for the sm_100 family
}

// Shared-memory matrix descriptor, 128-byte swizzle, K-major: 8-row x
// 128-byte atoms (1024-byte aligned), sbo = byte distance between atoms along
// the rows; the leading offset is unused (one MMA's K never leaves a row).
// A K step of 16 fp16 elements inside the atom adds 32 bytes to the start.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t sbo) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu)
           | (1ull << 16)                             // leading offset: 16 bytes, ignored
           | (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32)
           | (1ull << 46)                             // descriptor version for the sm_100 family
           | (2ull << 61);                            // 128-byte swizzle
}

// ----------------------------------------------------------- TMEM ld / st
// 32 lanes x 32 bits, 16 consecutive columns per thread.
__device__ __forceinline__ void ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
// 32 lanes x 32 bits, 8 consecutive columns per thread.
__device__ __forceinline__ void ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
__device__ __forceinline__ void st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
// 16 lanes x 256 bits, twice along the columns: per 8-column group, thread t
// holds (lane t/4, columns 2(t%4), 2(t%4)+1) and (lane t/4 + 8, the same
// columns) -- the layout of an mma.sync m16n8 accumulator; r[4g..4g+3] is
// column group g.
__device__ __forceinline__ void ld16x256b_x2(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
// Column-count-generic forms (8 or 16).
template <int W> __device__ __forceinline__ void ldw(uint32_t taddr, uint32_t (&r)[W]) {
    if constexpr (W == 8) ld8(taddr, r); else ld16(taddr, r);
}
template <int W> __device__ __forceinline__ void stw(uint32_t taddr, const uint32_t (&r)[W]) {
    if constexpr (W == 8) st8(taddr, r); else st16(taddr, r);
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// --------------------------------------------------------------- TMA 2-D
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(smem_dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Four rows r0..r3 of a 2-D tensor map whose box is one row high, from column
// x, landing one after another at smem_dst (128-byte aligned).
__device__ __forceinline__ void tma_gather4(void* smem_dst, const CUtensorMap* map, int x, int r0, int r1, int r2,
                                            int r3, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], "
        "[%1, {%2, %3, %4, %5, %6}], [%7];"
        ::"r"(smem_u32(smem_dst)), "l"(map), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Barrier over `nthreads` threads (whole warps) that also ANDs a predicate across them.
__device__ __forceinline__ bool named_and(uint32_t id, uint32_t nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ----------------------------------------------------- packed fp32 pairs
// Two independent IEEE round-to-nearest operations per instruction.
__device__ __forceinline__ uint64_t pk(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void upk(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// ------------------------------------------------------------ host: tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (so the
// library needs no link-time driver symbol); null when the driver lacks it.
inline EncodeTiledFn encode_tiled_fn() {
    static const EncodeTiledFn fn = [] {
        void* q = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) ==
                cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(q);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

}  // namespace tc
}  // namespace cq
