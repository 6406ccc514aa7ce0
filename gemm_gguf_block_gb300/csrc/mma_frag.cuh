// Exact integer block dots of the 32-element GGUF formats on mma.sync
// m16n8k16 (fp16 operands, fp32 accumulators), for the batched GEMV; the
// prefill GEMM of the same formats takes the block traits and byte helpers.
//
// Every weight quant enters the A operand as BIAS + v (v its value), built
// from the packed bytes by one lop3 per pair; every activation quant enters B
// as its exact fp16 value; the accumulator starts at -BIAS * sum(x). All
// operands and partial sums are integers below 2^23, so the two chained
// k-steps of a block give the exact integer dot. For the 4-bit formats the
// high nibbles (k-step 1) are masked in place: A = 1024 + 16 n, with the
// k-step's activations pre-scaled by 1/16 (exact in fp16), so that
// A * B = 64 x + n x and the accumulator starts at
// -(BIAS_LO * sum(x_lo) + BIAS_HI * sum(x_hi)) instead.
//
// The k order inside a 32-block: k-step 0 takes elements 0..15, k-step 1
// elements 16..31; within a k-step, fragment column 2t holds element 4t,
// 2t+1 -> 4t+2, 2t+8 -> 4t+1, 2t+9 -> 4t+3. Both operands use this order, so
// the products are the same; what it buys is that lane t's weight quants are
// the four consecutive bytes 4t..4t+3 of a 16-element run.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

#include "cq_device.cuh"
#include "tc.cuh"

namespace cq {
namespace mf {

// BB / QO: weight block bytes and offset of its quants; ABB / AQO: the same
// for the paired activation block; BIAS: the A operand holds BIAS + v.
template <int WF> struct MF;
// BIAS_LO / BIAS_HI: the accumulator's start per unit of the activation sums of
// k-step 0 (elements 0..15) and k-step 1 (16..31).
template <> struct MF<CQ_Q4_0> {
    static constexpr int BB = 18, QO = 2, ABB = 34, AQO = 2, BIAS = 1032, BIAS_LO = 1032, BIAS_HI = 72;
};
template <> struct MF<CQ_Q4_1> {
    static constexpr int BB = 20, QO = 4, ABB = 36, AQO = 4, BIAS = 1024, BIAS_LO = 1024, BIAS_HI = 64;
};
template <> struct MF<CQ_Q8_0> {
    static constexpr int BB = 34, QO = 2, ABB = 34, AQO = 2, BIAS = 1152, BIAS_LO = 1152, BIAS_HI = 1152;
};

// Bytes per weight row in a stage of 8 blocks, padded for Q4_1 (160 -> 176
// bytes: 44 words, so the 8 rows one load instruction touches fall in 8
// different bank groups; the padding is the start of the next segment, or
// zero fill past the end of the row).
__host__ __device__ constexpr int stage_pitch(int bb) { return bb == 20 ? 176 : 8 * bb; }

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// D = A * B + (c0, c1, c0, c1), and D += A * B.
__device__ __forceinline__ void mma16816c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, float c0,
                                          float c1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%10,%11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void mma16816acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (w & sel) with bits of `set` forced on: one lop3. With sel = 0x000F000F and
// set = 0x64006400 the two 16-bit lanes become the binary16 values 1024 + n of
// the nibbles in bits 0-3 and 16-19.
__device__ __forceinline__ uint32_t and_or(uint32_t w, uint32_t sel, uint32_t set) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(sel), "r"(set));   // (a & b) | c
    return r;
}
// The same for signed bytes in bits 0-7 and 16-23: 1024 + (b + 128) = 1152 + b.
__device__ __forceinline__ uint32_t s8pair_1152(uint32_t w) {
    return and_or(w ^ 0x00800080u, 0x00FF00FFu, 0x64006400u);
}

// A fragments of rows g (q0) and g+8 (q1) for one block: BIAS + value per element.
template <int WF>
__device__ __forceinline__ void a_frags(uint32_t q0a, uint32_t q1a, uint32_t q0b, uint32_t q1b, uint32_t (&a0)[4],
                                        uint32_t (&a1)[4]) {
    if constexpr (WF == CQ_Q8_0) {
        // q?a: quants 4t..4t+3, q?b: 16+4t..16+4t+3 (signed bytes)
        a0[0] = s8pair_1152(q0a);        a0[1] = s8pair_1152(q1a);
        a0[2] = s8pair_1152(q0a >> 8);   a0[3] = s8pair_1152(q1a >> 8);
        a1[0] = s8pair_1152(q0b);        a1[1] = s8pair_1152(q1b);
        a1[2] = s8pair_1152(q0b >> 8);   a1[3] = s8pair_1152(q1b >> 8);
    } else {
        // q?a: bytes 4t..4t+3; low nibbles = elements 4t.. (1024 + n), high
        // nibbles = elements 16+4t.. masked in place (1024 + 16 n)
        constexpr uint32_t LO = 0x000F000Fu, HI = 0x00F000F0u, SET = 0x64006400u;
        const uint32_t s0 = q0a >> 8, s1 = q1a >> 8;
        a0[0] = and_or(q0a, LO, SET);    a0[1] = and_or(q1a, LO, SET);
        a0[2] = and_or(s0, LO, SET);     a0[3] = and_or(s1, LO, SET);
        a1[0] = and_or(q0a, HI, SET);    a1[1] = and_or(q1a, HI, SET);
        a1[2] = and_or(s0, HI, SET);     a1[3] = and_or(s1, HI, SET);
        (void)q0b;
        (void)q1b;
    }
}

// Four bytes at a 2-byte-aligned shared-memory address.
__device__ __forceinline__ uint32_t ld_u32_a2(const uint8_t* p) {
    const uint16_t* h = reinterpret_cast<const uint16_t*>(p);
    return __byte_perm(h[0], h[1], 0x5410);
}

// Row g and g + 8 of one weight block in a stage (w0, w1 their block starts):
// the A fragments of both k-steps, and the rows' d_w (and m_w for Q4_1) as
// (v, v) pairs.
template <int WF>
__device__ __forceinline__ void weight_frags(const uint8_t* w0, const uint8_t* w1, int t, uint32_t (&a0)[4],
                                             uint32_t (&a1)[4], uint64_t& dw0, uint64_t& dw1, uint64_t& mw0,
                                             uint64_t& mw1) {
    using F = MF<WF>;
    uint32_t q0a, q1a, q0b = 0, q1b = 0;
    if constexpr (WF == CQ_Q4_1) {
        q0a = *reinterpret_cast<const uint32_t*>(w0 + F::QO + 4 * t);
        q1a = *reinterpret_cast<const uint32_t*>(w1 + F::QO + 4 * t);
    } else {
        q0a = ld_u32_a2(w0 + F::QO + 4 * t);
        q1a = ld_u32_a2(w1 + F::QO + 4 * t);
        if constexpr (WF == CQ_Q8_0) {
            q0b = ld_u32_a2(w0 + F::QO + 16 + 4 * t);
            q1b = ld_u32_a2(w1 + F::QO + 16 + 4 * t);
        }
    }
    a_frags<WF>(q0a, q1a, q0b, q1b, a0, a1);
    if constexpr (WF == CQ_Q4_1) {
        const uint32_t dm0 = *reinterpret_cast<const uint32_t*>(w0);
        const uint32_t dm1 = *reinterpret_cast<const uint32_t*>(w1);
        const float d0 = h2f(dm0), d1 = h2f(dm1), m0 = h2f(dm0 >> 16), m1 = h2f(dm1 >> 16);
        dw0 = tc::pk(d0, d0);
        dw1 = tc::pk(d1, d1);
        mw0 = tc::pk(m0, m0);
        mw1 = tc::pk(m1, m1);
    } else {
        const float d0 = h2f(*reinterpret_cast<const uint16_t*>(w0));
        const float d1 = h2f(*reinterpret_cast<const uint16_t*>(w1));
        dw0 = tc::pk(d0, d0);
        dw1 = tc::pk(d1, d1);
        mw0 = mw1 = 0;
    }
}

// One activation block (Q8_0 or Q8_1 at blk) as the B operand: four 16-byte
// chunks, chunk t = fp16 of elements [4t, 4t+2, 4t+1, 4t+3, 16+4t, 18+4t,
// 17+4t, 19+4t] (lane t's B fragments of both k-steps; for the 4-bit weight
// formats the k-step 1 half scaled by 1/16); its d, its s (Q8_1) and the
// accumulator's start -(BIAS_LO * sum(q_0..15) + BIAS_HI * sum(q_16..31)).
template <int WF>
__device__ __forceinline__ void act_frags(const uint8_t* blk, uint4 (&ch)[4], float& d, float& s, int& bias) {
    using F = MF<WF>;
    const uint16_t* h = reinterpret_cast<const uint16_t*>(blk);
    uint32_t w[8];
    int sum_lo = 0, sum_hi = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        w[j] = __byte_perm(h[F::AQO / 2 + 2 * j], h[F::AQO / 2 + 2 * j + 1], 0x5410);
        if (j < 4) sum_lo = __dp4a(static_cast<int>(w[j]), 0x01010101, sum_lo);
        else sum_hi = __dp4a(static_cast<int>(w[j]), 0x01010101, sum_hi);
    }
    bias = -(F::BIAS_LO * sum_lo + F::BIAS_HI * sum_hi);
    constexpr bool HI16 = WF != CQ_Q8_0;
    const __half2 k16 = __halves2half2(__ushort_as_half(HI16 ? 0x2C00 : 0x3C00),
                                       __ushort_as_half(HI16 ? 0x2C00 : 0x3C00));   // 1/16 or 1
    d = h2f(h[0]);
    s = WF == CQ_Q4_1 ? h2f(h[1]) : 0.0f;
    // exact fp16 of the signed bytes: (1152 + b) - 1152
    const __half2 k1152 = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint32_t e02 = h2u(__hsub2(u2h(s8pair_1152(w[t])), k1152));
        const uint32_t e13 = h2u(__hsub2(u2h(s8pair_1152(w[t] >> 8)), k1152));
        const uint32_t f02 = h2u(__hmul2(__hsub2(u2h(s8pair_1152(w[t + 4])), k1152), k16));
        const uint32_t f13 = h2u(__hmul2(__hsub2(u2h(s8pair_1152(w[t + 4] >> 8)), k1152), k16));
        ch[t] = make_uint4(e02, e13, f02, f13);
    }
}

}  // namespace mf
}  // namespace cq
