// Per-chunk block arithmetic shared by the GEMV and routed-expert kernels.
//
// A chunk is 256 elements of one weight row: eight 32-blocks (Q4_0, Q4_1,
// Q8_0) or one Q4_K superblock. chunk_dot<WF, MT> forms, for up to MT tokens,
// the chunk's value in the library's fixed fp32 order (include/cq.h): exact
// int32 block dots with dp4a, then the block scale terms with explicit
// round-to-nearest operations, blocks in increasing k.
//
// Block formulas: alice-llm docs "Computation Path (Q4_K)" (d * d_q8 *
// sum(scale*q4*q8) - dmin * d_q8 * sum(min*bsum)); GGUF layouts for Q4_0
// (d * (q - 8)), Q4_1 (d * q + m, offset term m * s with the Q8_1 block sum
// s) and Q8_0 (d * q), the Q8_0/Q4_K field order as in alice-llm's
// "Quantization Block Specs" table.
#pragma once
#include "cq_device.cuh"

namespace cq {

template <int WF> struct Fmt;
template <> struct Fmt<CQ_Q4_0> { static constexpr int CH = WCHUNK_Q4_0, ACH = ACHUNK_Q8_0, ACP = 272; };
template <> struct Fmt<CQ_Q8_0> { static constexpr int CH = WCHUNK_Q8_0, ACH = ACHUNK_Q8_0, ACP = 272; };
template <> struct Fmt<CQ_Q4_1> { static constexpr int CH = WCHUNK_Q4_1, ACH = ACHUNK_Q8_1, ACP = 304; };
template <> struct Fmt<CQ_Q4_K> { static constexpr int CH = WCHUNK_Q4_K, ACH = ACHUNK_Q8_K, ACP = 304; };

// Load NU 16-byte units starting at unit i0 of a 16-byte aligned pointer.
template <int NU>
__device__ __forceinline__ void ld_units(const uint8_t* p, int i0, uint32_t (&u)[4 * NU]) {
    const uint4* q = reinterpret_cast<const uint4*>(p) + i0;
#pragma unroll
    for (int i = 0; i < NU; ++i) {
        const uint4 v = q[i];
        u[4 * i] = v.x; u[4 * i + 1] = v.y; u[4 * i + 2] = v.z; u[4 * i + 3] = v.w;
    }
}

// Block with an fp16 scale at byte `off` (even) of u[] followed by the quant
// bytes; returns the scale bits and quant word i (4 consecutive quant bytes).
__device__ __forceinline__ uint32_t half_at(const uint32_t* u, int off) {
    return (off & 2) ? (u[off >> 2] >> 16) : (u[off >> 2] & 0xffffu);
}
__device__ __forceinline__ uint32_t word_after_half(const uint32_t* u, int off, int i) {
    const int b = off >> 2;
    return (off & 2) ? u[b + 1 + i] : __funnelshift_r(u[b + i], u[b + i + 1], 16);
}

// ------------------------------------------------------------ chunk dots
// wc: weight chunk in shared memory (16-byte aligned); xc: the chunk's
// activations of token 0 in shared memory, token m at xc + m * tok_pitch.
// c[m] receives the chunk value of token m in the fixed order.

template <int MT>
__device__ __forceinline__ void chunk_q8_0(const uint8_t* wc, const uint8_t* xc, int tok_pitch, int M,
                                           float (&c)[MT]) {
#pragma unroll
    for (int m = 0; m < MT; ++m) c[m] = 0.0f;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int off = (34 * b) & 15, unit = (34 * b) >> 4;
        uint32_t u[12];
        ld_units<3>(wc, unit, u);
        const float dw = h2f(half_at(u, off));
        int qw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) qw[i] = static_cast<int>(word_after_half(u, off, i));
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                uint32_t a[12];
                ld_units<3>(xc + m * tok_pitch, unit, a);
                const float dx = h2f(half_at(a, off));
                int isum = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) isum = __dp4a(qw[i], static_cast<int>(word_after_half(a, off, i)), isum);
                c[m] = __fmaf_rn(__fmul_rn(dw, dx), __int2float_rn(isum), c[m]);
            }
        }
    }
}

template <int MT>
__device__ __forceinline__ void chunk_q4_0(const uint8_t* wc, const uint8_t* xc, int tok_pitch, int M,
                                           float (&c)[MT]) {
#pragma unroll
    for (int m = 0; m < MT; ++m) c[m] = 0.0f;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int woff = (18 * b) & 15, wunit = (18 * b) >> 4;
        uint32_t u[8];
        ld_units<2>(wc, wunit, u);
        const float dw = h2f(half_at(u, woff));
        int lo[4], hi[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t q = word_after_half(u, woff, i);
            lo[i] = nib_minus8(q & 0x0f0f0f0fu);
            hi[i] = nib_minus8((q >> 4) & 0x0f0f0f0fu);
        }
        const int aoff = (34 * b) & 15, aunit = (34 * b) >> 4;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                uint32_t a[12];
                ld_units<3>(xc + m * tok_pitch, aunit, a);
                const float dx = h2f(half_at(a, aoff));
                int isum = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    isum = __dp4a(lo[i], static_cast<int>(word_after_half(a, aoff, i)), isum);
                    isum = __dp4a(hi[i], static_cast<int>(word_after_half(a, aoff, i + 4)), isum);
                }
                c[m] = __fmaf_rn(__fmul_rn(dw, dx), __int2float_rn(isum), c[m]);
            }
        }
    }
}

template <int MT>
__device__ __forceinline__ void chunk_q4_1(const uint8_t* wc, const uint8_t* xc, int tok_pitch, int M,
                                           float (&c)[MT]) {
#pragma unroll
    for (int m = 0; m < MT; ++m) c[m] = 0.0f;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int wbase = ((20 * b) & 15) >> 2, wunit = (20 * b) >> 4;
        uint32_t u[8];
        ld_units<2>(wc, wunit, u);
        const float dw = h2f(u[wbase]);
        const float mw = h2f(u[wbase] >> 16);
        int lo[4], hi[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t q = u[wbase + 1 + i];
            lo[i] = static_cast<int>(q & 0x0f0f0f0fu);
            hi[i] = static_cast<int>((q >> 4) & 0x0f0f0f0fu);
        }
        const int abase = ((36 * b) & 15) >> 2, aunit = (36 * b) >> 4;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                uint32_t a[12];
                ld_units<3>(xc + m * tok_pitch, aunit, a);
                const float dx = h2f(a[abase]);
                const float sx = h2f(a[abase] >> 16);
                int isum = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    isum = __dp4a(lo[i], static_cast<int>(a[abase + 1 + i]), isum);
                    isum = __dp4a(hi[i], static_cast<int>(a[abase + 5 + i]), isum);
                }
                float cm = __fmaf_rn(__fmul_rn(dw, dx), __int2float_rn(isum), c[m]);
                c[m] = __fmaf_rn(mw, sx, cm);
            }
        }
    }
}

// Six-bit scale and min of sub-block j from the twelve scale bytes held in
// s0 (bytes 0-3), s1 (4-7), s2 (8-11).
__device__ __forceinline__ void q4k_scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int j, int& sc, int& mn) {
    auto byte = [](uint32_t w, int i) { return static_cast<int>((w >> (8 * i)) & 0xffu); };
    if (j < 4) {
        sc = byte(s0, j) & 63;
        mn = byte(s1, j) & 63;
    } else {
        sc = (byte(s2, j - 4) & 15) | ((byte(s0, j - 4) >> 6) << 4);
        mn = (byte(s2, j - 4) >> 4) | ((byte(s1, j - 4) >> 6) << 4);
    }
}

template <int MT>
__device__ __forceinline__ void chunk_q4_k(const uint8_t* wc, const uint8_t* xc, int tok_pitch, int M,
                                           float (&c)[MT]) {
    uint32_t w[36];
    ld_units<9>(wc, 0, w);
    const float d = h2f(w[0]);
    const float dmin = h2f(w[0] >> 16);
    int isc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) isc[m] = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        int sc, mn;
        q4k_scale_min(w[1], w[2], w[3], j, sc, mn);
        (void)mn;
        int nib[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t q = w[4 + 8 * (j >> 1) + i];
            nib[i] = static_cast<int>((j & 1) ? ((q >> 4) & 0x0f0f0f0fu) : (q & 0x0f0f0f0fu));
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                uint32_t a[12];
                ld_units<3>(xc + m * tok_pitch, 2 * j, a);   // bytes 32j .. 32j+47: quants at +4
                int s = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) s = __dp4a(nib[i], static_cast<int>(a[1 + i]), s);
                isc[m] += sc * s;
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m < M) {
            const uint8_t* xm = xc + m * tok_pitch;
            uint32_t bs[12];
            ld_units<3>(xm, 16, bs);                        // bytes 256..303: bsum pair j in word 1+j
            const float dx = __uint_as_float(*reinterpret_cast<const uint32_t*>(xm));
            int im = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int sc, mn;
                q4k_scale_min(w[1], w[2], w[3], j, sc, mn);
                const uint32_t p = bs[1 + j];
                const int pair = static_cast<int>(static_cast<int16_t>(p & 0xffffu)) +
                                 static_cast<int>(static_cast<int16_t>(p >> 16));
                im += mn * pair;
            }
            const float a = __fmul_rn(dx, d);
            const float bm = __fmul_rn(dx, dmin);
            c[m] = __fmaf_rn(a, __int2float_rn(isc[m]), -__fmul_rn(bm, __int2float_rn(im)));
        }
    }
}

template <int WF, int MT>
__device__ __forceinline__ void chunk_dot(const uint8_t* wc, const uint8_t* xc, int tok_pitch, int M, float (&c)[MT]) {
    if constexpr (WF == CQ_Q8_0) chunk_q8_0<MT>(wc, xc, tok_pitch, M, c);
    else if constexpr (WF == CQ_Q4_0) chunk_q4_0<MT>(wc, xc, tok_pitch, M, c);
    else if constexpr (WF == CQ_Q4_1) chunk_q4_1<MT>(wc, xc, tok_pitch, M, c);
    else chunk_q4_k<MT>(wc, xc, tok_pitch, M, c);
}

}  // namespace cq
