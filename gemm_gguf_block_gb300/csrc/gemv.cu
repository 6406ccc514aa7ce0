// Decode GEMV / batched LM-head projection, 1 <= M <= 16 tokens.
//
// cera README "Quantization": integer GEMV over quantized weights with
// activations quantized to 8 bits; alice-llm "The GPU Optimization Journey"
// phases 1.5-2 (fused dequant-matvec, register-level reductions) and
// "Batch-4 Speculative Decoding" (weights decoded once, one accumulator per
// token); cera README "Other features" (the LM head projected for all
// verified positions in one pass, so it is read once per round).
//
// The work. A weight row of K elements is nc chunks: 128 elements (four
// 32-blocks) for Q4_0 / Q4_1 / Q8_0, one 256-element superblock for Q4_K.
// A warp owns "items" of at most 32 chunks: R = 32/nc whole rows when a row
// is shorter than 32 chunks, else a 32-chunk segment of one row. An item is
// one contiguous byte range, so a single bulk copy (cp.async.bulk, the
// one-dimensional TMA engine) lands it in the warp's ring of shared-memory
// stages; the copy of item i+S is issued as soon as item i is in registers.
// Lane l takes chunk l of the item: it unpacks its weights in registers and
// forms exact int32 block dots with dp4a against the activations, which the
// CTA has staged once in shared memory in an aligned split layout (quants on
// 16-byte boundaries, scales in the padding, chunk pitch an odd number of
// 16-byte units so the lanes' 128-bit loads do not collide). Chunk values go
// to a small per-warp buffer; every B rows, lane (m, r) adds row r's values
// for token m in increasing k (for Q4_K: y = fma(d_x, t, y) per superblock) --
// the fixed evaluation order of include/cq.h.
#include <algorithm>

#include "cq_device.cuh"
#include "cq_internal.h"

namespace cq {
namespace {

constexpr int WPC_MAX = 16;       // warps per CTA (one CTA per SM)
constexpr int CBUF_FLOATS = 512;  // per-warp buffer of chunk values (2 KB)

// Weight chunk bytes, chunk elements, staged activation chunk pitch, and the
// 32-bit words a lane holds the chunk in (Q6_K's 210 bytes: 53).
template <int WF> struct G;
template <> struct G<CQ_Q8_0> { static constexpr int WCH = 136, CE = 128, ACP = 144, WR = 34; };
template <> struct G<CQ_Q4_0> { static constexpr int WCH = 72, CE = 128, ACP = 144, WR = 18; };
template <> struct G<CQ_Q4_1> { static constexpr int WCH = 80, CE = 128, ACP = 176, WR = 20; };
template <> struct G<CQ_Q4_K> { static constexpr int WCH = 144, CE = 256, ACP = 304, WR = 36; };
template <> struct G<CQ_Q5_K> { static constexpr int WCH = 176, CE = 256, ACP = 304, WR = 44; };
template <> struct G<CQ_Q6_K> { static constexpr int WCH = 210, CE = 256, ACP = 336, WR = 53; };
template <int WF> __host__ __device__ constexpr bool superblock_fmt() {
    return WF == CQ_Q4_K || WF == CQ_Q5_K || WF == CQ_Q6_K;
}

struct GemvParams {
    const uint8_t* W;
    const uint8_t* xq;
    float* y;
    int* status;
    int64_t N;
    int64_t row_bytes;
    int M;
    int nc;           // chunks per row (paired: gate row then up row, 2 * nca)
    int nca;          // chunks of x (== nc unpaired)
    const uint8_t* W2;  // paired: the up matrix (W is the gate matrix)
    int64_t wrow;     // paired: bytes per gate / up row
    int cpitch;       // floats per row in the chunk-value buffer (odd where it fits: no bank conflicts)
    int R;            // rows per item
    int segc;         // chunks per item
    int nseg;         // items per row group (R == 1 whenever nseg > 1)
    int B;            // rows per batch of sequential sums (a multiple of R)
    int stages;
    int stage_bytes;
    int warp_bytes;
    int act_bytes;
    int tok_pitch;    // bytes per token of staged activations
    int wconst;       // weights constant in flight: prefetch them before the dependency wait
    const float* x;   // fp32 activations to quantize in the kernel (cq_gemv_x), else null
    uint8_t* xq_out;  // where CTA 0 writes their quantisation (with x)
    int xreg;         // one token, whole rows per item: the lane's chunk of x held in registers
    int l2pf;         // items past the ring prefetched into L2 before the dependency wait
};

// Exact float of an int with |i| < 2^22: the bits of 1.5 * 2^23 + i, minus 1.5 * 2^23.
__device__ __forceinline__ float i2f_exact(int i) {
    return __fsub_rn(__int_as_float(0x4B400000 + i), 12582912.0f);
}

template <int N>
__device__ __forceinline__ void lds64(const uint8_t* p, uint32_t (&u)[2 * N]) {
    const uint2* q = reinterpret_cast<const uint2*>(p);
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const uint2 v = q[i];
        u[2 * i] = v.x;
        u[2 * i + 1] = v.y;
    }
}
__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ void ld_f4(const uint8_t* p, float* f) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}

// ------------------------------------------------------- staging of activations
// Q8_0 / Q8_1 chunk of 4 blocks -> [qs 128 B][d0..d3 fp32] (Q8_1: [d,s] pairs);
// Q8_K superblock -> [qs 256 B][d fp32 @256][8 int32 bsum pairs @272] for
// Q4_K, [16 int32 bsums @272] for Q6_K (its sub-blocks are 16 elements).
template <int WF>
__device__ void stage_activations(const GemvParams& p, uint8_t* act) {
    const int nthr = blockDim.x;
    if constexpr (superblock_fmt<WF>()) {
        const int ns = p.nca;
        const int words = p.M * ns * 73;          // 292 bytes per superblock
        const uint32_t* src = reinterpret_cast<const uint32_t*>(p.xq);
        for (int i = threadIdx.x; i < words; i += nthr) {
            const int sb = i / 73, w = i - sb * 73;     // superblock (over tokens), word in it
            const int m = sb / ns, c = sb - m * ns;
            uint8_t* dst = act + m * p.tok_pitch + c * G<WF>::ACP;
            const uint32_t v = src[i];
            if (w == 0) {
                *reinterpret_cast<uint32_t*>(dst + 256) = v;
            } else if (w <= 64) {
                *reinterpret_cast<uint32_t*>(dst + 4 * (w - 1)) = v;
            } else {
                const int j = w - 65;                    // bsum[2j] and bsum[2j+1]
                const int b0 = static_cast<int16_t>(v & 0xffffu), b1 = static_cast<int16_t>(v >> 16);
                if constexpr (WF == CQ_Q6_K) {
                    reinterpret_cast<int*>(dst + 272)[2 * j] = b0;
                    reinterpret_cast<int*>(dst + 272)[2 * j + 1] = b1;
                } else {
                    *reinterpret_cast<int*>(dst + 272 + 4 * j) = b0 + b1;
                }
            }
        }
    } else {
        constexpr int BB = WF == CQ_Q4_1 ? 36 : 34;     // Q8_1 or Q8_0 block bytes
        constexpr int QO = WF == CQ_Q4_1 ? 4 : 2;       // quant offset in the block
        const int nblk = p.M * p.nca * 4;
        const uint16_t* src = reinterpret_cast<const uint16_t*>(p.xq);
        for (int i = threadIdx.x; i < nblk; i += nthr) {
            const int m = i / (p.nca * 4), r = i - m * p.nca * 4;
            const int c = r >> 2, b = r & 3;
            const uint16_t* s = src + static_cast<int64_t>(i) * (BB / 2);
            uint8_t* dst = act + m * p.tok_pitch + c * G<WF>::ACP;
            uint32_t* q = reinterpret_cast<uint32_t*>(dst + 32 * b);
#pragma unroll
            for (int w = 0; w < 8; ++w)
                q[w] = static_cast<uint32_t>(s[QO / 2 + 2 * w]) | (static_cast<uint32_t>(s[QO / 2 + 2 * w + 1]) << 16);
            if constexpr (WF == CQ_Q4_1) {
                reinterpret_cast<float*>(dst + 128)[2 * b] = h2f(s[0]);
                reinterpret_cast<float*>(dst + 128)[2 * b + 1] = h2f(s[1]);
            } else {
                reinterpret_cast<float*>(dst + 128)[b] = h2f(s[0]);
            }
        }
    }
}

// Quantise fp32 activations (cq_gemv_x) and stage them exactly as
// stage_activations stages the output of cq_quantize_act: the same rule in the
// same fp32 operations (q8_scale, q8_inv, quant_q8, RN fp16 scales), so the
// same bits. CTA 0 also writes the quantized rows to p.xq_out.
template <int WF>
__device__ void stage_activations_x(const GemvParams& p, uint8_t* act) {
    const int nthr = blockDim.x;
    const bool out = blockIdx.x == 0;
    const int64_t K = static_cast<int64_t>(p.nca) * G<WF>::CE;
    if constexpr (superblock_fmt<WF>()) {
        // A warp per superblock, eight consecutive elements per lane.
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = nthr >> 5;
        const int ns = p.nca;
        for (int sb = warp; sb < p.M * ns; sb += nw) {
            const int m = sb / ns, c = sb - m * ns;
            const float4* src = reinterpret_cast<const float4*>(p.x + m * K + c * 256 + 8 * lane);
            const float4 v0 = src[0], v1 = src[1];
            const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            float a = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
#pragma unroll
            for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            const float d = q8_scale(a);
            const float id = q8_inv(d);
            uint32_t packed[2] = {0u, 0u};
            int sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int q = quant_q8(v[i], id);
                sum += q;
                packed[i >> 2] |= (static_cast<uint32_t>(q) & 0xffu) << (8 * (i & 3));
            }
            const int s16 = sum + __shfl_xor_sync(0xffffffffu, sum, 1);      // 16 consecutive quants
            const int s32 = s16 + __shfl_xor_sync(0xffffffffu, s16, 2);      // 32: a bsum pair
            uint8_t* dst = act + m * p.tok_pitch + c * G<WF>::ACP;
            reinterpret_cast<uint32_t*>(dst + 8 * lane)[0] = packed[0];
            reinterpret_cast<uint32_t*>(dst + 8 * lane)[1] = packed[1];
            if (lane == 0) *reinterpret_cast<float*>(dst + 256) = d;
            if constexpr (WF == CQ_Q6_K) {
                if ((lane & 1) == 0) *reinterpret_cast<int*>(dst + 272 + 2 * lane) = s16;
            } else {
                if ((lane & 3) == 0) *reinterpret_cast<int*>(dst + 272 + lane) = s32;
            }
            if (out) {
                uint8_t* blk = p.xq_out + static_cast<int64_t>(sb) * 292;
                uint32_t* qw = reinterpret_cast<uint32_t*>(blk + 4 + 8 * lane);
                qw[0] = packed[0];
                qw[1] = packed[1];
                if ((lane & 1) == 0) *reinterpret_cast<int16_t*>(blk + 260 + lane) = static_cast<int16_t>(s16);
                if (lane == 0) *reinterpret_cast<float*>(blk) = d;
            }
        }
    } else {
        constexpr int BB = WF == CQ_Q4_1 ? 36 : 34;     // Q8_1 or Q8_0 block bytes
        constexpr int QO = WF == CQ_Q4_1 ? 4 : 2;       // quant offset in the block
        const int nblk = p.M * p.nca * 4;
        for (int i = threadIdx.x; i < nblk; i += nthr) {
            const int m = i / (p.nca * 4), r = i - m * p.nca * 4;
            const int c = r >> 2, b = r & 3;
            const float4* src = reinterpret_cast<const float4*>(p.x + m * K + 32 * r);
            float v[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 f = src[j];
                v[4 * j] = f.x;
                v[4 * j + 1] = f.y;
                v[4 * j + 2] = f.z;
                v[4 * j + 3] = f.w;
            }
            float a = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) a = fmaxf(a, fabsf(v[j]));
            const float d = q8_scale(a);
            const float id = q8_inv(d);
            uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            int sum = 0;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int q = quant_q8(v[j], id);
                sum += q;
                w[j >> 2] |= (static_cast<uint32_t>(q) & 0xffu) << (8 * (j & 3));
            }
            const __half dh = __float2half_rn(d);
            uint8_t* dst = act + m * p.tok_pitch + c * G<WF>::ACP;
            uint32_t* q = reinterpret_cast<uint32_t*>(dst + 32 * b);
#pragma unroll
            for (int j = 0; j < 8; ++j) q[j] = w[j];
            __half sh = __float2half_rn(0.0f);
            if constexpr (WF == CQ_Q4_1) {
                sh = __float2half_rn(__fmul_rn(d, static_cast<float>(sum)));
                reinterpret_cast<float*>(dst + 128)[2 * b] = __half2float(dh);
                reinterpret_cast<float*>(dst + 128)[2 * b + 1] = __half2float(sh);
            } else {
                reinterpret_cast<float*>(dst + 128)[b] = __half2float(dh);
            }
            if (out) {
                uint8_t* blk = p.xq_out + static_cast<int64_t>(i) * BB;
                *reinterpret_cast<__half*>(blk) = dh;
                if constexpr (WF == CQ_Q4_1) {
                    *reinterpret_cast<__half*>(blk + 2) = sh;
#pragma unroll
                    for (int j = 0; j < 8; ++j) reinterpret_cast<uint32_t*>(blk + QO)[j] = w[j];
                } else {
                    uint16_t* h = reinterpret_cast<uint16_t*>(blk + QO);     // 2 mod 4: 16-bit stores
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        h[2 * j] = static_cast<uint16_t>(w[j]);
                        h[2 * j + 1] = static_cast<uint16_t>(w[j] >> 16);
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------------- chunk values
// w: weight chunk in registers. x: the staged activations of the same chunk,
// read through an activation source: q(m, i) is the 16-byte piece i of token
// m's 128 quants, d(m, b) / s(m, b) block b's scale / Q8_1 sum.

// Activations read from shared memory: token m at xa + m * tp.
template <bool PAIRS>
struct SmemX {
    const uint8_t* xa;
    int tp;
    __device__ __forceinline__ uint4 q(int m, int i) const { return lds128(xa + m * tp + 16 * i); }
    __device__ __forceinline__ float d(int m, int b) const {
        return reinterpret_cast<const float*>(xa + m * tp + 128)[PAIRS ? 2 * b : b];
    }
    __device__ __forceinline__ float s(int m, int b) const {
        return reinterpret_cast<const float*>(xa + m * tp + 128)[2 * b + 1];
    }
};

// One token's activation chunk held in registers: when every item of a warp
// uses the same chunk of x (rows no longer than 32 chunks), it is read once.
template <bool PAIRS>
struct RegX {
    uint4 qv[8];
    float sc[PAIRS ? 8 : 4];
    __device__ __forceinline__ void load(const uint8_t* a) {
#pragma unroll
        for (int i = 0; i < 8; ++i) qv[i] = lds128(a + 16 * i);
        ld_f4(a + 128, sc);
        if constexpr (PAIRS) ld_f4(a + 144, sc + 4);
    }
    __device__ __forceinline__ uint4 q(int, int i) const { return qv[i]; }
    __device__ __forceinline__ float d(int, int b) const { return sc[PAIRS ? 2 * b : b]; }
    __device__ __forceinline__ float s(int, int b) const { return sc[2 * b + 1]; }
};

// Block dot of 32 signed bytes (as eight words) with an activation block.
__device__ __forceinline__ int dot32(const int (&q)[8], const uint4& a0, const uint4& a1) {
    int s = __dp4a(q[0], static_cast<int>(a0.x), 0);
    s = __dp4a(q[1], static_cast<int>(a0.y), s);
    s = __dp4a(q[2], static_cast<int>(a0.z), s);
    s = __dp4a(q[3], static_cast<int>(a0.w), s);
    s = __dp4a(q[4], static_cast<int>(a1.x), s);
    s = __dp4a(q[5], static_cast<int>(a1.y), s);
    s = __dp4a(q[6], static_cast<int>(a1.z), s);
    return __dp4a(q[7], static_cast<int>(a1.w), s);
}

template <int MT, class X>
__device__ __forceinline__ void chunk_q8_0(const uint32_t (&w)[34], const X& x, int M, float (&c)[MT]) {
#pragma unroll
    for (int m = 0; m < MT; ++m) c[m] = 0.0f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int o = 34 * b;                    // block offset in the chunk (0, 34, 68, 102)
        const int base = o >> 2;
        const bool odd = (o & 2) != 0;
        const float dw = h2f(odd ? (w[base] >> 16) : w[base]);
        int q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            q[i] = static_cast<int>(odd ? w[base + 1 + i] : __funnelshift_r(w[base + i], w[base + i + 1], 16));
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                const int s = dot32(q, x.q(m, 2 * b), x.q(m, 2 * b + 1));
                c[m] = __fmaf_rn(__fmul_rn(dw, x.d(m, b)), i2f_exact(s), c[m]);
            }
        }
    }
}

template <int MT, class X>
__device__ __forceinline__ void chunk_q4_0(const uint32_t (&w)[18], const X& x, int M, float (&c)[MT]) {
#pragma unroll
    for (int m = 0; m < MT; ++m) c[m] = 0.0f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int o = 18 * b;                    // 0, 18, 36, 54
        const int base = o >> 2;
        const bool odd = (o & 2) != 0;
        const float dw = h2f(odd ? (w[base] >> 16) : w[base]);
        int q[8];                                // low nibbles (elements 0..15), then high (16..31)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t v = odd ? w[base + 1 + i] : __funnelshift_r(w[base + i], w[base + i + 1], 16);
            q[i] = nib_minus8(v & 0x0f0f0f0fu);
            q[4 + i] = nib_minus8((v >> 4) & 0x0f0f0f0fu);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                const int s = dot32(q, x.q(m, 2 * b), x.q(m, 2 * b + 1));
                c[m] = __fmaf_rn(__fmul_rn(dw, x.d(m, b)), i2f_exact(s), c[m]);
            }
        }
    }
}

template <int MT, class X>
__device__ __forceinline__ void chunk_q4_1(const uint32_t (&w)[20], const X& x, int M, float (&c)[MT]) {
#pragma unroll
    for (int m = 0; m < MT; ++m) c[m] = 0.0f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int base = 5 * b;                  // 20-byte blocks: always word aligned
        const float dw = h2f(w[base]);
        const float mw = h2f(w[base] >> 16);
        int q[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t v = w[base + 1 + i];
            q[i] = static_cast<int>(v & 0x0f0f0f0fu);
            q[4 + i] = static_cast<int>((v >> 4) & 0x0f0f0f0fu);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                const int s = dot32(q, x.q(m, 2 * b), x.q(m, 2 * b + 1));
                const float cm = __fmaf_rn(__fmul_rn(dw, x.d(m, b)), i2f_exact(s), c[m]);
                c[m] = __fmaf_rn(mw, x.s(m, b), cm);
            }
        }
    }
}

// Six-bit scale and min of sub-block j from the twelve scale bytes s0|s1|s2.
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

// Q4_K and Q5_K: d / dmin in word 0, the twelve scale bytes in words 1-3,
// then (Q5_K) qh[32] in words 4-11, then qs[128]. A Q5_K quant is the Q4_K
// nibble with bit j of qh[l] (sub-block j, element l of it) as bit 4.
template <int MT, bool Q5, int NW>
__device__ __forceinline__ void chunk_q4_k(const uint32_t (&w)[NW], const uint8_t* xa, int tp, int M, float (&c)[MT]) {
    constexpr int QS = Q5 ? 12 : 4;
    const float d = h2f(w[0]);
    const float dmin = h2f(w[0] >> 16);
    int isc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) isc[m] = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        int sc, mn;
        q4k_scale_min(w[1], w[2], w[3], j, sc, mn);
        int nib[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t q = w[QS + 8 * (j >> 1) + i];
            uint32_t v = (j & 1) ? ((q >> 4) & 0x0f0f0f0fu) : (q & 0x0f0f0f0fu);
            if constexpr (Q5) v |= ((w[4 + i] >> j) & 0x01010101u) << 4;
            nib[i] = static_cast<int>(v);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                const uint8_t* xm = xa + m * tp;
                const uint4 a0 = lds128(xm + 32 * j), a1 = lds128(xm + 32 * j + 16);
                int s = __dp4a(nib[0], static_cast<int>(a0.x), 0);
                s = __dp4a(nib[1], static_cast<int>(a0.y), s);
                s = __dp4a(nib[2], static_cast<int>(a0.z), s);
                s = __dp4a(nib[3], static_cast<int>(a0.w), s);
                s = __dp4a(nib[4], static_cast<int>(a1.x), s);
                s = __dp4a(nib[5], static_cast<int>(a1.y), s);
                s = __dp4a(nib[6], static_cast<int>(a1.z), s);
                s = __dp4a(nib[7], static_cast<int>(a1.w), s);
                isc[m] += sc * s;
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m < M) {
            const uint8_t* xm = xa + m * tp;
            const float dx = *reinterpret_cast<const float*>(xm + 256);
            const uint4 p0 = lds128(xm + 272), p1 = lds128(xm + 288);
            const int pr[8] = {static_cast<int>(p0.x), static_cast<int>(p0.y), static_cast<int>(p0.z),
                               static_cast<int>(p0.w), static_cast<int>(p1.x), static_cast<int>(p1.y),
                               static_cast<int>(p1.z), static_cast<int>(p1.w)};
            int im = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int sc, mn;
                q4k_scale_min(w[1], w[2], w[3], j, sc, mn);
                im += mn * pr[j];
            }
            (void)dx;
            c[m] = __fmaf_rn(d, __int2float_rn(isc[m]), -__fmul_rn(dmin, __int2float_rn(im)));
        }
    }
}

// Q6_K superblock (words of the 210-byte chunk): ql at word 0, qh at word 32,
// the sixteen int8 scales at word 48, d in the low half of word 52. Sub-block
// j (16 elements) lies in half h = j / 8, quadrant q = (j / 2) % 4, elements
// l = 16 (j % 2) .. +15 of that quadrant; four consecutive elements' six-bit
// quants are one word: the ql nibbles (low for q < 2, high otherwise) or'd
// with qh's bit pair q moved to bits 4-5 of each byte. Per sub-block
// S_j = sum q6 * q8 - 32 * bsum_j exactly; isum = sum_j sc_j S_j; the chunk
// value is t = D(d) * (float)isum, folded into y as fma(d_x, t, y).
template <int MT>
__device__ __forceinline__ void chunk_q6_k(const uint32_t (&w)[53], const uint8_t* xa, int tp, int M, float (&c)[MT]) {
    int isum[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) isum[m] = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int h = j >> 3, q = (j >> 1) & 3, l0 = 16 * (j & 1);
        int v[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int l = l0 + 4 * p;
            const uint32_t qlw = w[16 * h + (l >> 2) + 8 * (q & 1)];
            const uint32_t lo = q < 2 ? (qlw & 0x0f0f0f0fu) : ((qlw >> 4) & 0x0f0f0f0fu);
            const uint32_t hi = ((w[32 + 8 * h + (l >> 2)] >> (2 * q)) & 0x03030303u) << 4;
            v[p] = static_cast<int>(lo | hi);
        }
        const int sc = static_cast<int>(static_cast<int8_t>((w[48 + (j >> 2)] >> (8 * (j & 3))) & 0xffu));
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                const uint8_t* xm = xa + m * tp;
                const uint4 a = lds128(xm + 16 * j);
                int sj = __dp4a(v[0], static_cast<int>(a.x), 0);
                sj = __dp4a(v[1], static_cast<int>(a.y), sj);
                sj = __dp4a(v[2], static_cast<int>(a.z), sj);
                sj = __dp4a(v[3], static_cast<int>(a.w), sj);
                sj -= 32 * reinterpret_cast<const int*>(xm + 272)[j];
                isum[m] += sc * sj;
            }
        }
    }
    const float d = h2f(w[52]);
#pragma unroll
    for (int m = 0; m < MT; ++m) c[m] = __fmul_rn(d, __int2float_rn(isum[m]));
}

// The weight chunk, copied from its stage to registers (so the stage can be
// refilled while the chunk value is formed).
template <int WF>
__device__ __forceinline__ void chunk_load(const uint8_t* wc, uint32_t (&w)[G<WF>::WR]) {
    if constexpr (WF == CQ_Q6_K) {
        // 210-byte chunks sit on 2-byte boundaries: 54 aligned words, each
        // pair funnel-shifted by the chunk's offset (0 or 16 bits).
        const uintptr_t a = reinterpret_cast<uintptr_t>(wc);
        const uint32_t* base = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
        const uint32_t sh = static_cast<uint32_t>(a & 3u) * 8u;
        uint32_t prev = base[0];
#pragma unroll
        for (int i = 0; i < 53; ++i) {
            const uint32_t next = base[i + 1];
            w[i] = __funnelshift_r(prev, next, sh);
            prev = next;
        }
    } else if constexpr (WF == CQ_Q4_K || WF == CQ_Q5_K) {
#pragma unroll
        for (int i = 0; i < G<WF>::WR / 4; ++i) {
            const uint4 v = lds128(wc + 16 * i);
            w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
    } else {
        lds64<G<WF>::WCH / 8>(wc, w);
    }
}

template <int WF, int MT, class X>
__device__ __forceinline__ void chunk_value(const uint32_t (&wc)[G<WF>::WR], const X& x, int M, float (&c)[MT]) {
    if constexpr (WF == CQ_Q8_0) chunk_q8_0<MT>(wc, x, M, c);
    else if constexpr (WF == CQ_Q4_0) chunk_q4_0<MT>(wc, x, M, c);
    else if constexpr (WF == CQ_Q4_1) chunk_q4_1<MT>(wc, x, M, c);
    else if constexpr (WF == CQ_Q6_K) chunk_q6_k<MT>(wc, x.xa, x.tp, M, c);
    else if constexpr (WF == CQ_Q5_K) chunk_q4_k<MT, true>(wc, x.xa, x.tp, M, c);
    else chunk_q4_k<MT, false>(wc, x.xa, x.tp, M, c);
}

// ------------------------------------------------------------------ kernel
// Warps per CTA at most (the launch bound, so the register budget). One
// token: Q8_0 and Q4_1 hold the lane's chunk of x in registers (see
// gemv_kernel) and need the registers of 16 / 20 warps; Q4_0 and Q4_K read x
// from shared memory and run 24 warps.
template <int WF, int MT> __host__ __device__ constexpr bool x_in_regs() { return MT == 1 && (WF == CQ_Q8_0 || WF == CQ_Q4_1); }
template <int WF, int MT> __host__ __device__ constexpr int wpc_limit() {
    return MT == 1 ? (WF == CQ_Q8_0 || WF == CQ_Q6_K ? 16 : WF == CQ_Q4_1 ? 20 : 24) : MT <= 4 ? WPC_MAX : WPC_MAX / 2;
}

// SWI (paired): the rows are (gate row f | up row f) of two matrices, one
// virtual row of 2 * nca chunks each; y[m][f] = silu(g) * u from the two sums.
template <int WF, int MT, bool SWI>
__global__ void __launch_bounds__(wpc_limit<WF, MT>() * 32) gemv_kernel(const GemvParams p) {
    pdl_trigger();
    using F = G<WF>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wpc = blockDim.x >> 5;
    const int64_t groups = (p.N + p.R - 1) / p.R;
    const int64_t wtot = static_cast<int64_t>(gridDim.x) * wpc;
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * wpc + warp;
    const bool active = wid < groups;
    const int64_t nsteps = active ? ((groups - 1 - wid) / wtot + 1) * p.nseg : 0;

    uint8_t* act = smem;
    uint8_t* region = smem + p.act_bytes + warp * p.warp_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(region);
    uint8_t* stages = region + 128;
    float* cbuf = reinterpret_cast<float*>(stages + p.stages * p.stage_bytes);
    const int S = p.stages;
    const uint64_t policy = policy_evict_first();

    // The warp's steps walk (group, segment) pairs: group wid, wid + wtot, ...,
    // segments 0..nseg-1 of each. Two cursors walk them without divisions: one
    // for the copies (ahead by S steps) and one for the compute.
    struct Cursor {
        int64_t g;
        int seg;
        int stage;
        uint32_t phase;
    };
    auto advance = [&](Cursor& c) {
        if (++c.seg == p.nseg) { c.seg = 0; c.g += wtot; }
        if (++c.stage == S) { c.stage = 0; c.phase ^= 1u; }
    };
    // An item is one contiguous byte range, or (paired) up to two: the gate
    // part and the up part, landing at their places in the stage.
    struct Range {
        const uint8_t* src;
        uint32_t bytes;
        uint32_t dst;
    };
    auto item = [&](const Cursor& c, Range (&r)[2]) -> int {
        const int64_t row0 = c.g * p.R;
        if constexpr (!SWI) {
            if (p.nseg == 1) {
                r[0] = {p.W + row0 * p.row_bytes,
                        static_cast<uint32_t>(min(static_cast<int64_t>(p.R), p.N - row0) * p.row_bytes), 0u};
            } else {
                const int c0 = c.seg * 32;
                r[0] = {p.W + row0 * p.row_bytes + static_cast<int64_t>(c0) * F::WCH,
                        static_cast<uint32_t>(min(32, p.nc - c0) * F::WCH), 0u};
            }
            return 1;
        } else {
            if (p.nseg == 1) {
                // R gate rows, then R up rows
                const uint32_t b = static_cast<uint32_t>(min(static_cast<int64_t>(p.R), p.N - row0) * p.wrow);
                r[0] = {p.W + row0 * p.wrow, b, 0u};
                r[1] = {p.W2 + row0 * p.wrow, b, static_cast<uint32_t>(p.R * p.wrow)};
                return 2;
            }
            const int c0 = c.seg * 32, c1 = min(c0 + 32, p.nc);
            int n = 0;
            if (c0 < p.nca)
                r[n++] = {p.W + row0 * p.wrow + static_cast<int64_t>(c0) * F::WCH,
                          static_cast<uint32_t>((min(c1, p.nca) - c0) * F::WCH), 0u};
            if (c1 > p.nca) {
                const int u0 = max(c0, p.nca);
                r[n++] = {p.W2 + row0 * p.wrow + static_cast<int64_t>(u0 - p.nca) * F::WCH,
                          static_cast<uint32_t>((c1 - u0) * F::WCH), static_cast<uint32_t>((u0 - c0) * F::WCH)};
            }
            return n;
        }
    };
    auto issue = [&](const Cursor& c) {
        Range r[2];
        const int n = item(c, r);
        uint64_t* bar = &bars[c.stage];
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, n == 2 ? r[0].bytes + r[1].bytes : r[0].bytes);
        for (int i = 0; i < n; ++i)
            bulk_g2s(stages + c.stage * p.stage_bytes + r[i].dst, r[i].src, r[i].bytes, bar, policy);
    };

    // Start the weight stream first; stage the activations while it flies.
    // Shared-memory copies of the weights may start before the preceding grid
    // has completed only when the caller has declared them constant; the L2
    // prefetch of the items after them may always (L2 is coherent, so a later
    // write by that grid still reaches the copies made after the wait).
    Cursor ic{wid, 0, 0, 0u};
    int64_t issued = 0;
    auto prefetch = [&](int64_t from, int64_t count) {
        Cursor pc = ic;
        for (int64_t j = from; j < min(from + count, nsteps); ++j) {
            Range r[2];
            const int n = item(pc, r);
            for (int i = 0; i < n; ++i) bulk_prefetch_l2(r[i].src, r[i].bytes);
            advance(pc);
        }
    };
    if (active && lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
        if (p.wconst) {
            for (; issued < min(static_cast<int64_t>(S), nsteps); ++issued) {
                issue(ic);
                advance(ic);
            }
        }
        prefetch(issued, p.l2pf + (p.wconst ? 0 : S));
    }
    pdl_wait();
    if (active && lane == 0 && !p.wconst) {
        for (; issued < min(static_cast<int64_t>(S), nsteps); ++issued) {
            issue(ic);
            advance(ic);
        }
    }
    if (p.x != nullptr)
        stage_activations_x<WF>(p, act);
    else
        stage_activations<WF>(p, act);
    __syncthreads();
    if (!active) return;

    // This lane's chunk in an item: row lr, chunk lj (one division per launch).
    const int lr = p.nseg == 1 ? lane / p.nc : 0;
    const int lj = p.nseg == 1 ? lane - lr * p.nc : lane;
    // One token and whole rows in an item: the lane's chunk of x never changes.
    constexpr bool PAIRS = WF == CQ_Q4_1;
    constexpr bool XREG = x_in_regs<WF, MT>();
    // The x chunk of virtual chunk c (paired: the up part reuses x from 0).
    auto xchunk = [&](int c) { return SWI && c >= p.nca ? c - p.nca : c; };
    // Offset of (row lr, chunk lj) in a stage: rows of row_bytes, or (paired,
    // whole rows) R gate rows then R up rows.
    auto woff = [&](int lr_, int lj_) -> int {
        if constexpr (SWI) {
            if (p.nseg == 1)
                return lj_ < p.nca ? lr_ * static_cast<int>(p.wrow) + lj_ * F::WCH
                                   : (p.R + lr_) * static_cast<int>(p.wrow) + (lj_ - p.nca) * F::WCH;
        }
        return lr_ * static_cast<int>(p.row_bytes) + lj_ * F::WCH;
    };
    RegX<PAIRS> xr;
    if (XREG && p.xreg) xr.load(act + xchunk(lj) * F::ACP);
    Cursor cc{wid, 0, 0, 0u};
    int64_t kfail = -1;
    int slot0 = 0;          // batch slots filled so far (R per row group)
    for (int64_t k = 0; k < nsteps; ++k) {
        const bool ok = mbar_wait_bounded(&bars[cc.stage], cc.phase, WAIT_LIMIT_NS);
        if (!__all_sync(0xffffffffu, ok)) { kfail = k; break; }

        const int64_t row0 = cc.g * p.R;
        const int c0 = cc.seg * 32;
        const int cn = p.nseg == 1 ? p.nc : min(32, p.nc - c0);
        const int rows_valid = static_cast<int>(min(static_cast<int64_t>(p.R), p.N - row0));
        const uint8_t* st = stages + cc.stage * p.stage_bytes;
        const bool have = lr < rows_valid && lj < cn;
        uint32_t wr[F::WR];
        if (have) chunk_load<WF>(st + woff(lr, lj), wr);
        // The stage is read: refill it before the arithmetic.
        __syncwarp();
        if (lane == 0 && issued < nsteps) {
            issue(ic);
            advance(ic);
            ++issued;
        }
        if (have) {
            float c[MT];
            const SmemX<PAIRS> xs{act + xchunk(c0 + lj) * F::ACP, p.tok_pitch};
            if constexpr (XREG) {
                if (p.xreg) chunk_value<WF, MT>(wr, xr, p.M, c);
                else chunk_value<WF, MT>(wr, xs, p.M, c);
            } else {
                chunk_value<WF, MT>(wr, xs, p.M, c);
            }
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m < p.M) cbuf[(m * p.B + slot0 + lr) * p.cpitch + c0 + lj] = c[m];
        }
        const int64_t g = cc.g;
        const bool row_done = cc.seg == p.nseg - 1;
        advance(cc);
        if (row_done) {
            slot0 += p.R;
            if (slot0 == p.B || k == nsteps - 1) {
                __syncwarp();       // every lane's chunk values are in the buffer
                // Fixed order: y = 0, then y = y + c over the row's chunks in increasing k.
                // Slot r holds row (r % R) of group g - ((slot0 - 1 - r) / R) * wtot.
                for (int q = lane; q < p.M * slot0; q += 32) {
                    const int m = q / slot0, r = q - m * slot0;
                    const float* cb = cbuf + (m * p.B + r) * p.cpitch;
                    // The sum over chunks [j0, j0 + n) of the row, x chunks from 0.
                    auto rowsum = [&](int j0, int n) {
                        float acc = 0.0f;
                        if constexpr (superblock_fmt<WF>()) {
                            // y = fma(d_x, t, y) per superblock, d_x from the staged activations
                            const uint8_t* xd = act + m * p.tok_pitch + 256;
#pragma unroll 8
                            for (int j = 0; j < n; ++j)
                                acc = __fmaf_rn(*reinterpret_cast<const float*>(xd + j * F::ACP), cb[j0 + j], acc);
                        } else {
#pragma unroll 8
                            for (int j = 0; j < n; ++j) acc = __fadd_rn(acc, cb[j0 + j]);
                        }
                        return acc;
                    };
                    float acc;
                    if constexpr (SWI) {
                        // h = silu(g) * u, silu(g) = g / (1 + exp(-g)), all fp32
                        const float gs = rowsum(0, p.nca), us = rowsum(p.nca, p.nca);
                        acc = __fmul_rn(__fdiv_rn(gs, __fadd_rn(1.0f, expf(-gs))), us);
                    } else {
                        acc = rowsum(0, p.nc);
                    }
                    const int back = (slot0 - 1 - r) / p.R;
                    const int64_t row = (g - back * wtot) * p.R + (r - (r / p.R) * p.R);
                    if (row < p.N) p.y[static_cast<int64_t>(m) * p.N + row] = acc;
                }
                slot0 = 0;
                __syncwarp();
            }
        }
    }
    if (kfail >= 0) {
        // A copy never completed: record it, then give the copies still in
        // flight (bounded) time to land before the CTA's shared memory goes.
        if (lane == 0) {
            atomicOr(p.status, CQ_DEV_WAIT_TIMEOUT);
            for (int64_t k = kfail; k < issued; ++k) {
                (void)mbar_wait_bounded(&bars[cc.stage], cc.phase, WAIT_LIMIT_NS / 8);
                advance(cc);
            }
        }
        __syncwarp();
    }
}

// Items a warp prefetches into L2 past its ring before the dependency wait,
// so DRAM stays busy while the preceding grids drain: 8 for Q8_0 (decode
// step 118.9 -> 111.7 us), 4 for the 4-bit formats, whose CTAs run more
// warps (more than that crowds the L2), none for Q6_K, whose items of four
// rows already fill the L2 at four (standalone LM head 41.0 us with none,
// 43.0 with 4, 47.1 with 8).
constexpr int l2_prefetch_items(int w_fmt) { return w_fmt == CQ_Q8_0 ? 8 : w_fmt == CQ_Q6_K ? 0 : 4; }

template <int WF, int MT, bool SWI>
cudaError_t launch_typed(const DeviceInfo& dev, GemvParams p, int64_t groups, cudaStream_t s) {
    const int lim = std::min(dev.smem_optin, 227 * 1024);
    const int budget = lim - 1024;
    // Shared memory per warp: barriers, S stages, chunk-value buffer.
    auto warp_bytes = [&](int S) { return (128 + S * p.stage_bytes + 4 * CBUF_FLOATS + 127) / 128 * 128; };
    auto warps_for = [&](int S) { return std::min(wpc_limit<WF, MT>(), (budget - p.act_bytes) / warp_bytes(S)); };
    // Two stages a warp and as many warps as fit: at equal bytes in flight,
    // deeper rings ran slower (a landed stage waits behind an earlier one).
    constexpr int S = 2;
    int wpc = warps_for(S);
    if (wpc < 1) return cudaErrorInvalidConfiguration;
    p.stages = S;
    p.warp_bytes = warp_bytes(S);
    // Balance: every warp gets the same number of row groups, give or take one,
    // spread over all SMs before warps are stacked on one SM.
    const int64_t wmax = static_cast<int64_t>(dev.sm_count) * wpc;
    const int64_t per_warp = (groups + wmax - 1) / wmax;
    const int64_t warps = (groups + per_warp - 1) / per_warp;
    wpc = static_cast<int>(std::min<int64_t>(wpc, (warps + dev.sm_count - 1) / dev.sm_count));
    const unsigned grid = static_cast<unsigned>((warps + wpc - 1) / wpc);
    const int smem = p.act_bytes + wpc * p.warp_bytes;
    const cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(gemv_kernel<WF, MT, SWI>), lim);
    if (e != cudaSuccess) return e;
    cudaError_t le = launch_kernel(gemv_kernel<WF, MT, SWI>, dim3(grid), dim3(wpc * 32), smem, s, p);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

template <int WF, bool SWI>
cudaError_t launch_fmt(const DeviceInfo& dev, const GemvParams& p, int64_t groups, cudaStream_t s) {
    if (p.M <= 1) return launch_typed<WF, 1, SWI>(dev, p, groups, s);
    if (p.M <= 4) return launch_typed<WF, 4, SWI>(dev, p, groups, s);
    if (p.M <= 8) return launch_typed<WF, 8, SWI>(dev, p, groups, s);
    return launch_typed<WF, 16, SWI>(dev, p, groups, s);
}

// W2 != null: paired (gate W, up W2), y = silu(W . x) * (W2 . x).
template <int WF>
cudaError_t launch_gemv_fmt(const DeviceInfo& dev, int M, int64_t N, int64_t K, const void* W, const void* W2,
                            const void* xq, float* y, const float* x, cudaStream_t s) {
    using F = G<WF>;
    const bool swi = W2 != nullptr;
    const int nca = static_cast<int>(K / F::CE);
    const int nc = swi ? 2 * nca : nca;
    if (nc > CBUF_FLOATS) return cudaErrorInvalidValue;
    const int64_t wrow = static_cast<int64_t>(nca) * F::WCH;
    const int64_t row_bytes = static_cast<int64_t>(nc) * F::WCH;
    const int act_row = static_cast<int>(K / CHUNK_ELEMS) * achunk_bytes(act_fmt_for(WF));
    const int tok_pitch = nca * F::ACP;
    // Tokens per launch: staged activations within 100 KB, and the chunk-value
    // buffer holding at least one row of every token.
    int max_tok = std::max(1, std::min(M, (100 * 1024) / tok_pitch));
    max_tok = std::min(max_tok, std::max(1, CBUF_FLOATS / nc));
    for (int m0 = 0; m0 < M; m0 += max_tok) {
        GemvParams p{};
        p.M = std::min(max_tok, M - m0);
        p.W = static_cast<const uint8_t*>(W);
        p.xq = static_cast<const uint8_t*>(xq) + static_cast<int64_t>(m0) * act_row;
        if (x != nullptr) {
            p.x = x + static_cast<int64_t>(m0) * K;
            p.xq_out = const_cast<uint8_t*>(p.xq);
        }
        p.y = y + static_cast<int64_t>(m0) * N;
        p.status = dev.status;
        p.N = N;
        p.row_bytes = row_bytes;
        p.nc = nc;
        p.nca = nca;
        p.W2 = static_cast<const uint8_t*>(W2);
        p.wrow = wrow;
        if (nc <= 32) {
            p.R = 32 / nc;
            p.segc = nc;
            p.nseg = 1;
        } else {
            p.R = 1;
            p.segc = 32;
            p.nseg = (nc + 31) / 32;
        }
        p.stage_bytes = static_cast<int>(((p.nseg == 1 ? p.R * row_bytes : int64_t(32) * F::WCH) + 127) / 128 * 128);
        // Rows per batch of sequential sums: a multiple of R, buffer within CBUF_FLOATS.
        // An odd row pitch in the chunk-value buffer where one item still fits.
        p.cpitch = (nc % 2 == 0 && p.R * p.M * (nc + 1) <= CBUF_FLOATS) ? nc + 1 : nc;
        const int cpitch = p.cpitch;
        const int rows_fit = CBUF_FLOATS / (p.M * cpitch);
        p.B = std::max(p.R, std::min(32, rows_fit) / p.R * p.R);
        if (p.B * p.M * cpitch > CBUF_FLOATS) return cudaErrorInvalidValue;
        p.tok_pitch = tok_pitch;
        p.xreg = x_in_regs<WF, 1>() && p.M == 1 && p.nseg == 1 ? 1 : 0;
        p.wconst = weights_const() ? 1 : 0;
        p.l2pf = l2_prefetch_items(WF);
        p.act_bytes = (p.M * tok_pitch + 127) / 128 * 128;
        const int64_t groups = (N + p.R - 1) / p.R;
        cudaError_t e = swi ? launch_fmt<WF, true>(dev, p, groups, s) : launch_fmt<WF, false>(dev, p, groups, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemv(const DeviceInfo& dev, int w_fmt, int M, int64_t N, int64_t K, const void* W,
                        const void* xq, float* y, const float* x, cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    const int afmt = act_fmt_for(w_fmt);
    if (afmt < 0) return cudaErrorInvalidValue;
    if (N <= 0) return x != nullptr ? launch_quantize(afmt, M, K, x, const_cast<void*>(xq), s) : cudaSuccess;
    // Several tokens: the tensor-core kernel when the activations fit its
    // shared memory (same fixed order, so the same bits). It stages quantized
    // activations, so fp32 ones are quantized by their own launch first. Q8_0
    // at two or three tokens stays on the dp4a kernel below, whose work per token
    // is lightest for Q8_0 (LM head 128256 x 4096: M = 2 88.2 us here against
    // 112.6 on the tensor cores, M = 3 106.5 against 112.7, M = 4 131.1
    // against 114.7; for Q4_0 and Q4_1 the tensor cores win or tie from M = 2).
    // Q4_K with many tokens: the tcgen05 prefill GEMM (its rows are the bits of
    // this kernel's). With the activation workspace from the library's pool the
    // GEMM costs the same from 1 to 128 tokens (14336 x 4096: 38.0 us; 4096 x
    // 14336: 95-97; 128256 x 4096: 202-204), and this kernel passes it at M = 7
    // for 8192 rows or more (M = 6 / 7: 38.9 / 43.0 us and 206.8 / 225.3 here)
    // and at M = 8 below (4096 x 14336: 90.1 / 100.4 us here at M = 7 / 8).
    // Without a workspace (stream capture, or the pool short of memory) the
    // GEMM converts the activations in every CTA, and the crossover measured
    // for that is M = 9 for 8192 rows or more (14336 x 4096: 47.1 us here at
    // M = 8, 41.0 through the GEMM) and M = 11 below (4096 x 14336: 110.6 /
    // 131.1 us here at M = 10 / 11, 114.7 / 116.7 through the GEMM).
    if (w_fmt == CQ_Q4_K && M >= 7) {
        const bool tall = N >= 8192;
        void* ws = M >= (tall ? 7 : 8) ? scratch_alloc(gemm_workspace_size(w_fmt, M, K), s) : nullptr;
        if (ws != nullptr || M >= 11 || (M >= 9 && tall)) {
            cudaError_t e = cudaSuccess;
            if (x != nullptr) e = launch_quantize(afmt, M, K, x, const_cast<void*>(xq), s);
            if (e == cudaSuccess) e = launch_gemm(dev, w_fmt, M, N, K, W, xq, y, ws, s);
            const cudaError_t f = scratch_free(ws, s);
            return e != cudaSuccess ? e : f;
        }
    }
    const int need = gemv_mma_smem(w_fmt, M, K);
    const bool dp4a_better = w_fmt == CQ_Q8_0 && M <= 3;
    if (M >= 2 && !dp4a_better && need > 0 && need <= std::min(dev.smem_optin, 227 * 1024)) {
        if (x != nullptr) {
            const cudaError_t e = launch_quantize(afmt, M, K, x, const_cast<void*>(xq), s);
            if (e != cudaSuccess) return e;
        }
        return launch_gemv_mma(dev, w_fmt, M, N, K, W, xq, y, s);
    }
    switch (w_fmt) {
    case CQ_Q4_0: return launch_gemv_fmt<CQ_Q4_0>(dev, M, N, K, W, nullptr, xq, y, x, s);
    case CQ_Q8_0: return launch_gemv_fmt<CQ_Q8_0>(dev, M, N, K, W, nullptr, xq, y, x, s);
    case CQ_Q4_1: return launch_gemv_fmt<CQ_Q4_1>(dev, M, N, K, W, nullptr, xq, y, x, s);
    case CQ_Q4_K: return launch_gemv_fmt<CQ_Q4_K>(dev, M, N, K, W, nullptr, xq, y, x, s);
    case CQ_Q5_K: return launch_gemv_fmt<CQ_Q5_K>(dev, M, N, K, W, nullptr, xq, y, x, s);
    case CQ_Q6_K: return launch_gemv_fmt<CQ_Q6_K>(dev, M, N, K, W, nullptr, xq, y, x, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemv_swiglu(const DeviceInfo& dev, int w_fmt, int M, int64_t F, int64_t K, const void* Wg,
                               const void* Wu, const void* xq, float* h, cudaStream_t s) {
    if (M <= 0 || F <= 0) return cudaSuccess;
    switch (w_fmt) {
    case CQ_Q4_0: return launch_gemv_fmt<CQ_Q4_0>(dev, M, F, K, Wg, Wu, xq, h, nullptr, s);
    case CQ_Q8_0: return launch_gemv_fmt<CQ_Q8_0>(dev, M, F, K, Wg, Wu, xq, h, nullptr, s);
    case CQ_Q4_1: return launch_gemv_fmt<CQ_Q4_1>(dev, M, F, K, Wg, Wu, xq, h, nullptr, s);
    case CQ_Q4_K: return launch_gemv_fmt<CQ_Q4_K>(dev, M, F, K, Wg, Wu, xq, h, nullptr, s);
    case CQ_Q5_K: return launch_gemv_fmt<CQ_Q5_K>(dev, M, F, K, Wg, Wu, xq, h, nullptr, s);
    case CQ_Q6_K: return launch_gemv_fmt<CQ_Q6_K>(dev, M, F, K, Wg, Wu, xq, h, nullptr, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace cq
