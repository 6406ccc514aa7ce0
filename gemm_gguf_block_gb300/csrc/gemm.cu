// Prefill GEMM, Q4_K weights x Q8_K activations, on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in tensor memory).
//
// alice-llm docs, "Computation Path (Q4_K)": per 256-element superblock
//   y += d_x * d * sum_j(sc_j * S_j) - d_x * dmin * sum_j(m_j * bsum_j),
// S_j the integer dot of 32-element sub-block j; cera README: batched-GEMM
// prefill, and decode matching prefill bit for bit (cera 0.5 notes).
//
// Exact integer contraction on fp16 tensor cores. tcgen05 has no int8 MMA on
// sm_103a, so the operands are fp16 values that hold integers exactly:
//   A[n][k] = sc_j(n) * q4(n, k)   in [0, 945]   (weights, MMA M = 128 rows)
//   B[m][k] = q8(m, k)             in [-127, 127] (tokens, MMA N = 128)
// A superblock's products sum to at most 30.7e6 > 2^24 in magnitude, so each
// superblock is split into two K = 128 halves, each accumulated in its own
// fp32 tensor-memory accumulator (|partial| <= 15.4e6 < 2^24: exact). The min
// term sum_j m_j * bsum_j is one more K = 16 MMA: A = [m_0..m_7, m_0..m_7],
// B = [64 h_0..64 h_7, l_0..l_7] with bsum_j = 64 h_j + l_j, all exact in fp16.
// The epilogue then applies, per (row, token, superblock), exactly the fixed
// fp32 order of include/cq.h -- RN(h0 + h1) is (float)isum_sc; then
// t = fma(d, S, -(dmin * I)) and y = fma(d_x, t, y) -- so every row equals the
// cq_gemv row bit for bit.
//
// Warp roles (576 or 832 threads): warp 0 TMA producer of raw Q4_K tiles (2-D tensor
// map, 128 rows x 144 bytes per superblock); warp 1 allocates tensor memory and
// one lane issues the MMAs; warps 2-9 convert raw weights and Q8_K
// activations into fp16 tiles in the canonical K-major no-swizzle layout;
// warps 10-17 (10-25 with the workspace) are the epilogue (tensor-memory
// lanes 32*(warp%4)...). Every wait
// is bounded; a timeout flags CQ_DEV_WAIT_TIMEOUT and the CTA winds down.
#include <algorithm>

#include <cuda_fp16.h>

#include "cq_device.cuh"
#include "cq_internal.h"
#include "tc.cuh"

namespace cq {
namespace {

constexpr int BM = 128;          // weight rows per tile (MMA M, TMEM lanes)
constexpr int BN = 128;          // tokens per tile (MMA N)
constexpr int KH = 128;          // K per operand stage (half a superblock)
constexpr int NSTAGE = 2;        // operand stages
constexpr int NRAW = 3;          // raw weight superblock stages
constexpr int RAW_BYTES = BM * 144;
constexpr int A_BYTES = BM * KH * 2;        // 32 KB
constexpr int B_BYTES = BN * KH * 2;        // 32 KB
constexpr int AMIN_BYTES = BM * 16 * 2;     // 4 KB
constexpr int BMIN_BYTES = BN * 16 * 2;     // 4 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + AMIN_BYTES + BMIN_BYTES;
constexpr int NCONV = 256;       // converter threads (warps 2-9)
// Epilogue warps (from warp 10): 16 when the activations come pre-converted
// (the converters then need few registers), each thread draining 32 token
// columns of its row per superblock in 8-column loads; else 8 warps of 64
// columns in 16-column loads.
template <bool PRE> struct Epi {
    static constexpr int WARPS = PRE ? 16 : 8;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int COLS = BN / (WARPS / 4);      // token columns per thread
    static constexpr int CW = PRE ? 8 : 16;            // columns per tensor-memory load
};
template <bool PRE> constexpr int kernel_threads() { return (2 + 8) * 32 + Epi<PRE>::THREADS; }
constexpr uint32_t TMEM_COLS = 512;         // h0 | h1 | mins | y, 128 columns each
constexpr uint32_t COL_H0 = 0, COL_H1 = 128, COL_MIN = 256, COL_Y = 384;

// Shared-memory layout (offsets from the 1024-aligned dynamic base).
constexpr int OFF_BAR = 0;                   // 16 barriers
constexpr int OFF_TMEM = 128;                // tensor-memory base address
constexpr int OFF_FLAG = 136;                // abort flag
constexpr int OFF_DX = 256;                  // [2][BN] floats
constexpr int OFF_RAW = 2048;
constexpr int OFF_STAGE = OFF_RAW + NRAW * RAW_BYTES;
constexpr int SMEM_BYTES = OFF_STAGE + NSTAGE * STAGE_BYTES + 1024;   // + alignment slack

enum { B_RAW_FULL = 0, B_RAW_EMPTY = 3, B_OP_FULL = 6, B_OP_EMPTY = 8, B_ACC_FULL = 10, B_ACC_EMPTY = 11 };

struct GemmParams {
    const uint8_t* W;
    const uint8_t* xq;
    float* y;
    int* status;
    int M, N, ns;        // tokens, rows, superblocks per row
    int64_t wrow;        // bytes per weight row
    int64_t xrow;        // bytes per activation row
    const uint8_t* bimg; // pre-converted B operands: [token tile][superblock] images of IMG_BYTES
    const float* dxs;    // pre-gathered activation scales: [token tile][superblock][BN]
};

// One (token tile, superblock) image of the pre-converted activations, laid
// out exactly as the B part of two operand stages: the K-half 0 and K-half 1
// fp16 tiles, then the mins operand.
constexpr int IMG_BYTES = 2 * (BN * KH * 2) + BN * 16 * 2;     // 69632

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Four nibble pairs (one byte each of w) -> the low nibbles as two half2 of
// sl * q and the high nibbles as two half2 of sh * q, each exact:
// (1024 + q) * s - 1024 * s in one fused multiply-add.
__device__ __forceinline__ void nibbles_to_half(uint32_t w, __half2 sl, __half2 bl, __half2 sh, __half2 bh,
                                                uint32_t (&lo)[2], uint32_t (&hi)[2]) {
    const uint32_t p01 = __byte_perm(w, 0u, 0x4140);   // bytes 0, 1 -> halves 0, 1
    const uint32_t p23 = __byte_perm(w, 0u, 0x4342);   // bytes 2, 3
    lo[0] = h2_bits(__hfma2(bits_h2((p01 & 0x000F000Fu) | 0x64006400u), sl, bl));
    lo[1] = h2_bits(__hfma2(bits_h2((p23 & 0x000F000Fu) | 0x64006400u), sl, bl));
    hi[0] = h2_bits(__hfma2(bits_h2(((p01 >> 4) & 0x000F000Fu) | 0x64006400u), sh, bh));
    hi[1] = h2_bits(__hfma2(bits_h2(((p23 >> 4) & 0x000F000Fu) | 0x64006400u), sh, bh));
}

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

// PRE: the activations come pre-converted (cq_gemm_ws): the producer
// bulk-copies each stage's B operand and the converters handle only weights.
template <bool PRE>
__global__ void __launch_bounds__(kernel_threads<PRE>(), 1) gemm_q4k_kernel(const __grid_constant__ CUtensorMap wmap,
                                                                             const GemmParams p) {
    constexpr int NEPI = Epi<PRE>::THREADS;
    pdl_trigger();
    pdl_wait();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);
    const SmemFlag abort_flag{smem_u32(smem + OFF_FLAG)};
    float* dxbuf = reinterpret_cast<float*>(smem + OFF_DX);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BM, m0 = blockIdx.y * BN;
    const int ns = p.ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NRAW; ++i) {
            mbar_init(&bars[B_RAW_FULL + i], 1);
            mbar_init(&bars[B_RAW_EMPTY + i], NCONV);
        }
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&bars[B_OP_FULL + i], PRE ? NCONV + 1 : NCONV);   // + the producer's copy
            mbar_init(&bars[B_OP_EMPTY + i], 1);
        }
        mbar_init(&bars[B_ACC_FULL], 1);
        mbar_init(&bars[B_ACC_EMPTY], NEPI);
        abort_flag.set(0);
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_holder, TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int s = 0; s < ns && !abort_flag.get(); ++s) {
                const int r = s % NRAW;
                if (!tc::wait_or_abort(&bars[B_RAW_EMPTY + r], ((s / NRAW) & 1) ^ 1, abort_flag, p.status)) break;
                mbar_arrive_expect_tx(&bars[B_RAW_FULL + r], RAW_BYTES);
                tc::tma_load_2d(smem + OFF_RAW + r * RAW_BYTES, &wmap, 144 * s, n0, &bars[B_RAW_FULL + r]);
                if constexpr (PRE) {
                    const uint8_t* img = p.bimg + (static_cast<int64_t>(blockIdx.y) * ns + s) * IMG_BYTES;
                    bool ok = true;
                    for (int h = 0; h < 2; ++h) {
                        const int q = 2 * s + h, st = q % NSTAGE;
                        if (!tc::wait_or_abort(&bars[B_OP_EMPTY + st], ((q / NSTAGE) & 1) ^ 1, abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        uint8_t* stg = smem + OFF_STAGE + st * STAGE_BYTES;
                        mbar_arrive_expect_tx(&bars[B_OP_FULL + st], B_BYTES + (h ? BMIN_BYTES : 0));
                        bulk_g2s(stg + A_BYTES, img + h * B_BYTES, B_BYTES, &bars[B_OP_FULL + st], pol);
                        if (h)
                            bulk_g2s(stg + A_BYTES + B_BYTES + AMIN_BYTES, img + 2 * B_BYTES, BMIN_BYTES,
                                     &bars[B_OP_FULL + st], pol);
                    }
                    if (!ok) break;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_f16_f32(BM, BN);
            const uint32_t stage0 = smem_u32(smem + OFF_STAGE);
            for (int s = 0; s < ns && !abort_flag.get(); ++s) {
                if (!tc::wait_or_abort(&bars[B_ACC_EMPTY], (s & 1) ^ 1, abort_flag, p.status)) break;
                bool ok = true;
                for (int h = 0; h < 2; ++h) {
                    const int q = 2 * s + h, st = q % NSTAGE;
                    if (!tc::wait_or_abort(&bars[B_OP_FULL + st], (q / NSTAGE) & 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t a0 = stage0 + st * STAGE_BYTES;
                    const uint32_t b0 = a0 + A_BYTES;
                    for (int t = 0; t < KH / 16; ++t)
                        tc::mma_f16(tmem + (h ? COL_H1 : COL_H0), tc::smem_desc(a0 + 256 * t, 128, KH * 16),
                                    tc::smem_desc(b0 + 256 * t, 128, KH * 16), idesc, t > 0);
                    if (h == 1)
                        tc::mma_f16(tmem + COL_MIN, tc::smem_desc(b0 + B_BYTES, 128, 256),
                                    tc::smem_desc(b0 + B_BYTES + AMIN_BYTES, 128, 256), idesc, 0);
                    tc::commit(&bars[B_OP_EMPTY + st]);
                }
                if (!ok) break;
                tc::commit(&bars[B_ACC_FULL]);
            }
        }
    } else if (warp < 10) {
        // --------------------------------------------------------- converters
        // Weights: a thread pair per weight row (one 64-element group each),
        // from the raw stage in shared memory. Activations: warp w converts
        // tokens 16w..16w+15; each load instruction reads 16 bytes of 8 tokens
        // (few cache lines) and each store fills whole core-matrix rows; the
        // next stage's words are loaded one stage ahead.
        const int tid = threadIdx.x - 64;               // 0..255
        const int r = tid >> 1, part = tid & 1;         // weight row r, group part
        const int cw = warp - 2;                        // converter warp 0..7
        const int a_row = (r >> 3) * (KH * 16) + (r & 7) * 16 + part * 1024;   // A tile row base (+ k offsets)
        uint32_t cur[16], nxt[16], bcur[4], bnxt[4];
        auto fetch = [&](int q, uint32_t (&dst)[16], uint32_t (&bs)[4]) {
            const int s = q >> 1, h = q & 1;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int token = m0 + 16 * cw + 8 * (i & 1) + (lane & 7);
                const int word = 4 * (i >> 1) + (lane >> 3);
                dst[i] = token < p.M ? __ldg(reinterpret_cast<const uint32_t*>(
                                           p.xq + static_cast<int64_t>(token) * p.xrow + 292 * s + 4 + 128 * h) + word)
                                     : 0u;
            }
            if (h == 1) {
                // bsum words: token 16cw + 4i + (lane >> 3), word lane & 7
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int token = m0 + 16 * cw + 4 * i + (lane >> 3);
                    bs[i] = token < p.M ? __ldg(reinterpret_cast<const uint32_t*>(
                                              p.xq + static_cast<int64_t>(token) * p.xrow + 292 * s + 260) + (lane & 7))
                                        : 0u;
                }
            }
        };
        if constexpr (!PRE) fetch(0, cur, bcur);
        for (int q = 0; q < 2 * ns; ++q) {
            const int s = q >> 1, h = q & 1, st = q % NSTAGE, rs = s % NRAW;
            if (abort_flag.get()) break;
            if constexpr (!PRE)
                if (q + 1 < 2 * ns) fetch(q + 1, nxt, bnxt);
            if (!tc::wait_or_abort(&bars[B_OP_EMPTY + st], ((q / NSTAGE) & 1) ^ 1, abort_flag, p.status)) break;
            if (!tc::wait_or_abort(&bars[B_RAW_FULL + rs], (s / NRAW) & 1, abort_flag, p.status)) break;
            uint8_t* stg = smem + OFF_STAGE + st * STAGE_BYTES;
            // A: weight row r, group g = 2h + part: 32 low nibbles (sub-block 2g) and
            // 32 high nibbles (sub-block 2g + 1)
            const uint8_t* raw = smem + OFF_RAW + rs * RAW_BYTES + r * 144;
            const uint4 hdr = *reinterpret_cast<const uint4*>(raw);
            {
                const int g = 2 * h + part;
                int sc_lo, sc_hi, mn_unused;
                q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * g, sc_lo, mn_unused);
                q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * g + 1, sc_hi, mn_unused);
                const __half2 slo = __half2half2(__int2half_rn(sc_lo));
                const __half2 shi = __half2half2(__int2half_rn(sc_hi));
                const __half2 blo = __half2half2(__int2half_rn(-1024 * sc_lo));
                const __half2 bhi = __half2half2(__int2half_rn(-1024 * sc_hi));
                const uint4 q0 = *reinterpret_cast<const uint4*>(raw + 16 + 32 * g);
                const uint4 q1 = *reinterpret_cast<const uint4*>(raw + 32 + 32 * g);
                const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                uint8_t* arow = stg + a_row;
#pragma unroll
                for (int c = 0; c < 4; ++c) {        // 8 elements (2 words) per core-matrix row
                    uint32_t l0[2], h0[2], l1[2], h1[2];
                    nibbles_to_half(qw[2 * c], slo, blo, shi, bhi, l0, h0);
                    nibbles_to_half(qw[2 * c + 1], slo, blo, shi, bhi, l1, h1);
                    *reinterpret_cast<uint4*>(arow + c * 128) = make_uint4(l0[0], l0[1], l1[0], l1[1]);
                    *reinterpret_cast<uint4*>(arow + (4 + c) * 128) = make_uint4(h0[0], h0[1], h1[0], h1[1]);
                }
            }
            // B: tokens 16cw .. 16cw + 15; load i holds token 16cw + 8(i&1) + lane%8,
            // quant word 4(i>>1) + lane/8 (elements 4*word .. +3 of the half), so a
            // half-warp's 8-byte stores fill one 128-byte core matrix.
            uint8_t* bt = stg + A_BYTES;
#pragma unroll
            for (int i = 0; i < 16 && !PRE; ++i) {
                const int t = 16 * cw + 8 * (i & 1) + (lane & 7);
                const int word = 4 * (i >> 1) + (lane >> 3);
                uint32_t o[2];
                tc::s8x4_half(cur[i], o[0], o[1]);
                *reinterpret_cast<uint2*>(bt + (t >> 3) * (KH * 16) + (t & 7) * 16 + (word >> 1) * 128 +
                                          (word & 1) * 8) = make_uint2(o[0], o[1]);
            }
            if (h == 1) {
                // mins MMA operands: A_min row r = [m_0..m_7, m_0..m_7] (part 0 threads),
                // B_min token t = [64 h_0 .. 64 h_7, l_0 .. l_7], bsum pair j = 64 h_j + l_j
                uint8_t* am = bt + B_BYTES;
                uint8_t* bm = am + AMIN_BYTES;
                if (part == 0) {
                    uint32_t mw[4];
#pragma unroll
                    for (int j = 0; j < 8; j += 2) {
                        int sc0, mn0, sc1, mn1;
                        q4k_scale_min(hdr.y, hdr.z, hdr.w, j, sc0, mn0);
                        q4k_scale_min(hdr.y, hdr.z, hdr.w, j + 1, sc1, mn1);
                        mw[j / 2] = h2_bits(__halves2half2(__int2half_rn(mn0), __int2half_rn(mn1)));
                    }
                    const uint4 mv = make_uint4(mw[0], mw[1], mw[2], mw[3]);
                    *reinterpret_cast<uint4*>(am + tc::tile_off(r, 0, 16)) = mv;
                    *reinterpret_cast<uint4*>(am + tc::tile_off(r, 8, 16)) = mv;
                }
#pragma unroll
                for (int i = 0; i < 4 && !PRE; ++i) {
                    const int t = 16 * cw + 4 * i + (lane >> 3), j = lane & 7;
                    const uint32_t v = bcur[i];
                    const int pr = static_cast<int>(static_cast<int16_t>(v & 0xffffu)) +
                                   static_cast<int>(static_cast<int16_t>(v >> 16));
                    const int hq = pr >> 6;                                  // floor division by 64
                    __half* bh = reinterpret_cast<__half*>(bm + tc::tile_off(t, 0, 16));
                    bh[j] = __int2half_rn(64 * hq);
                    bh[64 + j] = __int2half_rn(pr - 64 * hq);                // k = 8 + j: next core matrix (+128 B)
                }
            }
            fence_proxy_async_smem();
            tc::mbar_arrive(&bars[B_OP_FULL + st]);
            if (h == 1) tc::mbar_arrive(&bars[B_RAW_EMPTY + rs]);
#pragma unroll
            for (int i = 0; i < 16; ++i) cur[i] = nxt[i];
#pragma unroll
            for (int i = 0; i < 4; ++i) bcur[i] = bnxt[i];
        }
    } else {
        // ----------------------------------------------------------- epilogue
        // Warp w reads tensor-memory lanes 32*(w%4)..+31 (weight rows); the
        // warps of column group (w-10)/4 take COLS consecutive token columns.
        constexpr int COLS = Epi<PRE>::COLS, CW = Epi<PRE>::CW;
        const int et = threadIdx.x - 320;               // 0..NEPI-1
        const int quarter = warp & 3;
        const int c0 = ((warp - 10) >> 2) * COLS;       // first token column of this warp
        const int row = n0 + quarter * 32 + lane;
        const bool row_ok = row < p.N;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const int token = m0 + et;                      // et < 128: loads one token's scale
        auto fetch_scales = [&](int s, float& dxv, uint32_t& ddv) {
            if constexpr (PRE)
                dxv = et < BN ? __ldg(p.dxs + (static_cast<int64_t>(blockIdx.y) * ns + s) * BN + et) : 0.0f;
            else
                dxv = (et < BN && token < p.M)
                          ? __ldg(reinterpret_cast<const float*>(p.xq + static_cast<int64_t>(token) * p.xrow +
                                                                 292 * s))
                          : 0.0f;
            ddv = row_ok ? __ldg(reinterpret_cast<const uint32_t*>(p.W + row * p.wrow + 144 * s)) : 0u;
        };
        float dx_next;
        uint32_t dd_next;
        fetch_scales(0, dx_next, dd_next);
        float yr[PRE ? COLS : 1];                       // PRE: this thread's outputs
#pragma unroll
        for (int i = 0; i < (PRE ? COLS : 1); ++i) yr[i] = 0.0f;
        for (int s = 0; s < ns; ++s) {
            // this superblock's activation scales and row scales, fetched one superblock ahead
            if (et < BN) dxbuf[(s & 1) * BN + et] = dx_next;
            const uint32_t dd = dd_next;
            if (s + 1 < ns) fetch_scales(s + 1, dx_next, dd_next);
            const float d = h2f(dd), ndmin = -h2f(dd >> 16);
            // A bounded wait, then one decision for all epilogue warps (the named
            // barrier also publishes dxbuf).
            const bool got = mbar_wait_bounded(&bars[B_ACC_FULL], s & 1, WAIT_LIMIT_NS);
            if (!tc::named_and(1, NEPI, got)) {
                if (et == 0) { abort_flag.set(1); atomicOr(p.status, CQ_DEV_WAIT_TIMEOUT); }
                break;
            }
            tc::fence_after();
            // Fixed order: t = fma(d, RN(h0 + h1), -(dmin * I)); y = fma(d_x, t, y).
            const uint64_t d2 = tc::pk(d, d), nm2 = tc::pk(ndmin, ndmin);
            const float2* dx2 = reinterpret_cast<const float2*>(dxbuf + (s & 1) * BN + c0);
            if constexpr (PRE) {
                // y stays in registers (COLS per thread); three loads per chunk.
#pragma unroll
                for (int cb = 0; cb < COLS; cb += CW) {
                    uint32_t h0[CW], h1[CW], mi[CW];
                    tc::ldw<CW>(lane_addr + COL_H0 + c0 + cb, h0);
                    tc::ldw<CW>(lane_addr + COL_H1 + c0 + cb, h1);
                    tc::ldw<CW>(lane_addr + COL_MIN + c0 + cb, mi);
                    tc::wait_ld();
#pragma unroll
                    for (int i = 0; i < CW; i += 2) {
                        const uint64_t S = tc::add2(tc::pk(__uint_as_float(h0[i]), __uint_as_float(h0[i + 1])),
                                                    tc::pk(__uint_as_float(h1[i]), __uint_as_float(h1[i + 1])));
                        const uint64_t tn =
                            tc::mul2(nm2, tc::pk(__uint_as_float(mi[i]), __uint_as_float(mi[i + 1])));
                        const uint64_t t = tc::fma2(d2, S, tn);
                        const float2 x = dx2[(cb + i) >> 1];
                        tc::upk(tc::fma2(tc::pk(x.x, x.y), t, tc::pk(yr[cb + i], yr[cb + i + 1])), yr[cb + i],
                                yr[cb + i + 1]);
                    }
                }
            } else {
#pragma unroll 1
                for (int cb = 0; cb < COLS; cb += CW) {
                    uint32_t h0[CW], h1[CW], mi[CW], yv[CW];
                    tc::ldw<CW>(lane_addr + COL_H0 + c0 + cb, h0);
                    tc::ldw<CW>(lane_addr + COL_H1 + c0 + cb, h1);
                    tc::ldw<CW>(lane_addr + COL_MIN + c0 + cb, mi);
                    if (s > 0) tc::ldw<CW>(lane_addr + COL_Y + c0 + cb, yv);
                    tc::wait_ld();
#pragma unroll
                    for (int i = 0; i < CW; i += 2) {
                        const uint64_t S = tc::add2(tc::pk(__uint_as_float(h0[i]), __uint_as_float(h0[i + 1])),
                                                    tc::pk(__uint_as_float(h1[i]), __uint_as_float(h1[i + 1])));
                        const uint64_t tn =
                            tc::mul2(nm2, tc::pk(__uint_as_float(mi[i]), __uint_as_float(mi[i + 1])));
                        const uint64_t t = tc::fma2(d2, S, tn);
                        const float2 x = dx2[(cb + i) >> 1];
                        const uint64_t yp = s > 0 ? tc::pk(__uint_as_float(yv[i]), __uint_as_float(yv[i + 1]))
                                                  : tc::pk(0.0f, 0.0f);
                        float lo, hi;
                        tc::upk(tc::fma2(tc::pk(x.x, x.y), t, yp), lo, hi);
                        yv[i] = __float_as_uint(lo);
                        yv[i + 1] = __float_as_uint(hi);
                    }
                    tc::stw<CW>(lane_addr + COL_Y + c0 + cb, yv);
                }
                tc::wait_st();
            }
            tc::fence_before();
            tc::mbar_arrive(&bars[B_ACC_EMPTY]);
        }
        if (__all_sync(0xffffffffu, !abort_flag.get())) {
            // y[m][n] for this row: a warp's stores to one token are 32 consecutive floats.
            if constexpr (PRE) {
                if (row_ok) {
#pragma unroll
                    for (int i = 0; i < COLS; ++i) {
                        const int m = m0 + c0 + i;
                        if (m < p.M) p.y[static_cast<int64_t>(m) * p.N + row] = yr[i];
                    }
                }
            } else {
                for (int cb = 0; cb < COLS; cb += CW) {
                    uint32_t yv[CW];
                    tc::ldw<CW>(lane_addr + COL_Y + c0 + cb, yv);
                    tc::wait_ld();
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < CW; ++i) {
                            const int m = m0 + c0 + cb + i;
                            if (m < p.M) p.y[static_cast<int64_t>(m) * p.N + row] = __uint_as_float(yv[i]);
                        }
                    }
                }
            }
        }
    }

    // Wind down: every role has left its loop; make sure no copy or MMA is in
    // flight before the tensor memory and the CTA's shared memory go.
    tc::fence_before();
    __syncthreads();
    if (abort_flag.get() && threadIdx.x == 0) {
        for (int i = 0; i < NRAW; ++i) (void)mbar_wait_bounded(&bars[B_RAW_FULL + i], 0, WAIT_LIMIT_NS / 8);
        (void)mbar_wait_bounded(&bars[B_ACC_FULL], 0, WAIT_LIMIT_NS / 8);
    }
    __syncthreads();
    tc::fence_after();
    if (warp == 1) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// Pre-conversion of Q8_K activations for cq_gemm_ws: one CTA per (superblock
// s, token tile), thread (token t, K-half h). Writes the tile's B operand
// images -- the same values and layout the in-kernel converters produce --
// and the activation scales.
__global__ void __launch_bounds__(256) gemm_prep_kernel(const GemmParams p, uint8_t* bimg, float* dxs) {
    pdl_trigger();
    pdl_wait();
    const int s = blockIdx.x, tile = blockIdx.y, ns = p.ns;
    const int t = threadIdx.x >> 1, h = threadIdx.x & 1;
    const int m = tile * BN + t;
    const bool on = m < p.M;
    const uint8_t* blk = p.xq + static_cast<int64_t>(m) * p.xrow + 292 * s;
    uint8_t* img = bimg + (static_cast<int64_t>(tile) * ns + s) * IMG_BYTES;
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(blk + 4 + 128 * h);
    uint8_t* bt = img + h * (BN * KH * 2);
#pragma unroll 4
    for (int g = 0; g < KH / 8; ++g) {       // 8 elements (one core-matrix row) per store
        uint32_t o0[2] = {0u, 0u}, o1[2] = {0u, 0u};
        if (on) {
            tc::s8x4_half(__ldg(qw + 2 * g), o0[0], o0[1]);
            tc::s8x4_half(__ldg(qw + 2 * g + 1), o1[0], o1[1]);
        }
        *reinterpret_cast<uint4*>(bt + tc::tile_off(t, 8 * g, KH)) = make_uint4(o0[0], o0[1], o1[0], o1[1]);
    }
    if (h == 0) {
        dxs[(static_cast<int64_t>(tile) * ns + s) * BN + t] = on ? __ldg(reinterpret_cast<const float*>(blk)) : 0.0f;
    } else {
        // mins operand: token t = [64 h_0 .. 64 h_7, l_0 .. l_7], bsum pair j = 64 h_j + l_j
        __half* bh = reinterpret_cast<__half*>(img + 2 * (BN * KH * 2) + tc::tile_off(t, 0, 16));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int pr = 0;
            if (on) {
                const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(blk + 260) + j);
                pr = static_cast<int>(static_cast<int16_t>(v & 0xffffu)) + static_cast<int>(static_cast<int16_t>(v >> 16));
            }
            const int hq = pr >> 6;                                  // floor division by 64
            bh[j] = __int2half_rn(64 * hq);
            bh[64 + j] = __int2half_rn(pr - 64 * hq);                // k = 8 + j: next core matrix (+128 B)
        }
    }
}

// ------------------------------------------------------------ host side
}  // namespace

size_t gemm_workspace_size(int w_fmt, int64_t M, int64_t K) {
    if (w_fmt != CQ_Q4_K) return gemm32_workspace_size(w_fmt, M, K);
    if (M <= 0) return 0;
    const int64_t cells = (M + BN - 1) / BN * (K / 256);
    return static_cast<size_t>(cells) * (IMG_BYTES + BN * 4);
}

cudaError_t launch_gemm(const DeviceInfo& dev, int w_fmt, int64_t M, int64_t N, int64_t K, const void* W,
                        const void* xq, float* y, void* workspace, cudaStream_t s) {
    if (w_fmt != CQ_Q4_K) return cudaErrorInvalidValue;
    if (M <= 0 || N <= 0) return cudaSuccess;
    tc::EncodeTiledFn enc = tc::encode_tiled_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    GemmParams p{};
    p.W = static_cast<const uint8_t*>(W);
    p.xq = static_cast<const uint8_t*>(xq);
    p.y = y;
    p.status = dev.status;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.ns = static_cast<int>(K / 256);
    p.wrow = static_cast<int64_t>(p.ns) * 144;
    p.xrow = static_cast<int64_t>(p.ns) * 292;
    const int tiles_m = static_cast<int>((M + BN - 1) / BN);
    if (workspace != nullptr) {
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        p.bimg = ws;
        p.dxs = reinterpret_cast<const float*>(ws + static_cast<int64_t>(tiles_m) * p.ns * IMG_BYTES);
    }
    // Raw weights as a 2-D byte tensor [N rows][wrow bytes]; a box is one
    // superblock (144 bytes) of 128 rows; rows past N read as zero.
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.wrow), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.wrow)};
    const cuuint32_t box[2] = {144, BM};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(W), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (SMEM_BYTES > dev.smem_optin) return cudaErrorInvalidConfiguration;
    const int pre = workspace != nullptr;
    cudaError_t e = raise_smem_limit(
        reinterpret_cast<const void*>(pre ? gemm_q4k_kernel<true> : gemm_q4k_kernel<false>), SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>((N + BM - 1) / BM), static_cast<unsigned>(tiles_m));
    if (pre) {
        e = launch_kernel(gemm_prep_kernel, dim3(static_cast<unsigned>(p.ns), static_cast<unsigned>(tiles_m)),
                          dim3(256), 0, s, p, const_cast<uint8_t*>(p.bimg), const_cast<float*>(p.dxs));
        if (e != cudaSuccess) return e;
        return launch_kernel(gemm_q4k_kernel<true>, grid, dim3(kernel_threads<true>()), SMEM_BYTES, s, map, p);
    }
    return launch_kernel(gemm_q4k_kernel<false>, grid, dim3(kernel_threads<false>()), SMEM_BYTES, s, map, p);
}

}  // namespace cq
