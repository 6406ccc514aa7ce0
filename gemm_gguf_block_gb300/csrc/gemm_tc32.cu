// Prefill GEMM of Q4_0, Q4_1 and Q8_0 weights on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in tensor memory), with a workspace.
//
// cera README "Supported models": prompts are prefilled by a batched GEMM;
// cera 0.5.3 README "Breaking changes in 0.4.0": the batched and the
// per-token paths give the same bits. The library's fixed fp32 order
// (include/cq.h) needs the exact integer dot of every 32-element block on its
// own -- c = fma(D(d_w) * D(d_x), isum, c) [+ fma(D(m_w), D(s_x), c)] per
// block, y = y + c per four blocks -- so every block gets its own accumulator:
//   A[n][k] = q(n, k) as fp16 (the weight quant's integer value: Q8_0 int8,
//             Q4_0 nibble - 8, Q4_1 nibble; exact), MMA M = 128 rows
//   B[m][k] = q8(m, k) as fp16 (exact), MMA N = 64 tokens
// and |isum| <= 32 * 127 * 127 < 2^24, so each fp32 accumulator holds the
// exact integer. One chunk (four blocks) uses 4 x 64 tensor-memory columns;
// two chunk slots fill the 512 columns, so the MMAs of one chunk run while the
// epilogue drains the other.
//
// Warp roles (832 threads): warp 0 is the producer (TMA boxes of raw weights,
// 128 rows x 8 blocks, and bulk copies of the activation images that
// gemm32_tc_prep_kernel wrote into the workspace); warp 1 allocates tensor
// memory and one lane issues the MMAs; warps 2-9 convert the raw weights to
// the fp16 A tile (K-major, no swizzle) and the per-row scale table; warps
// 10-25 are the epilogue: tensor-memory lanes 32*(warp%4).. (weight rows),
// 16 token columns each, read as 16x256b fragments, y in registers. Every wait is bounded; a timeout
// flags CQ_DEV_WAIT_TIMEOUT and the CTA winds down.
#include <algorithm>

#include <cuda_fp16.h>

#include "cq_device.cuh"
#include "cq_internal.h"
#include "mma_frag.cuh"
#include "tc.cuh"

namespace cq {
namespace {

using mf::MF;

constexpr int BM = 128;          // weight rows per tile (MMA M, tensor-memory lanes)
constexpr int BN = 64;           // tokens per tile (MMA N)
constexpr int KC = 128;          // K per chunk: four 32-blocks
// Raw stages (one 8-block segment each): two, except for Q4_1 without a
// workspace, where one raw stage and three operand stages measured faster
// (M=512 N=14336 K=4096: 268.2 against 278.4 us; for Q8_0 the second raw
// stage is worth more: 237.5 against 255.0 us).
__host__ __device__ constexpr int nraw(bool pre, int abb) { return !pre && abb == 36 ? 1 : 2; }
// Operand stages (one chunk each): three, unless the raw stages also hold the
// tokens' activation blocks (no workspace) and three no longer fit.
constexpr int NCONV = 256;       // converter threads (warps 2-9)
constexpr int EPI_WARPS = 16;
constexpr int THREADS = (2 + 8 + EPI_WARPS) * 32;
constexpr int EPI_COLS = BN / (EPI_WARPS / 4);          // 16 token columns per epilogue warp
constexpr uint32_t TMEM_COLS = 512;                     // 2 chunk slots x 4 blocks x 64 columns
constexpr int A_BYTES = BM * KC * 2;                    // 32 KB
constexpr int B_BYTES = BN * KC * 2;                    // 16 KB

// Activation image of (64-token tile, chunk): the B tile, then d_x [4][64]
// and, for Q8_1, s_x [4][64] (fp32).
__host__ __device__ constexpr int img_bytes(bool q8_1) { return B_BYTES + (q8_1 ? 2 : 1) * 4 * BN * 4; }
// Per-row scales of a chunk: d_w [4][128] and, for Q4_1, m_w [4][128] (fp32).
__host__ __device__ constexpr int wsc_bytes(bool q4_1) { return (q4_1 ? 2 : 1) * 4 * BM * 4; }
__host__ __device__ constexpr int op_bytes(bool q4_1) { return A_BYTES + img_bytes(q4_1) + wsc_bytes(q4_1); }
__host__ __device__ constexpr int raw_bytes(int bb) { return BM * mf::stage_pitch(bb); }
// Raw activation box of one segment (64 tokens x 8 blocks), without a workspace.
__host__ __device__ constexpr int rawact_bytes(int abb) { return BN * 8 * abb; }
__host__ __device__ constexpr int raw_stage_bytes(bool pre, int bb, int abb) {
    return raw_bytes(bb) + (pre ? 0 : rawact_bytes(abb));
}

enum { B_RAW_FULL = 0, B_RAW_EMPTY = 2, B_OP_FULL = 4, B_OP_EMPTY = 7, B_ACC_FULL = 10, B_ACC_EMPTY = 12 };
constexpr int OFF_BAR = 0;
constexpr int OFF_TMEM = 128;
constexpr int OFF_FLAG = 136;
constexpr int OFF_RAW = 1024;
__host__ __device__ constexpr int off_op(bool pre, int bb, int abb) {
    return OFF_RAW + nraw(pre, abb) * raw_stage_bytes(pre, bb, abb);
}
__host__ __device__ constexpr int smem_with(int nop, bool pre, int bb, int abb) {
    return off_op(pre, bb, abb) + nop * op_bytes(abb == 36) + 1024;   // + alignment slack of the dynamic base
}
__host__ __device__ constexpr int nop(bool pre, int bb, int abb) {
    return smem_with(3, pre, bb, abb) <= 227 * 1024 ? 3 : 2;
}
__host__ __device__ constexpr int smem_bytes(bool pre, int bb, int abb) {
    return smem_with(nop(pre, bb, abb), pre, bb, abb);
}

struct Tc32Params {
    const uint8_t* xq;
    const uint8_t* img;     // workspace: [token tile][chunk] activation images
    float* y;
    int* status;
    int M, N;
    int nb;                 // 32-blocks per row
    int nchunk;             // chunks (128 columns) per row
};

// Nibbles of four bytes (selected by shift 0 = low, 4 = high) -> two half2
// holding nibble - off (off = 1024 + bias: Q4_0 1032, Q4_1 1024).
__device__ __forceinline__ void nib4_half(uint32_t w, int shift, __half2 off, uint32_t& o0, uint32_t& o1) {
    const uint32_t n = (w >> shift) & 0x0F0F0F0Fu;
    o0 = mf::h2u(__hsub2(mf::u2h(__byte_perm(n, 0x64646464u, 0x4140)), off));
    o1 = mf::h2u(__hsub2(mf::u2h(__byte_perm(n, 0x64646464u, 0x4342)), off));
}

// Four bytes at byte offset B (even) of a register window of words.
template <int B, int NW>
__device__ __forceinline__ uint32_t win_u32(const uint32_t (&w)[NW]) {
    static_assert(B + 4 <= 4 * NW, "window too short");
    if constexpr (B % 4 == 0) return w[B / 4];
    else return __funnelshift_r(w[B / 4], w[B / 4 + 1], 8 * (B % 4));
}
template <int B, int NW>
__device__ __forceinline__ uint32_t win_u16(const uint32_t (&w)[NW]) {
    static_assert(B % 2 == 0 && B + 2 <= 4 * NW, "bad half-word offset");
    return B % 4 == 0 ? (w[B / 4] & 0xffffu) : (w[B / 4] >> 16);
}

// One weight block starting at byte BASE of the window: its 32 quants as
// four 8-element core-matrix rows of the A tile (dst = the block's first
// row), and its d_w (and m_w for Q4_1).
template <int WF, int BASE, int NW>
__device__ __forceinline__ void convert_block(const uint32_t (&w)[NW], uint8_t* dst, float& d, float& mn) {
    if constexpr (WF == CQ_Q8_0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t o[4];
            // i is unrolled: the offsets are compile-time after unrolling
            const uint32_t a = i == 0 ? win_u32<BASE + 2, NW>(w) : i == 1 ? win_u32<BASE + 10, NW>(w)
                             : i == 2 ? win_u32<BASE + 18, NW>(w) : win_u32<BASE + 26, NW>(w);
            const uint32_t b = i == 0 ? win_u32<BASE + 6, NW>(w) : i == 1 ? win_u32<BASE + 14, NW>(w)
                             : i == 2 ? win_u32<BASE + 22, NW>(w) : win_u32<BASE + 30, NW>(w);
            tc::s8x4_half(a, o[0], o[1]);
            tc::s8x4_half(b, o[2], o[3]);
            *reinterpret_cast<uint4*>(dst + 128 * i) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        d = h2f(win_u16<BASE, NW>(w));
        mn = 0.0f;
    } else {
        constexpr bool Q41 = WF == CQ_Q4_1;
        constexpr int QO = Q41 ? 4 : 2;
        const __half2 off = mf::u2h(Q41 ? 0x64006400u : 0x64086408u);   // 1024 or 1032
        const uint32_t q[4] = {win_u32<BASE + QO, NW>(w), win_u32<BASE + QO + 4, NW>(w),
                               win_u32<BASE + QO + 8, NW>(w), win_u32<BASE + QO + 12, NW>(w)};
        // core rows 0, 1: low nibbles of bytes 0-7, 8-15; rows 2, 3: high nibbles
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int sh = i < 2 ? 0 : 4, wi = 2 * (i & 1);
            uint32_t o[4];
            nib4_half(q[wi], sh, off, o[0], o[1]);
            nib4_half(q[wi + 1], sh, off, o[2], o[3]);
            *reinterpret_cast<uint4*>(dst + 128 * i) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if constexpr (Q41) {
            const uint32_t dm = win_u32<BASE, NW>(w);
            d = h2f(dm);
            mn = h2f(dm >> 16);
        } else {
            d = h2f(win_u16<BASE, NW>(w));
            mn = 0.0f;
        }
    }
}

// A converter thread's two consecutive blocks, which start at byte OFF of its
// 16-byte-aligned window.
template <int WF, int OFF, int NW>
__device__ __forceinline__ void convert_pair(const uint32_t (&w)[NW], uint8_t* dst, float (&d)[2], float (&mn)[2]) {
    constexpr int BB = MF<WF>::BB;
    static_assert(OFF + 2 * BB <= 4 * NW, "the window must hold both blocks");
    convert_block<WF, OFF, NW>(w, dst, d[0], mn[0]);
    convert_block<WF, OFF + BB, NW>(w, dst + 512, d[1], mn[1]);   // next block: 4 core matrices on
}

// One activation block (Q8_0, or Q8_1 for Q4_1 weights) starting at byte OFF
// of a 48-byte register window: its 32 quants as fp16 into four core-matrix
// rows of the B tile (dst = the block's first row), its d_x (and s_x) into
// the image's scale tables -- the values gemm32_tc_prep_kernel writes.
template <int WF, int OFF>
__device__ __forceinline__ void convert_act(const uint32_t (&w)[12], uint8_t* dst, float* dx, float* sx) {
    constexpr int AQO = MF<WF>::AQO;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t o[4];
        const uint32_t a = i == 0 ? win_u32<OFF + AQO, 12>(w) : i == 1 ? win_u32<OFF + AQO + 8, 12>(w)
                         : i == 2 ? win_u32<OFF + AQO + 16, 12>(w) : win_u32<OFF + AQO + 24, 12>(w);
        const uint32_t b = i == 0 ? win_u32<OFF + AQO + 4, 12>(w) : i == 1 ? win_u32<OFF + AQO + 12, 12>(w)
                         : i == 2 ? win_u32<OFF + AQO + 20, 12>(w) : win_u32<OFF + AQO + 28, 12>(w);
        tc::s8x4_half(a, o[0], o[1]);
        tc::s8x4_half(b, o[2], o[3]);
        *reinterpret_cast<uint4*>(dst + 128 * i) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    *dx = h2f(win_u16<OFF, 12>(w));
    if constexpr (WF == CQ_Q4_1) *sx = h2f(win_u16<OFF + 2, 12>(w));
}

// PRE: the activation images come from the workspace (bulk copies);
// otherwise the producer also loads the tokens' raw activation blocks with
// each weight segment and the converters build the image in every CTA.
template <int WF, bool PRE>
__global__ void __launch_bounds__(THREADS, 1) gemm32_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                                                               const __grid_constant__ CUtensorMap amap,
                                                               const Tc32Params p) {
    pdl_trigger();
    pdl_wait();
    using F = MF<WF>;
    constexpr bool Q41 = WF == CQ_Q4_1;
    constexpr int PITCH = mf::stage_pitch(F::BB);
    constexpr int RAWB = raw_bytes(F::BB);
    constexpr int RSB = raw_stage_bytes(PRE, F::BB, F::ABB);
    constexpr int IMG = img_bytes(Q41);
    constexpr int OPB = op_bytes(Q41);
    constexpr int NOP = nop(PRE, F::BB, F::ABB);
    constexpr int NRAW = nraw(PRE, F::ABB);
    constexpr int OFF_OP = off_op(PRE, F::BB, F::ABB);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);
    const SmemFlag abort_flag{smem_u32(smem + OFF_FLAG)};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BN, n0 = blockIdx.y * BM;
    const int nq = p.nchunk;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NRAW; ++i) {
            mbar_init(&bars[B_RAW_FULL + i], 1);
            mbar_init(&bars[B_RAW_EMPTY + i], NCONV);
        }
        for (int i = 0; i < NOP; ++i) {
            mbar_init(&bars[B_OP_FULL + i], NCONV + (PRE ? 1 : 0));   // converters (+ the producer's image copy)
            mbar_init(&bars[B_OP_EMPTY + i], 1 + EPI_WARPS);   // the MMA commit + the epilogue's scale reads
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[B_ACC_FULL + i], 1);
            mbar_init(&bars[B_ACC_EMPTY + i], EPI_WARPS);
        }
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
        // ------------------------------------------------------ producer
        if (lane == 0) {
            for (int s = 0; 2 * s < nq && !abort_flag.get(); ++s) {
                const int r = s % NRAW;
                if (!tc::wait_or_abort(&bars[B_RAW_EMPTY + r], ((s / NRAW) & 1) ^ 1, abort_flag, p.status)) break;
                mbar_arrive_expect_tx(&bars[B_RAW_FULL + r], RSB);
                tc::tma_load_2d(smem + OFF_RAW + r * RSB, &wmap, s * 8 * F::BB / 2, n0, &bars[B_RAW_FULL + r]);
                if constexpr (!PRE) {
                    // the tokens' 8 activation blocks of this segment; tokens past M read as zero
                    tc::tma_load_2d(smem + OFF_RAW + r * RSB + RAWB, &amap, s * 8 * F::ABB / 2, m0,
                                    &bars[B_RAW_FULL + r]);
                    continue;
                }
                bool ok = true;
                for (int h = 0; h < 2; ++h) {
                    const int q = 2 * s + h, st = q % NOP;
                    if (!tc::wait_or_abort(&bars[B_OP_EMPTY + st], ((q / NOP) & 1) ^ 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars[B_OP_FULL + st], IMG);
                    bulk_g2s(smem + OFF_OP + st * OPB + A_BYTES,
                             p.img + (static_cast<int64_t>(blockIdx.x) * nq + q) * IMG, IMG, &bars[B_OP_FULL + st],
                             policy_evict_last());
                }
                if (!ok) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_f16_f32(BM, BN);
            const uint32_t op0 = smem_u32(smem + OFF_OP);
            for (int q = 0; q < nq && !abort_flag.get(); ++q) {
                const int slot = q & 1, st = q % NOP;
                if (!tc::wait_or_abort(&bars[B_ACC_EMPTY + slot], ((q >> 1) & 1) ^ 1, abort_flag, p.status)) break;
                if (!tc::wait_or_abort(&bars[B_OP_FULL + st], (q / NOP) & 1, abort_flag, p.status)) break;
                tc::fence_after();
                const uint32_t a0 = op0 + st * OPB, b0 = a0 + A_BYTES;
                for (int b = 0; b < 4; ++b)
                    for (int t = 0; t < 2; ++t)
                        tc::mma_f16(tmem + slot * 256 + 64 * b, tc::smem_desc(a0 + 512 * b + 256 * t, 128, KC * 16),
                                    tc::smem_desc(b0 + 512 * b + 256 * t, 128, KC * 16), idesc, t);
                tc::commit(&bars[B_OP_EMPTY + st]);
                tc::commit(&bars[B_ACC_FULL + slot]);
            }
        }
    } else if (warp < 10) {
        // --------------------------------------------------------- converters
        // Thread (row r, half `part` of the chunk): blocks 2*part, 2*part + 1
        // of the chunk, 32 elements each, as four 8-element core-matrix rows.
        // The thread loads the 16-byte-aligned window that holds its two
        // blocks with 128-bit loads: the raw rows are a multiple of 16 bytes
        // and an odd multiple of 16 modulo 128, so the 8 rows of a load phase
        // fall in 8 different bank groups. Its byte offset in the window
        // depends only on (h, part), so it is uniform across the warp.
        constexpr int NW = WF == CQ_Q8_0 ? 20 : WF == CQ_Q4_1 ? 16 : 12;
        const int tid = threadIdx.x - 64;               // 0..255
        const int r = tid & (BM - 1), part = tid >> 7;
        for (int q = 0; q < nq; ++q) {
            const int s = q >> 1, h = q & 1, st = q % NOP, rs = s % NRAW;
            if (abort_flag.get()) break;
            if (!tc::wait_or_abort(&bars[B_OP_EMPTY + st], ((q / NOP) & 1) ^ 1, abort_flag, p.status)) break;
            if (!tc::wait_or_abort(&bars[B_RAW_FULL + rs], (s / NRAW) & 1, abort_flag, p.status)) break;
            uint8_t* stg = smem + OFF_OP + st * OPB;
            float* wsd = reinterpret_cast<float*>(stg + A_BYTES + IMG);
            const int off = (4 * h + 2 * part) * F::BB;         // the two blocks' byte offset in the row
            const uint8_t* win = smem + OFF_RAW + rs * RSB + r * PITCH + (off & ~15);
            uint32_t w[NW];
#pragma unroll
            for (int i = 0; i < NW / 4; ++i) {
                const uint4 v = *reinterpret_cast<const uint4*>(win + 16 * i);
                w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
            }
            uint8_t* dst = stg + tc::tile_off(r, 64 * part, KC);
            float d[2], mn[2];
            switch (off & 15) {
            case 0: convert_pair<WF, 0>(w, dst, d, mn); break;
            case 4: convert_pair<WF, 4>(w, dst, d, mn); break;
            case 8: convert_pair<WF, 8>(w, dst, d, mn); break;
            default: convert_pair<WF, 12>(w, dst, d, mn); break;
            }
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
                wsd[(2 * part + bb) * BM + r] = d[bb];
                if constexpr (Q41) wsd[4 * BM + (2 * part + bb) * BM + r] = mn[bb];
            }
            if constexpr (!PRE) {
                // The chunk's activation image: thread (block cb = tid / 64, token
                // tk = tid % 64) -- cb is warp-uniform, so the block's offset in the
                // token's 16-byte-aligned window is too. Rows of 8 blocks are 272
                // (Q8_0) or 288 (Q8_1) bytes apart.
                const int cb = tid >> 6, tk = tid & 63;
                const int aoff = (4 * h + cb) * F::ABB;
                const uint8_t* awin = smem + OFF_RAW + rs * RSB + RAWB + tk * (8 * F::ABB) + (aoff & ~15);
                uint32_t aw[12];
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    const uint4 v = *reinterpret_cast<const uint4*>(awin + 16 * i);
                    aw[4 * i] = v.x; aw[4 * i + 1] = v.y; aw[4 * i + 2] = v.z; aw[4 * i + 3] = v.w;
                }
                uint8_t* bdst = stg + A_BYTES + tc::tile_off(tk, 32 * cb, KC);
                float* dxp = reinterpret_cast<float*>(stg + A_BYTES + B_BYTES) + cb * BN + tk;
                float* sxp = dxp + 4 * BN;
                switch (aoff & 15) {
                case 0: convert_act<WF, 0>(aw, bdst, dxp, sxp); break;
                case 2: if constexpr (!Q41) convert_act<WF, 2>(aw, bdst, dxp, sxp); break;
                case 4: convert_act<WF, 4>(aw, bdst, dxp, sxp); break;
                case 6: if constexpr (!Q41) convert_act<WF, 6>(aw, bdst, dxp, sxp); break;
                case 8: convert_act<WF, 8>(aw, bdst, dxp, sxp); break;
                case 10: if constexpr (!Q41) convert_act<WF, 10>(aw, bdst, dxp, sxp); break;
                case 12: convert_act<WF, 12>(aw, bdst, dxp, sxp); break;
                default: if constexpr (!Q41) convert_act<WF, 14>(aw, bdst, dxp, sxp); break;
                }
            }
            fence_proxy_async_smem();
            tc::mbar_arrive(&bars[B_OP_FULL + st]);
            if (h == 1) tc::mbar_arrive(&bars[B_RAW_EMPTY + rs]);
        }
    } else {
        // ----------------------------------------------------------- epilogue
        // Warp w drains tensor-memory lanes 32*(w%4).. (weight rows) for the 16
        // token columns of its column group, in 16x256b fragments: thread t holds
        // rows 16h + t/4 + 8e (h, e in {0, 1}) and tokens 8j + 2(t%4) + u (j, u in
        // {0, 1}) of that slice, so it reads only its own two token pairs' scales
        // (a warp-uniform scale vector would cost one shared-memory wavefront per
        // quarter warp).
        const int quarter = warp & 3;
        const int c0 = ((warp - 10) >> 2) * EPI_COLS;   // first token column of this warp
        const int g = lane >> 2, tq = lane & 3;
        uint64_t y[8], c[8];                            // [h][e][j], token pair u = 0, 1
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = 0;
        bool ok = true;
        for (int q = 0; q < nq; ++q) {
            const int slot = q & 1, st = q % NOP;
            const bool got = mbar_wait_bounded(&bars[B_ACC_FULL + slot], (q >> 1) & 1, WAIT_LIMIT_NS) &&
                             mbar_wait_bounded(&bars[B_OP_FULL + st], (q / NOP) & 1, WAIT_LIMIT_NS);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) { abort_flag.set(1); atomicOr(p.status, CQ_DEV_WAIT_TIMEOUT); }
                ok = false;
                break;
            }
            tc::fence_after();
            const uint8_t* stg = smem + OFF_OP + st * OPB;
            const float* dxs = reinterpret_cast<const float*>(stg + A_BYTES + B_BYTES);
            const float* wsd = reinterpret_cast<const float*>(stg + A_BYTES + IMG);
#pragma unroll
            for (int i = 0; i < 8; ++i) c[i] = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                uint32_t is[2][8];
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    tc::ld16x256b_x2(tmem + (static_cast<uint32_t>(quarter * 32 + 16 * h) << 16) + slot * 256 + 64 * b +
                                         c0,
                                     is[h]);
                float dw[2][2];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int e = 0; e < 2; ++e) dw[h][e] = wsd[b * BM + quarter * 32 + 16 * h + 8 * e + g];
                float2 dx[2];
#pragma unroll
                for (int jj = 0; jj < 2; ++jj)
                    dx[jj] = *reinterpret_cast<const float2*>(dxs + b * BN + c0 + 8 * jj + 2 * tq);
                tc::wait_ld();
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            uint64_t& cc = c[4 * h + 2 * e + jj];
                            // c = fma(d_w * d_x, isum, c), two tokens per instruction
                            cc = tc::fma2(tc::mul2(tc::pk(dw[h][e], dw[h][e]), tc::pk(dx[jj].x, dx[jj].y)),
                                          tc::pk(__uint_as_float(is[h][4 * jj + 2 * e]),
                                                 __uint_as_float(is[h][4 * jj + 2 * e + 1])),
                                          cc);
                        }
                if constexpr (Q41) {
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const float2 sx = *reinterpret_cast<const float2*>(dxs + 4 * BN + b * BN + c0 + 8 * jj + 2 * tq);
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const float mw = wsd[4 * BM + b * BM + quarter * 32 + 16 * h + 8 * e + g];
                                uint64_t& cc = c[4 * h + 2 * e + jj];
                                cc = tc::fma2(tc::pk(mw, mw), tc::pk(sx.x, sx.y), cc);
                            }
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = tc::add2(y[i], c[i]);
            tc::fence_before();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&bars[B_ACC_EMPTY + slot]);
                tc::mbar_arrive(&bars[B_OP_EMPTY + st]);
            }
        }
        if (ok) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int row = n0 + quarter * 32 + 16 * h + 8 * e + g;
                    if (row >= p.N) continue;
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        float v[2];
                        tc::upk(y[4 * h + 2 * e + jj], v[0], v[1]);
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int m = m0 + c0 + 8 * jj + 2 * tq + u;
                            if (m < p.M) p.y[static_cast<int64_t>(m) * p.N + row] = v[u];
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
        for (int i = 0; i < 2; ++i) (void)mbar_wait_bounded(&bars[B_ACC_FULL + i], 0, WAIT_LIMIT_NS / 8);
    }
    __syncthreads();
    tc::fence_after();
    if (warp == 1) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// The workspace images: one CTA per (chunk q, token tile), thread (token t,
// block b): the block's 32 quants as fp16 into the K-major B tile, and its
// d_x (and s_x for Q8_1). Tokens past M become zeros.
template <int WF>
__global__ void __launch_bounds__(256) gemm32_tc_prep_kernel(const Tc32Params p, uint8_t* img) {
    pdl_trigger();
    pdl_wait();
    using F = MF<WF>;
    constexpr int IMG = img_bytes(WF == CQ_Q4_1);
    const int q = blockIdx.x, tile = blockIdx.y;
    const int t = threadIdx.x >> 2, b = threadIdx.x & 3;
    const int m = tile * BN + t;
    uint8_t* dst = img + (static_cast<int64_t>(tile) * p.nchunk + q) * IMG;
    float* dxs = reinterpret_cast<float*>(dst + B_BYTES);
    float d = 0.0f, s = 0.0f;
    uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (m < p.M) {
        const uint8_t* blk = p.xq + (static_cast<int64_t>(m) * p.nb + 4 * q + b) * F::ABB;
        const uint16_t* hw = reinterpret_cast<const uint16_t*>(blk);
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = __byte_perm(hw[F::AQO / 2 + 2 * j], hw[F::AQO / 2 + 2 * j + 1], 0x5410);
        d = h2f(hw[0]);
        s = WF == CQ_Q4_1 ? h2f(hw[1]) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t o[4];
        tc::s8x4_half(w[2 * i], o[0], o[1]);
        tc::s8x4_half(w[2 * i + 1], o[2], o[3]);
        *reinterpret_cast<uint4*>(dst + tc::tile_off(t, 32 * b + 8 * i, KC)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    dxs[b * BN + t] = d;
    if constexpr (WF == CQ_Q4_1) dxs[4 * BN + b * BN + t] = s;
}

template <int WF, bool PRE>
cudaError_t launch_mode(const DeviceInfo& dev, const CUtensorMap& wmap, const CUtensorMap& amap, const Tc32Params& p,
                        unsigned tok_tiles, unsigned row_tiles, cudaStream_t s) {
    using F = MF<WF>;
    constexpr int SMEM = smem_bytes(PRE, F::BB, F::ABB);
    if (SMEM > dev.smem_optin) return cudaErrorInvalidConfiguration;
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(gemm32_tc_kernel<WF, PRE>), SMEM);
    if (e != cudaSuccess) return e;
    if constexpr (PRE) {
        e = launch_kernel(gemm32_tc_prep_kernel<WF>, dim3(static_cast<unsigned>(p.nchunk), tok_tiles), dim3(256), 0,
                          s, p, const_cast<uint8_t*>(p.img));
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(gemm32_tc_kernel<WF, PRE>, dim3(tok_tiles, row_tiles), dim3(THREADS), SMEM, s, wmap, amap,
                         p);
}

template <int WF>
cudaError_t launch_fmt(const DeviceInfo& dev, int64_t M, int64_t N, int64_t K, const void* W, const void* xq,
                       float* y, void* workspace, cudaStream_t s) {
    using F = MF<WF>;
    tc::EncodeTiledFn enc = tc::encode_tiled_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    const int nb = static_cast<int>(K / 32);
    const int64_t wrow = static_cast<int64_t>(nb) * F::BB, xrow = static_cast<int64_t>(nb) * F::ABB;
    // Raw weights [N rows][wrow / 2] and activations [M rows][xrow / 2] as 2-D
    // tensors of 2-byte elements; a box is one 8-block segment of 128 rows / 64
    // tokens; rows past N and tokens past M read as zero.
    CUtensorMap wmap, amap;
    const cuuint32_t estr[2] = {1, 1};
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(wrow / 2), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(wrow)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(mf::stage_pitch(F::BB) / 2), BM};
        if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(W), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(xrow / 2), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(xrow)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(8 * F::ABB / 2), BN};
        if (enc(&amap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(xq), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int64_t row_tiles = (N + BM - 1) / BM;
    if (row_tiles > 65535) return cudaErrorInvalidValue;      // grid y limit (N above 8.4 M rows)
    Tc32Params p{};
    p.xq = static_cast<const uint8_t*>(xq);
    p.img = static_cast<const uint8_t*>(workspace);
    p.y = y;
    p.status = dev.status;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.nb = nb;
    p.nchunk = nb / 4;
    const unsigned tok_tiles = static_cast<unsigned>((M + BN - 1) / BN);
    return workspace != nullptr
               ? launch_mode<WF, true>(dev, wmap, amap, p, tok_tiles, static_cast<unsigned>(row_tiles), s)
               : launch_mode<WF, false>(dev, wmap, amap, p, tok_tiles, static_cast<unsigned>(row_tiles), s);
}

}  // namespace

size_t gemm32_workspace_size(int w_fmt, int64_t M, int64_t K) {
    if ((w_fmt != CQ_Q4_0 && w_fmt != CQ_Q4_1 && w_fmt != CQ_Q8_0) || M <= 0) return 0;
    return static_cast<size_t>((M + BN - 1) / BN) * static_cast<size_t>(K / KC) *
           static_cast<size_t>(img_bytes(w_fmt == CQ_Q4_1));
}

cudaError_t launch_gemm_tc32(const DeviceInfo& dev, int w_fmt, int64_t M, int64_t N, int64_t K, const void* W,
                             const void* xq, float* y, void* workspace, cudaStream_t s) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    switch (w_fmt) {
    case CQ_Q4_0: return launch_fmt<CQ_Q4_0>(dev, M, N, K, W, xq, y, workspace, s);
    case CQ_Q4_1: return launch_fmt<CQ_Q4_1>(dev, M, N, K, W, xq, y, workspace, s);
    case CQ_Q8_0: return launch_fmt<CQ_Q8_0>(dev, M, N, K, W, xq, y, workspace, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace cq
