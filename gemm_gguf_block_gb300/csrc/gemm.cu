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
//   A[n][k] = sc_j(n) * q4(n, k)   in [0, 945]    (weights, MMA M = 128 rows)
//   B[m][k] = q8(m, k)             in [-127, 127] (tokens, MMA N = 128)
// A superblock's isum_sc = sum_j sc_j * S_j reaches 30.7e6 > 2^24, too much
// for one exact fp32 accumulator, but with the correction
//   C = 8 * sum_j sc_j * B_j   (B_j = bsum_2j + bsum_2j+1, the 32-element sums)
// the accumulator starts at -C (one K = 16 MMA) and then takes the 256
// products: after any subset S of them it holds
//   sum_{k in S} sc (q4 - 8) q8 - sum_{k not in S} 8 sc q8,
// whose magnitude is at most 256 * 504 * 127 = 16386048 < 2^24 whatever the
// order of the additions -- every value the accumulator passes through is an
// exact integer -- and it ends at X = isum_sc - C. A second copy of -C and
// the min term I = sum_j m_j * B_j come from two more K = 16 MMAs:
// A_C = [-8 sc_0..-8 sc_7 | the same], A_I = [m_0..m_7 | the same], B_min =
// [64 h_0..64 h_7 | l_0..l_7] with B_j = 64 h_j + l_j, all exact in fp16
// (|C| <= 8 * 63 * 8 * 4064 < 2^24). The epilogue then applies, per (row,
// token, superblock), exactly the fixed fp32 order of include/cq.h --
// RN(X - (-C)) is (float)isum_sc; then t = fma(d, S, -(dmin * I)) and
// y = fma(d_x, t, y) -- so every row equals the cq_gemv row bit for bit.
//
// Tensor memory: X in two alternating 128-column buffers, -C and I in 128
// columns each. The MMAs of superblock s+1 fill the other X buffer while the
// epilogue drains superblock s; only its two small -C / I MMAs wait for the
// epilogue to have read the previous ones.
//
// Operands move through four stages of a quarter superblock each (K = 64,
// one 64-element Q4_K group): 16 KB of A (weights) and 16 KB of B
// (activations), so the MMA warp keeps up to three quarters queued while a
// stage is refilled.
//
// Warp roles (896 threads): warp 0 TMA producer of raw Q4_K tiles (2-D tensor
// map, 128 rows x 144 bytes per superblock); warp 1 allocates tensor memory
// and one lane issues the MMAs; warp 2 bulk-copies, with a workspace, the
// pre-converted B operands and, in a CTA pair, this CTA's converted slice of
// each stage (weights with a workspace, activations without) into the peer's
// stage (a warp of its own, so that the raw weight boxes run ahead of the
// operand stages); warp 3 writes each superblock's min slot
// (A_C, A_I; with a workspace also B_min by bulk copy) and scale slot (the
// rows' d, dmin; with a workspace also d_x); warps 4-11 convert raw weights
// into fp16 A tiles (K-major, no swizzle); warps 12-27 are the epilogue
// (tensor-memory lanes 32*(warp%4), 32 token columns each, y in registers)
// and, without a workspace, also convert the Q8_K activations into the B
// tiles (K-major, 128-byte swizzle), B_min and d_x. Every wait is bounded;
// a timeout flags CQ_DEV_WAIT_TIMEOUT and the CTA winds down.
#include <algorithm>

#include <cuda_fp16.h>

#include "cq_device.cuh"
#include "cq_internal.h"
#include "tc.cuh"

namespace cq {
namespace {

constexpr int BM = 128;          // weight rows per tile (MMA M, TMEM lanes)
constexpr int BN = 128;          // tokens per tile (MMA N)
constexpr int KH = 128;          // K per thread of the workspace prep kernel (half a superblock)
constexpr int KQ = 64;           // K per operand stage (a quarter superblock: one 64-element Q4_K group)
constexpr int NSTAGE = 4;        // operand stages
constexpr int NMIN = 2;          // min slots (A_C, A_I, B_min of one superblock)
constexpr int NDX = 4;           // scale slots (the tokens' d_x and the rows' d, dmin of one superblock)
constexpr int RAW_BYTES = BM * 144;
constexpr int A_BYTES = BM * KQ * 2;        // 16 KB
constexpr int B_BYTES = BN * KQ * 2;        // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int AC_BYTES = BM * 16 * 2;       // 4 KB
constexpr int AI_BYTES = BM * 16 * 2;       // 4 KB
constexpr int BMIN_BYTES = BN * 16 * 2;     // 4 KB
constexpr int DX_BYTES = BN * 4;            // 512 B
constexpr int SCL_BYTES = DX_BYTES + BM * 4;   // a scale slot: d_x [BN] fp32, then (d, dmin) [BM] as fp16 pairs
constexpr int MIN_BYTES = AC_BYTES + AI_BYTES + BMIN_BYTES;   // 12288
constexpr int NCONV = 256;                  // converter threads
constexpr int CONV_WARPS = NCONV / 32;
constexpr int EPI_WARPS = 16;
constexpr int COLS = BN / (EPI_WARPS / 4);  // 32 token columns per epilogue thread
constexpr int SLOT_WARP = 3;                // writer of the min and scale slots
constexpr int CONV_WARP0 = 4;               // first converter warp
constexpr int EPI_WARP0 = CONV_WARP0 + 8;   // first epilogue warp
constexpr int THREADS = (EPI_WARP0 + EPI_WARPS) * 32;
constexpr uint32_t TMEM_COLS = 512;         // X0 | X1 | C | I, 128 columns each
constexpr uint32_t COL_C = 256, COL_I = 384;

constexpr int XS_BYTES = BN * 256;          // the next superblock's Q8_K quants of the tile's tokens
// Shared-memory layout (offsets from the 1024-aligned dynamic base). Without
// a workspace the raw weight ring is one stage shorter, which makes room for
// the activation staging area XS.
constexpr int OFF_BAR = 0;                   // 35 barriers
constexpr int OFF_TMEM = 512;                // tensor-memory base address
constexpr int OFF_FLAG = 520;                // abort flag
constexpr int OFF_RAW = 1024;
template <bool PRE>
struct Layout {
    static constexpr int NRAW = PRE ? 3 : 2;   // raw weight superblock stages
    static constexpr int OFF_STAGE = OFF_RAW + NRAW * RAW_BYTES;   // 1024-aligned (swizzled B tiles)
    static constexpr int OFF_MIN = OFF_STAGE + NSTAGE * STAGE_BYTES;
    static constexpr int OFF_DX = OFF_MIN + NMIN * MIN_BYTES;
    static constexpr int OFF_XS = OFF_DX + NDX * SCL_BYTES;
    static constexpr int SMEM_BYTES = OFF_XS + (PRE ? 0 : XS_BYTES) + 1024;   // + alignment slack of the base
};
static_assert(Layout<true>::OFF_STAGE % 1024 == 0 && Layout<false>::OFF_STAGE % 1024 == 0, "B tile alignment");

enum {
    B_RAW_FULL = 0, B_RAW_EMPTY = 3, B_OP_FULL = 6, B_OP_EMPTY = 10, B_MIN_FULL = 14, B_MIN_EMPTY = 16,
    B_ACC_FULL = 18, B_X_EMPTY = 20, B_CI_EMPTY = 22, B_DX_FULL = 23, B_DX_EMPTY = 27, B_SLICE = 31, N_BARS = 35
};
static_assert(N_BARS * 8 <= OFF_TMEM, "barriers overlap the tensor-memory address");

struct GemmParams {
    const uint8_t* W;
    const uint8_t* xq;
    float* y;
    int* status;
    int M, N, ns;        // tokens, rows, superblocks per row
    int64_t wrow;        // bytes per weight row
    int64_t xrow;        // bytes per activation row
    const uint8_t* bimg; // pre-converted activation operands: [token tile][superblock] images of IMG_BYTES
};

// One (token tile, superblock) image of the pre-converted activations, laid
// out as the B parts of the four operand stages (quarters 0..3), then the
// B_min operand (the end of a min slot) and the tokens' d_x (a d_x slot).
constexpr int IMG_BYTES = 4 * B_BYTES + BMIN_BYTES + DX_BYTES;   // 70144

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// K order inside every 4-element group of both operand tiles: elements
// (0, 2, 1, 3). The contraction sums over K, so any order shared by A and B
// gives the same integers; this one lets both converters take bytes 0 and 2
// (then 1 and 3) of a word into one half2 without byte permutes.
//
// Four nibble pairs (one byte each of w; low nibble = element i of the low
// sub-block, high nibble = element i of the high one) -> lo = (q0, q2) * sl,
// (q1, q3) * sl and hi = the same of the high nibbles times sh, each exact:
// (1024 + q) * sl - 1024 sl for a low nibble, and (1024 + 16 q) * (sh / 16) -
// 64 sh for a high nibble masked in place, each one fused multiply-add whose
// exact result is representable.
__device__ __forceinline__ void nibbles_to_half(uint32_t w, __half2 sl, __half2 bl, __half2 sh16, __half2 bh,
                                                uint32_t (&lo)[2], uint32_t (&hi)[2]) {
    const uint32_t w8 = w >> 8;                          // bytes 1, 3 into the half positions
    lo[0] = h2_bits(__hfma2(bits_h2((w & 0x000F000Fu) | 0x64006400u), sl, bl));
    lo[1] = h2_bits(__hfma2(bits_h2((w8 & 0x000F000Fu) | 0x64006400u), sl, bl));
    hi[0] = h2_bits(__hfma2(bits_h2((w & 0x00F000F0u) | 0x64006400u), sh16, bh));
    hi[1] = h2_bits(__hfma2(bits_h2((w8 & 0x00F000F0u) | 0x64006400u), sh16, bh));
}

// Four signed bytes (elements 0..3) -> two half2 in the (0, 2, 1, 3) K order:
// (b0, b2) and (b1, b3), each exact (see tc::s8x4_half).
__device__ __forceinline__ void s8x4_half_0213(uint32_t w, uint32_t& o0, uint32_t& o1) {
    const __half2 k1152 = bits_h2(0x64806480u);
    const uint32_t u = w ^ 0x80808080u;
    o0 = h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, 0x4240)), k1152));
    o1 = h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, 0x4341)), k1152));
}

// The sixteen 6-bit values of a Q4_K scale block (words s0, s1, s2 of its
// twelve bytes), one per byte: sc[0] = sc_0..3, sc[1] = sc_4..7, mn[0] =
// m_0..3, mn[1] = m_4..7. Bytes 0-3 hold sc_j and m_j in their low six bits
// and the top two bits of sc_j+4, m_j+4 in bits 6-7; bytes 8-11 hold the low
// nibbles of sc_j+4 (low) and m_j+4 (high).
__device__ __forceinline__ void q4k_scales(uint32_t s0, uint32_t s1, uint32_t s2, uint32_t (&sc)[2],
                                           uint32_t (&mn)[2]) {
    sc[0] = s0 & 0x3F3F3F3Fu;
    mn[0] = s1 & 0x3F3F3F3Fu;
    sc[1] = (s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u);
    mn[1] = ((s2 >> 4) & 0x0F0F0F0Fu) | ((s1 >> 2) & 0x30303030u);
}

// Bytes (selected by the byte_perm selector sel) of w under a 0x64 high byte:
// half2 (1024 + v0, 1024 + v1), exact for bytes below 1024.
__device__ __forceinline__ __half2 bytes_1024(uint32_t w, uint32_t sel) {
    return bits_h2(__byte_perm(w, 0x64646464u, sel));
}

// B_min entries of one token: bsum pair word v (bsum_2j, bsum_2j+1) -> B_j =
// 64 h + l with h = floor(B_j / 64), both parts exact in fp16.
__device__ __forceinline__ void bmin_entry(uint32_t v, __half& hpart, __half& lpart) {
    const int pr = static_cast<int>(static_cast<int16_t>(v & 0xffffu)) + static_cast<int>(static_cast<int16_t>(v >> 16));
    const int hq = pr >> 6;                                  // floor division by 64
    hpart = __int2half_rn(64 * hq);
    lpart = __int2half_rn(pr - 64 * hq);
}

// A converter warp's bounded wait, decided for the whole warp (its lanes then
// leave a loop together, so the warp-wide arrivals below cannot hang).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, SmemFlag flag, int* status) {
    return __all_sync(0xffffffffu, tc::wait_or_abort_sleep(bar, parity, flag, status));
}
// One arrival for the warp, after every lane's prior writes (and, when they
// feed the tensor cores, its proxy fence).
__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(bar);
}

// PRE: the activations come pre-converted (cq_gemm_ws): warp 2 bulk-copies
// each stage's B operand, warp 3 each min slot's B_min and each scale slot's
// d_x. Without it the epilogue warps convert the Q8_K activations of
// superblock s+1 (between draining superblocks s-1 and s). Either way the
// converters handle only weights.
//
// CS: CTAs per cluster (1 or 2). A pair shares one conversion, and warp 2
// bulk-copies each CTA's converted slice of a stage into the peer's stage
// (completing on the peer's operand barrier); the MMAs of both CTAs release a
// stage together (multicast commits, two arrivals).
//   with a workspace (SHARE_A): the pair holds token tiles 2i, 2i+1 of the
//     same 128 weight rows; each CTA converts weight rows 64*rank .. +63 of
//     every A quarter;
//   without one (SHARE_B): the pair holds weight tiles 2j, 2j+1 of the same
//     128 tokens; each CTA's epilogue warps convert tokens 64*rank .. +63 of
//     every B quarter.
//
// SPLIT (no workspace, single CTAs, at most 96 tokens): the short-tile
// epilogue described below.
template <bool PRE, int CS, bool SPLIT>
__global__ void __launch_bounds__(THREADS, 1) gemm_q4k_kernel(const __grid_constant__ CUtensorMap wmap,
                                                              const GemmParams p) {
    using L = Layout<PRE>;
    constexpr bool SHARE_A = CS > 1 && PRE, SHARE_B = CS > 1 && !PRE;
    constexpr int RPC = SHARE_A ? BM / CS : BM;     // weight rows this CTA converts
    constexpr int TPC = SHARE_B ? BN / CS : BN;     // tokens whose B quarters this CTA converts
    // the slice of a stage copied to the peer: contiguous 8-row groups of the A tile, or 128-byte token rows of B
    constexpr int SLICE_BYTES = SHARE_A ? RPC * KQ * 2 : TPC * 128;
    constexpr int NRAW = L::NRAW, OFF_STAGE = L::OFF_STAGE, OFF_MIN = L::OFF_MIN, OFF_DX = L::OFF_DX;
    pdl_trigger();
    pdl_wait();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);
    const SmemFlag abort_flag{smem_u32(smem + OFF_FLAG)};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BM, m0 = blockIdx.y * BN;
    const int ns = p.ns;

    // A short last token tile without a workspace (at most 96 tokens, a whole
    // column group of the drain idle): the epilogue warps of the idle column
    // groups write the activation operands, the others only drain.
    const int t_valid = min(BN, p.M - m0);
    const int ngroups = (t_valid + COLS - 1) / COLS;
    const bool split = SPLIT && ngroups < EPI_WARPS / 4;
    const int n_drain = split ? 4 * ngroups : EPI_WARPS;           // drain warps
    const int n_act = split ? EPI_WARPS - n_drain : EPI_WARPS;      // activation-writing warps
    if (threadIdx.x == 0) {
        for (int i = 0; i < NRAW; ++i) {
            mbar_init(&bars[B_RAW_FULL + i], 1);
            mbar_init(&bars[B_RAW_EMPTY + i], CONV_WARPS + 1);              // + the slot writer
        }
        for (int i = 0; i < NSTAGE; ++i) {
            // warp 2, plus the converters of whatever operand is not copied through it
            mbar_init(&bars[B_OP_FULL + i], 1 + (SHARE_B ? CONV_WARPS : (PRE ? 0 : n_act)));
            mbar_init(&bars[B_OP_EMPTY + i], CS);                         // the MMA commits of the cluster's CTAs
            mbar_init(&bars[B_SLICE + i], SHARE_B ? n_act : CONV_WARPS);  // this CTA's slice converted
        }
        for (int i = 0; i < NMIN; ++i) {
            mbar_init(&bars[B_MIN_FULL + i], PRE ? 1 : 1 + n_act);          // the slot writer (+ B_min writers)
            mbar_init(&bars[B_MIN_EMPTY + i], 1);                      // the MMA commit
        }
        for (int i = 0; i < NDX; ++i) {
            mbar_init(&bars[B_DX_FULL + i], PRE ? 1 : 1 + (split ? n_act : BN / 32));   // the slot writer (+ d_x writers)
            mbar_init(&bars[B_DX_EMPTY + i], n_drain);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[B_ACC_FULL + i], 1);
            mbar_init(&bars[B_X_EMPTY + i], n_drain);
        }
        mbar_init(&bars[B_CI_EMPTY], n_drain);
        abort_flag.set(0);
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_holder, TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    if constexpr (CS > 1) tc::cluster_sync();   // the peer's barriers exist before anything reaches them
    tc::fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            for (int s = 0; s < ns && !abort_flag.get(); ++s) {
                const int r = s % NRAW;
                if (!tc::wait_or_abort_sleep(&bars[B_RAW_EMPTY + r], ((s / NRAW) & 1) ^ 1, abort_flag, p.status)) break;
                mbar_arrive_expect_tx(&bars[B_RAW_FULL + r], RAW_BYTES);
                tc::tma_load_2d(smem + OFF_RAW + r * RAW_BYTES, &wmap, 144 * s, n0, &bars[B_RAW_FULL + r]);
            }
        }
    } else if (warp == SLOT_WARP) {
        // ----------------------------------------------- min and scale slots
        // Per superblock s, lane l takes weight rows l + 32i of the raw stage:
        // their A_C rows [-8 sc_0 .. -8 sc_7] twice and A_I rows [m_0 .. m_7]
        // twice (the min slot), and their (d, dmin) words (the scale slot).
        // With a workspace, lane 0 also bulk-copies B_min and d_x into the
        // same slots.
        const uint64_t pol = policy_evict_first();
        auto slots = [&](int s) -> bool {
            const int rs = s % NRAW, ms = s % NMIN, ds = s % NDX;
            const uint8_t* img = PRE ? p.bimg + (static_cast<int64_t>(blockIdx.y) * ns + s) * IMG_BYTES : nullptr;
            if (!warp_wait(&bars[B_RAW_FULL + rs], (s / NRAW) & 1, abort_flag, p.status)) return false;
            uint4 hdr[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                hdr[i] = *reinterpret_cast<const uint4*>(smem + OFF_RAW + rs * RAW_BYTES + (lane + 32 * i) * 144);
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[B_RAW_EMPTY + rs]);
            if (!warp_wait(&bars[B_MIN_EMPTY + ms], ((s / NMIN) & 1) ^ 1, abort_flag, p.status)) return false;
            uint8_t* slot = smem + OFF_MIN + ms * MIN_BYTES;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = lane + 32 * i;
                uint32_t sc[2], mn[2];
                q4k_scales(hdr[i].y, hdr[i].z, hdr[i].w, sc, mn);
                // -8 sc = (1024 + sc) * -8 + 8192 and m = (1024 + m) - 1024, both exact
                uint32_t cw[4], iw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t sel = (j & 1) ? 0x4342u : 0x4140u;
                    cw[j] = h2_bits(__hfma2(bytes_1024(sc[j >> 1], sel), bits_h2(0xC800C800u), bits_h2(0x70007000u)));
                    iw[j] = h2_bits(__hsub2(bytes_1024(mn[j >> 1], sel), bits_h2(0x64006400u)));
                }
                const uint4 cv = make_uint4(cw[0], cw[1], cw[2], cw[3]), iv = make_uint4(iw[0], iw[1], iw[2], iw[3]);
                *reinterpret_cast<uint4*>(slot + tc::tile_off(r, 0, 16)) = cv;
                *reinterpret_cast<uint4*>(slot + tc::tile_off(r, 8, 16)) = cv;
                *reinterpret_cast<uint4*>(slot + AC_BYTES + tc::tile_off(r, 0, 16)) = iv;
                *reinterpret_cast<uint4*>(slot + AC_BYTES + tc::tile_off(r, 8, 16)) = iv;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (PRE) {
                    mbar_arrive_expect_tx(&bars[B_MIN_FULL + ms], BMIN_BYTES);
                    bulk_g2s(slot + AC_BYTES + AI_BYTES, img + 4 * B_BYTES, BMIN_BYTES, &bars[B_MIN_FULL + ms], pol);
                } else {
                    tc::mbar_arrive(&bars[B_MIN_FULL + ms]);
                }
            }
            if (!warp_wait(&bars[B_DX_EMPTY + ds], ((s / NDX) & 1) ^ 1, abort_flag, p.status)) return false;
            uint8_t* scl = smem + OFF_DX + ds * SCL_BYTES;
#pragma unroll
            for (int i = 0; i < 4; ++i) reinterpret_cast<uint32_t*>(scl + DX_BYTES)[lane + 32 * i] = hdr[i].x;
            __syncwarp();
            if (lane == 0) {
                if (PRE) {
                    mbar_arrive_expect_tx(&bars[B_DX_FULL + ds], DX_BYTES);
                    bulk_g2s(scl, img + 4 * B_BYTES + BMIN_BYTES, DX_BYTES, &bars[B_DX_FULL + ds], pol);
                } else {
                    tc::mbar_arrive(&bars[B_DX_FULL + ds]);
                }
            }
            return true;
        };
        for (int s = 0; s < ns; ++s)
            if (!slots(s)) break;
    } else if (warp == 2) {
        // ------------------------------------------------ operand copies
        // Per quarter, once the stage is free in every CTA of the cluster:
        // with a workspace, the pre-converted B operand (bulk copy); with a
        // cluster, this CTA's converted slice (of A, or of B) into the peer's
        // stage. Its arrival on the stage's barrier certifies the local slice
        // and expects the peer's.
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const uint32_t peer = CS > 1 ? (tc::cluster_rank() ^ 1u) : 0u;
            const uint32_t slice_off = CS > 1 ? (SHARE_B ? A_BYTES : 0u) + (peer ^ 1u) * SLICE_BYTES : 0u;
            for (int s = 0; s < ns && !abort_flag.get(); ++s) {
                const uint8_t* img = PRE ? p.bimg + (static_cast<int64_t>(blockIdx.y) * ns + s) * IMG_BYTES : nullptr;
                bool got = true;
                for (int g = 0; g < 4 && got; ++g) {
                    const int q = 4 * s + g, st = q % NSTAGE;
                    uint64_t* full = &bars[B_OP_FULL + st];
                    uint8_t* stg = smem + OFF_STAGE + st * STAGE_BYTES;
                    got = tc::wait_or_abort_sleep(&bars[B_OP_EMPTY + st], ((q / NSTAGE) & 1) ^ 1, abort_flag, p.status);
                    if (!got) break;
                    if (PRE) {
                        tc::mbar_expect_tx(full, B_BYTES);
                        bulk_g2s(stg + A_BYTES, img + g * B_BYTES, B_BYTES, full, pol);
                    }
                    got = tc::wait_or_abort_sleep(&bars[B_SLICE + st], (q / NSTAGE) & 1, abort_flag, p.status);
                    if (!got) break;
                    if constexpr (CS > 1) {
                        tc::bulk_s2peer(tc::cluster_addr(smem_u32(stg + slice_off), peer), stg + slice_off, SLICE_BYTES,
                                        tc::cluster_addr(smem_u32(full), peer));
                        mbar_arrive_expect_tx(full, SLICE_BYTES);
                    } else {
                        tc::mbar_arrive(full);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_f16_f32(BM, BN);
            // Descriptors of stage 0 and min slot 0; others differ only in the
            // start-address field (bytes / 16), which no offset here overflows.
            // A tiles: no swizzle; B tiles: 128-byte swizzle (one 64-element
            // column block of BN rows).
            const uint64_t op_desc0 = tc::smem_desc(smem_u32(smem + OFF_STAGE), 128, KQ * 16);
            const uint64_t b_desc0 = tc::smem_desc_sw128(smem_u32(smem + OFF_STAGE + A_BYTES), 1024);
            const uint64_t min_desc0 = tc::smem_desc(smem_u32(smem + OFF_MIN), 128, 256);
            for (int s = 0; s < ns && !abort_flag.get(); ++s) {
                const int b = s & 1, ms = s % NMIN;
                if (!tc::wait_or_abort_sleep(&bars[B_X_EMPTY + b], ((s >> 1) & 1) ^ 1, abort_flag, p.status)) break;
                if (!tc::wait_or_abort_sleep(&bars[B_MIN_FULL + ms], (s / NMIN) & 1, abort_flag, p.status)) break;
                tc::fence_after();
                const uint32_t xcol = tmem + static_cast<uint32_t>(b * BN);
                const uint64_t acd = min_desc0 + static_cast<uint32_t>((ms * MIN_BYTES) >> 4);
                const uint64_t bmd = acd + ((AC_BYTES + AI_BYTES) >> 4);
                tc::mma_f16(xcol, acd, bmd, idesc, 0);                  // X = -C
                bool ok = true;
                for (int g = 0; g < 4; ++g) {
                    const int q = 4 * s + g, st = q % NSTAGE;
                    if (!tc::wait_or_abort_sleep(&bars[B_OP_FULL + st], (q / NSTAGE) & 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint64_t ad = op_desc0 + static_cast<uint32_t>((st * STAGE_BYTES) >> 4);
                    const uint64_t bd = b_desc0 + static_cast<uint32_t>((st * STAGE_BYTES) >> 4);
#pragma unroll
                    for (int t = 0; t < KQ / 16; ++t) tc::mma_f16(xcol, ad + 16 * t, bd + 2 * t, idesc, 1);
                    if constexpr (CS > 1)
                        tc::commit_multicast(&bars[B_OP_EMPTY + st], static_cast<uint16_t>((1u << CS) - 1u));
                    else
                        tc::commit(&bars[B_OP_EMPTY + st]);
                }
                if (!ok) break;
                if (!tc::wait_or_abort_sleep(&bars[B_CI_EMPTY], (s & 1) ^ 1, abort_flag, p.status)) break;
                tc::fence_after();
                tc::mma_f16(tmem + COL_C, acd, bmd, idesc, 0);          // -C
                tc::mma_f16(tmem + COL_I, acd + (AC_BYTES >> 4), bmd, idesc, 0);                  // I
                tc::commit(&bars[B_MIN_EMPTY + ms]);
                tc::commit(&bars[B_ACC_FULL + b]);
            }
        }
    } else if (warp < EPI_WARP0) {
        // --------------------------------------------------------- converters
        // Weights: this CTA's RPC rows. Thread (row r = RPC*rank + tid % RPC,
        // part = tid / RPC) converts, in each quarter stage (64-element group
        // g of the superblock), bytes PB*part .. +PB-1 of the group's 32 quant
        // bytes: those elements of sub-block 2g (low nibbles) and of sub-block
        // 2g + 1 (high nibbles). All four groups' words are read, and the raw
        // stage released, when the superblock starts. A quarter warp covers 8
        // consecutive rows, so its loads (row pitch 144 bytes) and its 16-byte
        // stores into the A tile (row pitch 16 bytes within a core matrix) hit
        // 8 distinct bank groups.
        constexpr int NPART = NCONV / RPC, PB = 32 / NPART, WPG = PB / 4;   // parts, bytes and words per part
        const int tid = threadIdx.x - 32 * CONV_WARP0;  // 0..255
        const int part = tid / RPC;
        const int r = RPC * static_cast<int>(SHARE_A ? tc::cluster_rank() : 0u) + tid % RPC;
        const int a_row = (r >> 3) * (KQ * 16) + (r & 7) * 16 + part * (WPG / 2) * 128;   // A tile row base
        uint32_t scw[2] = {0u, 0u}, mnw[2] = {0u, 0u};  // the row's scales (and mins, unused here), one per byte
        uint32_t qw[4 * WPG];                           // the thread's quant words, WPG per group
        for (int s = 0; s < ns; ++s) {
            const int rs = s % NRAW;
            if (__any_sync(0xffffffffu, abort_flag.get())) break;
            if (!warp_wait(&bars[B_RAW_FULL + rs], (s / NRAW) & 1, abort_flag, p.status)) break;
            {
                const uint8_t* raw = smem + OFF_RAW + rs * RAW_BYTES + r * 144;
                const uint4 hdr = *reinterpret_cast<const uint4*>(raw);
                q4k_scales(hdr.y, hdr.z, hdr.w, scw, mnw);
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    if constexpr (WPG == 4) {
                        const uint4 v = *reinterpret_cast<const uint4*>(raw + 16 + 32 * g + 16 * part);
                        qw[4 * g] = v.x; qw[4 * g + 1] = v.y; qw[4 * g + 2] = v.z; qw[4 * g + 3] = v.w;
                    } else {
                        const uint2 v = *reinterpret_cast<const uint2*>(raw + 16 + 32 * g + 8 * part);
                        qw[2 * g] = v.x; qw[2 * g + 1] = v.y;
                    }
                }
                // every read of the raw stage is done (the arrive orders them before the refill)
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bars[B_RAW_EMPTY + rs]);
            }
            bool ok = true;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int q = 4 * s + g, st = q % NSTAGE;
                if (!warp_wait(&bars[B_OP_EMPTY + st], ((q / NSTAGE) & 1) ^ 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                // A: weight row r, elements PB part .. of sub-blocks 2g (low nibbles, k = PB part + ..)
                // and 2g + 1 (high nibbles, k = 32 + PB part + ..), as sc * q; their scales are bytes
                // 2(g % 2) and 2(g % 2) + 1 of scw[g / 2]
                const __half2 k1024 = bits_h2(0x64006400u), km1024 = bits_h2(0xE400E400u);
                const uint32_t sw = scw[g >> 1];
                const __half2 slo = __hsub2(bytes_1024(sw, (g & 1) ? 0x4242u : 0x4040u), k1024);
                const __half2 shi16 =
                    __hmul2(__hsub2(bytes_1024(sw, (g & 1) ? 0x4343u : 0x4141u), k1024), bits_h2(0x2C002C00u));   // sc / 16
                const __half2 blo = __hmul2(slo, km1024);
                const __half2 bhi = __hmul2(shi16, km1024);                                                    // -64 sc
                uint8_t* arow = smem + OFF_STAGE + st * STAGE_BYTES + a_row;
#pragma unroll
                for (int c = 0; c < WPG / 2; ++c) {  // 8 elements (2 words) per core-matrix row
                    uint32_t l0[2], h0[2], l1[2], h1[2];
                    nibbles_to_half(qw[WPG * g + 2 * c], slo, blo, shi16, bhi, l0, h0);
                    nibbles_to_half(qw[WPG * g + 2 * c + 1], slo, blo, shi16, bhi, l1, h1);
                    *reinterpret_cast<uint4*>(arow + c * 128) = make_uint4(l0[0], l0[1], l1[0], l1[1]);
                    *reinterpret_cast<uint4*>(arow + 512 + c * 128) = make_uint4(h0[0], h0[1], h1[0], h1[1]);
                }
                fence_proxy_async_smem();   // for the local MMAs (and warp 2's copy to the peer)
                warp_arrive(&bars[(SHARE_B ? B_OP_FULL : B_SLICE) + st], lane);
            }
            if (!ok) break;
        }
    } else {
        // ----------------------------------------------------------- epilogue
        // Warp w drains tensor-memory lanes 32*(w%4).. (weight rows) for the 32
        // token columns of its column group, in 16x256b fragments: thread t holds
        // rows 16h + t/4 + 8e (h, e in {0, 1}) and tokens 8g + 2(t%4) + u (g in
        // 0..3, u in {0, 1}) of that slice, so it reads only its own token pairs'
        // d_x (a warp-uniform scale vector would cost a shared-memory wavefront per
        // quarter warp) and its rows' (d, dmin) from the scale slot.
        //
        // Without a workspace these warps also write the activation operands
        // of the next superblock: thread etid the B_min entries 2(etid%4), +1
        // of token etid/4, the first four warps the tokens' d_x, then per
        // quarter stage warp ew converts TPW tokens, tb + TPW*ew + 2i + l/16
        // for lane l (quant word l%16 of the quarter; in the swizzled B tile a
        // store instruction fills two whole 128-byte rows) -- all 128 tokens,
        // or this CTA's half of them in a pair. The quant words travel one
        // superblock ahead by asynchronous copies into the staging area XS
        // (each thread reads back only what it copied; a copy instruction
        // covers 64 contiguous bytes of each of two tokens), the bsums and d_x
        // in registers.
        //
        // In a short tile without a workspace (split), warps ew >= n_drain only
        // write the activation operands, all superblocks in turn as stages
        // free up: the B rows of the valid tokens this CTA converts (token
        // pair j = aw, aw + n_act, ..., lane l: token 2j + l/16, quant word
        // l%16), B_min and d_x of all valid tokens; the other warps only drain.
        constexpr int TPW = TPC / EPI_WARPS, NI = TPW / 2;   // tokens per warp, token pairs per warp
        const int quarter = warp & 3;
        const int ew = warp - EPI_WARP0, etid = threadIdx.x - 32 * EPI_WARP0;
        const int hi = lane >> 4, wq = lane & 15;
        if (split && ew >= n_drain) {
            const int aw = ew - n_drain;
            const int tlo = TPC * static_cast<int>(SHARE_B ? tc::cluster_rank() : 0u);   // first token converted here
            const int thi = min(tlo + TPC, t_valid);
            const int npairs = thi > tlo ? (thi - tlo + 1) / 2 : 0;
            uint32_t* xsb = reinterpret_cast<uint32_t*>(smem + L::OFF_XS) + wq;   // [token][64 words]
            auto afetch = [&](int s) {
                for (int j = aw; j < npairs; j += n_act) {
                    const int t = tlo + 2 * j + hi;
                    const uint32_t n = t < thi ? 4u : 0u;
                    const uint32_t* row = reinterpret_cast<const uint32_t*>(
                        p.xq + static_cast<int64_t>(m0 + (t < thi ? t : 0)) * p.xrow + 292 * s + 4) + wq;
#pragma unroll
                    for (int g = 0; g < 4; ++g) cp_async4(xsb + 64 * t + 16 * g, row + 16 * g, n);
                }
                cp_async_commit();
            };
            auto aput = [&](int s) -> bool {
                cp_async_wait_all();
                const int ms = s % NMIN, ds = s % NDX;
                if (!warp_wait(&bars[B_MIN_EMPTY + ms], ((s / NMIN) & 1) ^ 1, abort_flag, p.status)) return false;
                uint8_t* bm = smem + OFF_MIN + ms * MIN_BYTES + AC_BYTES + AI_BYTES;
                for (int it = 32 * aw + lane; it < 8 * t_valid; it += 32 * n_act) {   // (token, bsum pair word)
                    const int t = it >> 3, j = it & 7;
                    const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(
                                                 p.xq + static_cast<int64_t>(m0 + t) * p.xrow + 292 * s + 260) + j);
                    __half* bh = reinterpret_cast<__half*>(bm + tc::tile_off(t, 0, 16));
                    bmin_entry(v, bh[j], bh[64 + j]);
                }
                fence_proxy_async_smem();
                warp_arrive(&bars[B_MIN_FULL + ms], lane);
                if (!warp_wait(&bars[B_DX_EMPTY + ds], ((s / NDX) & 1) ^ 1, abort_flag, p.status)) return false;
                for (int t = 32 * aw + lane; t < t_valid; t += 32 * n_act)
                    reinterpret_cast<float*>(smem + OFF_DX + ds * SCL_BYTES)[t] =
                        __ldg(reinterpret_cast<const float*>(p.xq + static_cast<int64_t>(m0 + t) * p.xrow + 292 * s));
                warp_arrive(&bars[B_DX_FULL + ds], lane);
#pragma unroll
                for (int g2 = 0; g2 < 4; g2 += 2) {
#pragma unroll
                    for (int g = g2; g < g2 + 2; ++g) {
                        const int q = 4 * s + g, st = q % NSTAGE;
                        if (!warp_wait(&bars[B_OP_EMPTY + st], ((q / NSTAGE) & 1) ^ 1, abort_flag, p.status))
                            return false;
                        uint8_t* bstage = smem + OFF_STAGE + st * STAGE_BYTES + A_BYTES;
                        for (int j = aw; j < npairs; j += n_act) {
                            const int t = tlo + 2 * j + hi;
                            uint32_t o0, o1;
                            s8x4_half_0213(xsb[64 * t + 16 * g], o0, o1);
                            *reinterpret_cast<uint2*>(bstage + tc::tile_off_sw128(t, 4 * wq, BN)) = make_uint2(o0, o1);
                        }
                    }
                    fence_proxy_async_smem();   // for the local MMAs (and warp 2's copy to the peer)
                    __syncwarp();
                    if (lane == 0) {
                        constexpr int BAR = SHARE_B ? B_SLICE : B_OP_FULL;
                        tc::mbar_arrive(&bars[BAR + (4 * s + g2) % NSTAGE]);
                        tc::mbar_arrive(&bars[BAR + (4 * s + g2 + 1) % NSTAGE]);
                    }
                }
                return true;
            };
            afetch(0);
            for (int s = 0; s < ns; ++s) {
                if (!aput(s)) break;
                if (s + 1 < ns) afetch(s + 1);
            }
            cp_async_wait_all();   // no copy into the staging area outlives the loop
        } else {
        const int tb = TPC * static_cast<int>(SHARE_B ? tc::cluster_rank() : 0u) + TPW * ew + hi;   // token of pair 0
        uint32_t* xs = reinterpret_cast<uint32_t*>(smem + L::OFF_XS) + tb * 64 + wq;   // [token][64 words]
        uint32_t bsw[2] = {0u, 0u};
        float dxw = 0.0f;
        auto fetch_b = [&](int s) {
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const int tok = m0 + tb + 2 * i;
                const uint32_t n = tok < p.M ? 4u : 0u;
                const uint32_t* row = reinterpret_cast<const uint32_t*>(
                    p.xq + static_cast<int64_t>(tok < p.M ? tok : 0) * p.xrow + 292 * s + 4) + wq;
#pragma unroll
                for (int g = 0; g < 4; ++g) cp_async4(xs + 128 * i + 16 * g, row + 16 * g, n);
            }
            cp_async_commit();
            const int btok = m0 + (etid >> 2);
            const uint32_t* bs = reinterpret_cast<const uint32_t*>(
                p.xq + static_cast<int64_t>(btok < p.M ? btok : 0) * p.xrow + 292 * s + 260);
            bsw[0] = btok < p.M ? __ldg(bs + 2 * (etid & 3)) : 0u;
            bsw[1] = btok < p.M ? __ldg(bs + 2 * (etid & 3) + 1) : 0u;
            const int dtok = m0 + etid;
            dxw = (etid < BN && dtok < p.M)
                      ? __ldg(reinterpret_cast<const float*>(p.xq + static_cast<int64_t>(dtok) * p.xrow + 292 * s))
                      : 0.0f;
        };
        auto put_b = [&](int s) -> bool {
            cp_async_wait_all();
            const int ms = s % NMIN;
            if (!warp_wait(&bars[B_MIN_EMPTY + ms], ((s / NMIN) & 1) ^ 1, abort_flag, p.status)) return false;
            __half* bh = reinterpret_cast<__half*>(smem + OFF_MIN + ms * MIN_BYTES + AC_BYTES + AI_BYTES +
                                                   tc::tile_off(etid >> 2, 0, 16));
            const int j = 2 * (etid & 3);
            bmin_entry(bsw[0], bh[j], bh[64 + j]);           // k = 8 + j: next core matrix (+128 B)
            bmin_entry(bsw[1], bh[j + 1], bh[65 + j]);
            fence_proxy_async_smem();
            warp_arrive(&bars[B_MIN_FULL + ms], lane);
            if (etid < BN) {
                const int ds = s % NDX;
                if (!warp_wait(&bars[B_DX_EMPTY + ds], ((s / NDX) & 1) ^ 1, abort_flag, p.status)) return false;
                reinterpret_cast<float*>(smem + OFF_DX + ds * SCL_BYTES)[etid] = dxw;
                warp_arrive(&bars[B_DX_FULL + ds], lane);
            }
            // word wq of token t = tb + 2i: elements 4wq..4wq+3 of the quarter, at
            // tile_off_sw128(t, 4wq) = 128 t + 16 ((wq / 2) ^ (t % 8)) + 8 (wq % 2), t % 8 = (tb % 8) ^ 2i
            const int cx = (((wq >> 1) ^ (tb & 7)) << 4) + (wq & 1) * 8;
            // two quarters per fence and arrival pair
#pragma unroll
            for (int g2 = 0; g2 < 4; g2 += 2) {
#pragma unroll
                for (int g = g2; g < g2 + 2; ++g) {
                    const int q = 4 * s + g, st = q % NSTAGE;
                    if (!warp_wait(&bars[B_OP_EMPTY + st], ((q / NSTAGE) & 1) ^ 1, abort_flag, p.status)) return false;
                    uint8_t* bt = smem + OFF_STAGE + st * STAGE_BYTES + A_BYTES + tb * 128;
#pragma unroll
                    for (int i = 0; i < NI; ++i) {
                        uint32_t o0, o1;
                        s8x4_half_0213(xs[128 * i + 16 * g], o0, o1);
                        *reinterpret_cast<uint2*>(bt + 256 * i + (cx ^ (i << 5))) = make_uint2(o0, o1);
                    }
                }
                fence_proxy_async_smem();   // for the local MMAs (and warp 2's copy to the peer)
                __syncwarp();
                if (lane == 0) {
                    constexpr int BAR = SHARE_B ? B_SLICE : B_OP_FULL;
                    tc::mbar_arrive(&bars[BAR + (4 * s + g2) % NSTAGE]);
                    tc::mbar_arrive(&bars[BAR + (4 * s + g2 + 1) % NSTAGE]);
                }
            }
            return true;
        };
        const int c0 = ((warp - EPI_WARP0) >> 2) * COLS;   // first token column of this warp
        // With a workspace, a warp whose 32 token columns are all past M (a
        // short last tile) skips the drain arithmetic: those columns are never
        // stored. (Without one, the same skip measured slower on full tiles.)
        const bool math_live = !PRE || m0 + c0 < p.M;
        const int gq = lane >> 2, tq = lane & 3;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        uint64_t y[16];                                   // [h][e][g]: token pair u = 0, 1
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = 0;
        const uint64_t m1 = tc::pk(-1.0f, -1.0f);
        bool ok = true;
        if (!PRE && !split) {
            fetch_b(0);
            ok = put_b(0);
            if (ns > 1) fetch_b(1);
        }
        for (int s = 0; s < ns && ok; ++s) {
            if (!PRE && !split)
                if (s + 1 < ns) {
                    if (!put_b(s + 1)) {
                        ok = false;
                        break;
                    }
                    if (s + 2 < ns) fetch_b(s + 2);
                }
            const int b = s & 1, ds = s % NDX;
            const bool got = mbar_wait_bounded_sleep(&bars[B_ACC_FULL + b], (s >> 1) & 1, WAIT_LIMIT_NS) &&
                             mbar_wait_bounded_sleep(&bars[B_DX_FULL + ds], (s / NDX) & 1, WAIT_LIMIT_NS);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) { abort_flag.set(1); atomicOr(p.status, CQ_DEV_WAIT_TIMEOUT); }
                ok = false;
                break;
            }
            tc::fence_after();
            const float* dxs = reinterpret_cast<const float*>(smem + OFF_DX + ds * SCL_BYTES);
            const uint32_t* dds = reinterpret_cast<const uint32_t*>(smem + OFF_DX + ds * SCL_BYTES + DX_BYTES);
            // Fixed order: t = fma(d, RN(X - (-C)), -(dmin * I)); y = fma(d_x, t, y).
            if (math_live) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint64_t d2[2], nm2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const uint32_t dd = dds[quarter * 32 + 16 * h + 8 * e + gq];
                        const float d = h2f(dd), ndmin = -h2f(dd >> 16);
                        d2[e] = tc::pk(d, d);
                        nm2[e] = tc::pk(ndmin, ndmin);
                    }
                    const uint32_t la = lane_base + (static_cast<uint32_t>(16 * h) << 16) + c0;
#pragma unroll
                    for (int gp = 0; gp < 2; ++gp) {
                        uint32_t xv[8], cv[8], iv[8];
                        tc::ld16x256b_x2(la + b * BN + 16 * gp, xv);
                        tc::ld16x256b_x2(la + COL_C + 16 * gp, cv);
                        tc::ld16x256b_x2(la + COL_I + 16 * gp, iv);
                        tc::wait_ld();
#pragma unroll
                        for (int gg = 0; gg < 2; ++gg) {
                            const int g = 2 * gp + gg;
                            const float2 dx = *reinterpret_cast<const float2*>(dxs + c0 + 8 * g + 2 * tq);
                            const uint64_t dx2 = tc::pk(dx.x, dx.y);
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int i = 4 * gg + 2 * e;
                                const uint64_t S = tc::fma2(tc::pk(__uint_as_float(cv[i]), __uint_as_float(cv[i + 1])), m1,
                                                            tc::pk(__uint_as_float(xv[i]), __uint_as_float(xv[i + 1])));
                                const uint64_t tn =
                                    tc::mul2(nm2[e], tc::pk(__uint_as_float(iv[i]), __uint_as_float(iv[i + 1])));
                                const uint64_t t = tc::fma2(d2[e], S, tn);
                                uint64_t& yy = y[(2 * h + e) * 4 + g];
                                yy = tc::fma2(dx2, t, yy);
                            }
                        }
                    }
                }
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&bars[B_X_EMPTY + b]);
                tc::mbar_arrive(&bars[B_CI_EMPTY]);
                tc::mbar_arrive(&bars[B_DX_EMPTY + ds]);
            }
        }
        if (!PRE) cp_async_wait_all();   // no copy into the staging area outlives the loop
        if (ok && __all_sync(0xffffffffu, !abort_flag.get())) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int row = n0 + quarter * 32 + 16 * h + 8 * e + gq;
                    if (row >= p.N) continue;
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        float v[2];
                        tc::upk(y[(2 * h + e) * 4 + g], v[0], v[1]);
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int m = m0 + c0 + 8 * g + 2 * tq + u;
                            if (m < p.M) p.y[static_cast<int64_t>(m) * p.N + row] = v[u];
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
        for (int i = 0; i < 2; ++i) (void)mbar_wait_bounded(&bars[B_ACC_FULL + i], 0, WAIT_LIMIT_NS / 8);
        if (CS > 1) {   // let a copy the peer issued before it gave up land in this CTA's shared memory
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 50000u) __nanosleep(1000);
        }
    }
    __syncthreads();
    // The peer may still copy into, or arrive on, this CTA's shared memory
    // until it is done: neither leaves before both are.
    if constexpr (CS > 1) tc::cluster_sync();
    tc::fence_after();
    if (warp == 1) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// Pre-conversion of Q8_K activations for cq_gemm_ws: one CTA per (superblock
// s, token tile), thread (token t, K-half h). Writes the tile's image -- the
// B operands, B_min and d_x, the same values and layout the in-kernel
// converters produce.
__global__ void __launch_bounds__(256) gemm_prep_kernel(const GemmParams p, uint8_t* bimg) {
    pdl_trigger();
    pdl_wait();
    const int s = blockIdx.x, tile = blockIdx.y, ns = p.ns;
    const int t = threadIdx.x >> 1, h = threadIdx.x & 1;
    const int m = tile * BN + t;
    const bool on = m < p.M;
    const uint8_t* blk = p.xq + static_cast<int64_t>(m) * p.xrow + 292 * s;
    uint8_t* img = bimg + (static_cast<int64_t>(tile) * ns + s) * IMG_BYTES;
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(blk + 4 + 128 * h);
    uint8_t* bt = img + 2 * h * B_BYTES;    // quarters 2h and 2h + 1
#pragma unroll 4
    for (int g = 0; g < KH / 8; ++g) {       // 8 elements (one core-matrix row) per store
        uint32_t o0[2] = {0u, 0u}, o1[2] = {0u, 0u};
        if (on) {
            s8x4_half_0213(__ldg(qw + 2 * g), o0[0], o0[1]);
            s8x4_half_0213(__ldg(qw + 2 * g + 1), o1[0], o1[1]);
        }
        *reinterpret_cast<uint4*>(bt + tc::tile_off_sw128(t, 8 * g, BN)) = make_uint4(o0[0], o0[1], o1[0], o1[1]);
    }
    if (h == 0) {
        reinterpret_cast<float*>(img + 4 * B_BYTES + BMIN_BYTES)[t] =
            on ? __ldg(reinterpret_cast<const float*>(blk)) : 0.0f;
    } else {
        // B_min: token t = [64 h_0 .. 64 h_7, l_0 .. l_7], B_j = 64 h_j + l_j
        __half* bh = reinterpret_cast<__half*>(img + 4 * B_BYTES + tc::tile_off(t, 0, 16));
#pragma unroll
        for (int j = 0; j < 8; ++j)
            bmin_entry(on ? __ldg(reinterpret_cast<const uint32_t*>(blk + 260) + j) : 0u, bh[j], bh[64 + j]);
    }
}

// ------------------------------------------------------------ host side
}  // namespace

size_t gemm_workspace_size(int w_fmt, int64_t M, int64_t K) {
    if (w_fmt != CQ_Q4_K) return gemm32_workspace_size(w_fmt, M, K);
    if (M <= 0) return 0;
    const int64_t cells = (M + BN - 1) / BN * (K / 256);
    return static_cast<size_t>(cells) * IMG_BYTES;
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
    if (workspace != nullptr) p.bimg = static_cast<const uint8_t*>(workspace);
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
    const int pre = workspace != nullptr;
    const int tiles_n = static_cast<int>((N + BM - 1) / BM);
    // Two-CTA clusters when the paired dimension is even: with a workspace
    // token tiles (sharing the weight conversion), without one weight tiles
    // (sharing the activation conversion).
    // A single short token tile without a workspace (M <= 96) runs alone, with
    // the split epilogue.
    const bool short_tile = !pre && M <= 3 * (BN / 4);
    const int cs = !short_tile && (pre ? tiles_m : tiles_n) % 2 == 0 ? 2 : 1;
    const int smem_bytes = pre ? Layout<true>::SMEM_BYTES : Layout<false>::SMEM_BYTES;
    if (smem_bytes > dev.smem_optin) return cudaErrorInvalidConfiguration;
    const void* kern = pre ? (cs == 2 ? reinterpret_cast<const void*>(gemm_q4k_kernel<true, 2, false>)
                                      : reinterpret_cast<const void*>(gemm_q4k_kernel<true, 1, false>))
                           : short_tile ? reinterpret_cast<const void*>(gemm_q4k_kernel<false, 1, true>)
                           : (cs == 2 ? reinterpret_cast<const void*>(gemm_q4k_kernel<false, 2, false>)
                                      : reinterpret_cast<const void*>(gemm_q4k_kernel<false, 1, false>));
    cudaError_t e = raise_smem_limit(kern, smem_bytes);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>((N + BM - 1) / BM), static_cast<unsigned>(tiles_m));
    if (pre) {
        e = launch_kernel(gemm_prep_kernel, dim3(static_cast<unsigned>(p.ns), static_cast<unsigned>(tiles_m)),
                          dim3(256), 0, s, p, const_cast<uint8_t*>(p.bimg));
        if (e != cudaSuccess) return e;
        // A cluster launch the device cannot place (e.g. too few SMs in a
        // partition) is refused before anything runs: fall back to single CTAs.
        if (cs == 2 && launch_kernel_cluster(gemm_q4k_kernel<true, 2, false>, grid, dim3(THREADS), smem_bytes, s,
                                             dim3(1, 2, 1), map, p) == cudaSuccess)
            return cudaSuccess;
        if (cs == 2) (void)cudaGetLastError();   // the refused launch's error is not the caller's
        e = raise_smem_limit(reinterpret_cast<const void*>(gemm_q4k_kernel<true, 1, false>), smem_bytes);
        if (e != cudaSuccess) return e;
        return launch_kernel(gemm_q4k_kernel<true, 1, false>, grid, dim3(THREADS), smem_bytes, s, map, p);
    }
    if (short_tile) return launch_kernel(gemm_q4k_kernel<false, 1, true>, grid, dim3(THREADS), smem_bytes, s, map, p);
    if (cs == 2 && launch_kernel_cluster(gemm_q4k_kernel<false, 2, false>, grid, dim3(THREADS), smem_bytes, s,
                                         dim3(2, 1, 1), map, p) == cudaSuccess)
        return cudaSuccess;
    if (cs == 2) (void)cudaGetLastError();
    e = raise_smem_limit(reinterpret_cast<const void*>(gemm_q4k_kernel<false, 1, false>), smem_bytes);
    if (e != cudaSuccess) return e;
    return launch_kernel(gemm_q4k_kernel<false, 1, false>, grid, dim3(THREADS), smem_bytes, s, map, p);
}

}  // namespace cq
