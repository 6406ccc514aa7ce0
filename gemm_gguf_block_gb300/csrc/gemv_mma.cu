// Batched GEMV for up to 16 tokens on the tensor cores (Q4_0, Q4_1, Q8_0):
// cq_gemv from 2 tokens, and cq_gemv_packed (weights repacked by cq_repack)
// from 1.
//
// cera README "Other features" and 0.5 release notes: the speculative-decoding
// verify path projects all 1 + k positions through the LM head in one batched
// pass, so the head is read once per round; alice-llm "Batch-4 Speculative
// Decoding": weights decoded once, one accumulator set per position, and the
// batched result equal to the single-position one.
//
// Per 32-element block the integer dot is an exact fp16 tensor-core product,
// mma.sync m16n8k16 twice per block. The weight operand holds BIAS + v for a
// quant of value v (4-bit high nibbles: 1024 + 16 v against activations
// scaled by 1/16), built from the packed bytes by one lop3 per pair, and the
// accumulator starts at minus the matching multiple of the activation sums:
// every operand and partial sum is an integer below 2^23, so the result is
// the exact integer dot (mma_frag.cuh). The block's
// scale terms are then applied on the CUDA cores, two tokens per f32x2
// instruction, in the library's fixed order (include/cq.h):
// c = fma(d_w * d_x, isum, c) [+ fma(m_w, s_x, c) for Q4_1] over four
// blocks, y = y + c per chunk. Every (row, token) chain lives in one thread,
// so each row equals the single-token GEMV row bit for bit.
//
// A persistent CTA stages the tokens' activations once as fp16 in shared
// memory, then a producer warp streams weight tiles of 16 * RW * RG rows
// through a ring of stages: 2-D TMA boxes of the tile's rows x 8 or 4 blocks
// (GGUF layout), or one bulk copy of the tile's 16-row x 4-block units
// (packed layout). Each of the RG consumer warps owns RW row groups of 16 rows
// and all the tokens (NT n-tiles of 8). The activation fragments and scale
// records a warp reads from shared memory per block serve all its row groups:
// with one row group per warp they made two thirds of the shared-memory
// wavefronts and kept that pipe about 60% busy, so the long tiles take two
// (choose_tile below).
#include <algorithm>

#include <cuda_fp16.h>

#include "cq_device.cuh"
#include "cq_internal.h"
#include "mma_frag.cuh"
#include "tc.cuh"

namespace cq {
namespace {

constexpr int MAX_STAGES = 4;

using mf::MF;
using mf::stage_pitch;

// Bytes per weight row in a stage of sb blocks: 8 blocks as the shared
// stage_pitch; 4 Q4_1 blocks are 80 bytes (20 words: the 8 rows one load
// instruction touches fall in 8 different bank groups).
__host__ __device__ constexpr int seg_pitch(int bb, int sb) { return sb == 8 ? stage_pitch(bb) : sb * bb; }

struct MmaParams {
    const uint8_t* W;
    const uint8_t* xq;
    float* y;
    int* status;
    int M, N, K;
    int nb;             // blocks per row
    int64_t wrow;       // bytes per weight row
    int act_pitch;      // bytes per staged token row (fp16, padded)
    int stage_bytes;
    int stages;
    int smem_act;       // offset of the staged activations
    int smem_scale;     // offset of the per-(block, token pair) scale table
    int smem_stage;     // offset of the weight stages
    int ngroups;        // packed weights: 16-row groups (ceil(N / 16))
};

// Packed weights (cq_repack): a unit of 16 rows x 4 blocks is 64 * BB bytes,
// the rows' scale fields (4 * SCALE bytes per row) first, then the quant
// words, per (half, row, lane t) the words of blocks 0..3 as 16 bytes.
template <int WF> struct Pk {
    static constexpr int UNIT = 64 * MF<WF>::BB;
    static constexpr int SCALE = WF == CQ_Q4_1 ? 4 : 2;     // scale bytes per block
    static constexpr int QUANTS = 64 * SCALE;               // offset of the quant words
};
__device__ __forceinline__ uint32_t word(const uint4& v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// One unit's share of a lane for rows g and g+8 of a row group: quant words of
// blocks 0..3 (and, Q8_0, the second halves) and the scale fields.
template <int WF>
struct PkRows {
    uint4 q0, q1, q0b, q1b, s0, s1;
    __device__ __forceinline__ void load(const uint8_t* unit, int g, int t) {
        const uint8_t* q = unit + Pk<WF>::QUANTS + 16 * (4 * g + t);
        q0 = *reinterpret_cast<const uint4*>(q);
        q1 = *reinterpret_cast<const uint4*>(q + 16 * 32);
        if constexpr (WF == CQ_Q8_0) {
            q0b = *reinterpret_cast<const uint4*>(q + 1024);
            q1b = *reinterpret_cast<const uint4*>(q + 1024 + 16 * 32);
        }
        if constexpr (WF == CQ_Q4_1) {
            s0 = *reinterpret_cast<const uint4*>(unit + 16 * g);
            s1 = *reinterpret_cast<const uint4*>(unit + 16 * (g + 8));
        } else {
            const uint2 a = *reinterpret_cast<const uint2*>(unit + 8 * g);
            const uint2 b = *reinterpret_cast<const uint2*>(unit + 8 * (g + 8));
            s0 = make_uint4(a.x, a.y, 0, 0);
            s1 = make_uint4(b.x, b.y, 0, 0);
        }
    }
    // Block j's A fragments and (v, v) scale pairs, as mf::weight_frags gives them.
    __device__ __forceinline__ void frags(int j, uint32_t (&a0)[4], uint32_t (&a1)[4], uint64_t& dw0, uint64_t& dw1,
                                          uint64_t& mw0, uint64_t& mw1) const {
        uint32_t qb0 = 0, qb1 = 0;
        if constexpr (WF == CQ_Q8_0) {
            qb0 = word(q0b, j);
            qb1 = word(q1b, j);
        }
        mf::a_frags<WF>(word(q0, j), word(q1, j), qb0, qb1, a0, a1);
        if constexpr (WF == CQ_Q4_1) {
            const uint32_t dm0 = word(s0, j), dm1 = word(s1, j);
            const float d0 = h2f(dm0), d1 = h2f(dm1), m0 = h2f(dm0 >> 16), m1 = h2f(dm1 >> 16);
            dw0 = tc::pk(d0, d0);
            dw1 = tc::pk(d1, d1);
            mw0 = tc::pk(m0, m0);
            mw1 = tc::pk(m1, m1);
        } else {
            const uint32_t w0 = word(s0, j >> 1), w1 = word(s1, j >> 1);
            const float d0 = h2f(j & 1 ? w0 >> 16 : w0), d1 = h2f(j & 1 ? w1 >> 16 : w1);
            dw0 = tc::pk(d0, d0);
            dw1 = tc::pk(d1, d1);
            mw0 = mw1 = 0;
        }
    }
};

template <int WF, int RG, int NT, int RW, int SB, bool PK>
__global__ void __launch_bounds__((RG + 1) * 32, 1)
    gemv_mma_kernel(const __grid_constant__ CUtensorMap wmap, const MmaParams p) {
    pdl_trigger();
    pdl_wait();
    using F = MF<WF>;
    constexpr int NPAIR = NT * 4;                  // token pairs
    constexpr int CONSUMERS = RG;
    constexpr int ROWS = 16 * RW * RG;
    constexpr int NBOX = (ROWS + 255) / 256;      // TMA boxes per stage
    static_assert(ROWS % NBOX == 0, "tile rows split evenly into boxes");
    static_assert(PK || seg_pitch(F::BB, SB) % 16 == 0, "a stage row is a whole number of 16-byte units");
    static_assert(!PK || (SB == 4 && RW * RG * 16 == ROWS), "packed stages are one unit per row group");
    constexpr int GPT = ROWS / 16;                // 16-row groups per tile
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + MAX_STAGES;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.stages;
    const int tiles = (p.N + ROWS - 1) / ROWS;
    const int nseg = p.nb / SB;
    const int my_tiles = blockIdx.x < tiles ? (tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t steps = static_cast<int64_t>(my_tiles) * nseg;

    const bool producer = warp == CONSUMERS && lane == 0;
    auto issue = [&](int64_t k) {
        const int st = static_cast<int>(k % S);
        const int tile = blockIdx.x + static_cast<int>(k / nseg) * gridDim.x;
        const int seg = static_cast<int>(k % nseg);
        if constexpr (PK) {
            // the tile's groups of segment seg are one contiguous range
            const int g0 = tile * GPT;
            const int ng = min(GPT, p.ngroups - g0);
            const uint32_t bytes = static_cast<uint32_t>(ng * Pk<WF>::UNIT);
            mbar_arrive_expect_tx(&full[st], bytes);
            bulk_g2s(smem + p.smem_stage + st * p.stage_bytes,
                     p.W + (static_cast<int64_t>(seg) * p.ngroups + g0) * Pk<WF>::UNIT, bytes, &full[st],
                     policy_evict_first());
            return;
        }
        mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(p.stage_bytes));
        // x counts 2-byte elements of the row; a box holds at most 256 rows
#pragma unroll
        for (int j = 0; j < NBOX; ++j)
            tc::tma_load_2d(smem + p.smem_stage + st * p.stage_bytes + j * (ROWS / NBOX) * seg_pitch(F::BB, SB), &wmap,
                            seg * SB * F::BB / 2, tile * ROWS + j * (ROWS / NBOX), &full[st]);
    };
    // The weight stream starts before the activations are staged: the first
    // S stages need no release.
    int64_t k0 = 0;
    if (producer) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], CONSUMERS);
        }
        fence_mbar_init();
        for (; k0 < steps && k0 < S; ++k0) issue(k0);
    }
    // Stage the activations once. Per (token m, block b): the 32 quants as
    // fp16 in four 16-byte chunks, chunk t = elements [4t, 4t+2, 4t+1, 4t+3,
    // 16+4t, 18+4t, 17+4t, 19+4t] (lane t's B fragments of both k-steps, see
    // mf::act_frags); per (block b, token pair j): {d_x, d_x', bias, bias'}
    // and, for Q8_1, {s_x, s_x'}. Tokens >= M are zero.
    {
        float* sc = reinterpret_cast<float*>(smem + p.smem_scale);
        const int total = NT * 8 * p.nb;
        for (int i = threadIdx.x; i < total; i += blockDim.x) {
            const int m = i / p.nb, b = i - m * p.nb;
            uint4 ch[4] = {};
            float d = 0.0f, sx = 0.0f;
            int bias = 0;
            if (m < p.M) mf::act_frags<WF>(p.xq + (static_cast<int64_t>(m) * p.nb + b) * F::ABB, ch, d, sx, bias);
            uint4* dst = reinterpret_cast<uint4*>(smem + p.smem_act + m * p.act_pitch + 64 * b);
#pragma unroll
            for (int t = 0; t < 4; ++t) dst[t] = ch[t];
            const int j = m >> 1, hi = m & 1;
            float* e = sc + (b * NPAIR + j) * 4;
            e[hi] = d;
            e[2 + hi] = static_cast<float>(bias);
            if constexpr (WF == CQ_Q4_1) sc[p.nb * NPAIR * 4 + (b * NPAIR + j) * 2 + hi] = sx;
        }
    }
    __syncthreads();

    if (warp == CONSUMERS) {
        // -------------------------------------------------------- producer
        if (producer) {
            for (int64_t k = k0; k < steps; ++k) {
                const int st = static_cast<int>(k % S);
                if (!mbar_wait_bounded(&empty[st], static_cast<uint32_t>(((k / S) & 1) ^ 1), WAIT_LIMIT_NS)) {
                    atomicOr(p.status, CQ_DEV_WAIT_TIMEOUT);
                    break;
                }
                issue(k);
            }
        }
    } else {
        // -------------------------------------------------------- consumers
        // Tile rows 16 RW w .. 16 RW (w + 1) - 1, all tokens.
        const int g = lane >> 2, t = lane & 3;
        const uint8_t* act = smem + p.smem_act + g * p.act_pitch + 16 * t;
        const float4* sc4 = reinterpret_cast<const float4*>(smem + p.smem_scale) + t;
        const float2* sx2 = reinterpret_cast<const float2*>(smem + p.smem_scale + p.nb * NPAIR * 16) + t;
        constexpr int seg_row_bytes = seg_pitch(F::BB, SB);
        uint64_t c[RW][NT][2], y[RW][NT][2];   // group r: (row g | row g+8) x (token 8n+2t, 8n+2t+1)
        int64_t k = 0;
        bool ok = true;
        for (int ti = 0; ti < my_tiles && ok; ++ti) {
            const int tile = blockIdx.x + ti * gridDim.x;
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int n = 0; n < NT; ++n) y[r][n][0] = y[r][n][1] = 0;
            for (int seg = 0; seg < nseg; ++seg, ++k) {
                const int st = static_cast<int>(k % S);
                if (!mbar_wait_bounded(&full[st], static_cast<uint32_t>((k / S) & 1), WAIT_LIMIT_NS)) {
                    if (lane == 0) atomicOr(p.status, CQ_DEV_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                const uint8_t* r0p = smem + p.smem_stage + st * p.stage_bytes + (16 * RW * warp + g) * seg_row_bytes;
                PkRows<WF> pk[PK ? RW : 1];
                if constexpr (PK) {
#pragma unroll
                    for (int r = 0; r < RW; ++r)
                        pk[r].load(smem + p.smem_stage + st * p.stage_bytes + (RW * warp + r) * Pk<WF>::UNIT, g, t);
                }
#pragma unroll 4
                for (int bi = 0; bi < SB; ++bi) {
                    const int b = seg * SB + bi;                  // block index along K
                    uint32_t a0[RW][4], a1[RW][4];
                    uint64_t dw0[RW], dw1[RW], mw0[RW], mw1[RW];
#pragma unroll
                    for (int r = 0; r < RW; ++r) {
                        if constexpr (PK) {
                            pk[r].frags(bi, a0[r], a1[r], dw0[r], dw1[r], mw0[r], mw1[r]);
                        } else {
                            const uint8_t* wr = r0p + 16 * r * seg_row_bytes + bi * F::BB;
                            mf::weight_frags<WF>(wr, wr + 8 * seg_row_bytes, t, a0[r], a1[r], dw0[r], dw1[r], mw0[r],
                                                 mw1[r]);
                        }
                    }
                    if ((b & 3) == 0) {
#pragma unroll
                        for (int r = 0; r < RW; ++r)
#pragma unroll
                            for (int n = 0; n < NT; ++n) c[r][n][0] = c[r][n][1] = 0;
                    }
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const uint4 bv = *reinterpret_cast<const uint4*>(act + 8 * n * p.act_pitch + 64 * b);
                        const float4 s4 = sc4[b * NPAIR + 4 * n];
                        const uint64_t dx = tc::pk(s4.x, s4.y);
                        uint64_t sx = 0;
                        if constexpr (WF == CQ_Q4_1) {
                            const float2 s2 = sx2[b * NPAIR + 4 * n];
                            sx = tc::pk(s2.x, s2.y);
                        }
#pragma unroll
                        for (int r = 0; r < RW; ++r) {
                            float acc[4];
                            mf::mma16816c(acc, a0[r], bv.x, bv.y, s4.z, s4.w);
                            mf::mma16816acc(acc, a1[r], bv.z, bv.w);
                            // c = fma(d_w * d_x, isum, c) per element, two tokens per instruction
                            c[r][n][0] = tc::fma2(tc::mul2(dw0[r], dx), tc::pk(acc[0], acc[1]), c[r][n][0]);
                            c[r][n][1] = tc::fma2(tc::mul2(dw1[r], dx), tc::pk(acc[2], acc[3]), c[r][n][1]);
                            if constexpr (WF == CQ_Q4_1) {
                                c[r][n][0] = tc::fma2(mw0[r], sx, c[r][n][0]);
                                c[r][n][1] = tc::fma2(mw1[r], sx, c[r][n][1]);
                            }
                        }
                    }
                    if ((b & 3) == 3) {
#pragma unroll
                        for (int r = 0; r < RW; ++r)
#pragma unroll
                            for (int n = 0; n < NT; ++n) {
                                y[r][n][0] = tc::add2(y[r][n][0], c[r][n][0]);
                                y[r][n][1] = tc::add2(y[r][n][1], c[r][n][1]);
                            }
                    }
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&empty[st]);
            }
            if (!ok) break;
            // y[token][row]: rows 16 (RW w + r) + g (+ 8), tokens 8n+2t, 8n+2t+1
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int r0 = tile * ROWS + 16 * (RW * warp + r) + g;
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const int m0 = 8 * n + 2 * t;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float v[2];
                        tc::upk(y[r][n][h], v[0], v[1]);
                        const int row = r0 + 8 * h;
#pragma unroll
                        for (int i = 0; i < 2; ++i)
                            if (row < p.N && m0 + i < p.M) p.y[static_cast<int64_t>(m0 + i) * p.N + row] = v[i];
                    }
                }
            }
        }
    }
    // Let the producer's last copies land before the CTA's shared memory goes.
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int64_t k = steps > S ? steps - S : 0; k < steps; ++k)
            (void)mbar_wait_bounded(&full[k % S], static_cast<uint32_t>((k / S) & 1), WAIT_LIMIT_NS / 8);
    }
}

// Shared-memory layout for M tokens, K columns and RG row groups: barriers,
// the fp16 activation tile, the scale table, then the weight stages.
struct MmaSmem {
    int act_pitch, act, scale, stage, stage_bytes, fixed;
};
MmaSmem mma_smem(int bb, int M, int64_t K, int rows, int sb) {
    MmaSmem m{};
    const int NT = M <= 8 ? 1 : 2;
    const int nb = static_cast<int>(K / 32);
    m.act_pitch = static_cast<int>(K) * 2 + 64;      // 64 mod 128: token rows g, g+1 on different bank halves
    m.act = 1024;
    m.scale = m.act + (NT * 8 * m.act_pitch + 127) / 128 * 128;
    const int scale_bytes = nb * NT * 4 * (bb == 20 ? 24 : 16);
    m.stage = m.scale + (scale_bytes + 1023) / 1024 * 1024;
    m.stage_bytes = rows * seg_pitch(bb, sb);
    m.fixed = m.stage;
    return m;
}

// Tile shapes: RG consumer warps x RW row groups of 16 rows, SB blocks per
// stage. Each warp streams its rows over all of K, so a CTA's time goes with
// the rows of its largest share of tiles. Of the shapes that fit with their
// stages, the first in order of preference whose rows per CTA are within a
// slack of the least is taken: for up to 8 tokens 14 x 32 rows (Q4_1 with
// 4-block stages), then 7 x 32, then 8 x 16; for up to 16 tokens 9 x 32 for
// Q4_1 (4-block stages) and 7 x 32 for the others (at 16 tokens the
// activation fragments and scale records a warp reads per block are most of
// the shared-memory traffic, and a second row group halves them per row; 14
// warps would not fit their registers), then 12 x 16, then 8 x 16. The
// 128256-row LM head gets 2 tiles of 448 rows per SM up to 8 tokens (the same
// 896 rows as 7 tiles of 128) and, for Q4_1, 3 of 288 up to 16.
// Packed weights (one 4-block unit per row group and stage) take the same
// shapes with 4-block stages for every format.
struct TileShape {
    int rg, rw, sb;
    int rows() const { return 16 * rg * rw; }
};
TileShape choose_tile(int bb, int M, int64_t N, int64_t K, int sms, int lim, bool pk) {
    const TileShape cand1[] = {{14, 2, bb == 20 ? 4 : 8}, {7, 2, 8}, {8, 1, 8}};
    const TileShape cand2[] = {bb == 20 ? TileShape{9, 2, 4} : TileShape{7, 2, 8}, {12, 1, 8}, {8, 1, 8}};
    const TileShape pk1[] = {{14, 2, 4}, {7, 2, 4}, {8, 1, 4}};
    const TileShape pk2[] = {bb == 20 ? TileShape{9, 2, 4} : TileShape{7, 2, 4}, {12, 1, 4}, {8, 1, 4}};
    const TileShape* cand = pk ? (M <= 8 ? pk1 : pk2) : (M <= 8 ? cand1 : cand2);
    const int nc = 3;
    // Three stages up to 8 tokens, except for Q8_0, whose 272-byte rows fit
    // only two of the 7 x 32 tile: two of those measured faster than three of
    // 8 x 16 (LM head M = 4: 110.5 against 114.6 us).
    const int min_stages = M <= 8 && bb != 34 ? 3 : 2;
    auto rows_per_cta = [&](int rows) {
        const int64_t tiles = (N + rows - 1) / rows;
        return (tiles + sms - 1) / sms * rows;
    };
    int64_t best = INT64_MAX;
    for (int i = 0; i < nc; ++i) best = std::min(best, rows_per_cta(cand[i].rows()));
    const int64_t slack = M <= 8 ? 0 : best / 8;
    for (int i = 0; i < nc - 1; ++i) {
        const MmaSmem L = mma_smem(bb, M, K, cand[i].rows(), cand[i].sb);
        if ((lim - L.fixed) / L.stage_bytes >= min_stages && rows_per_cta(cand[i].rows()) <= best + slack)
            return cand[i];
    }
    return cand[nc - 1];
}

template <int WF, int RG, int NT, int RW, int SB, bool PK = false>
cudaError_t launch_mma_typed(const DeviceInfo& dev, MmaParams p, const CUtensorMap& map, cudaStream_t s) {
    const int smem = p.smem_stage + p.stages * p.stage_bytes;
    const cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(gemv_mma_kernel<WF, RG, NT, RW, SB, PK>),
                                           std::min(dev.smem_optin, 227 * 1024));
    if (e != cudaSuccess) return e;
    const int tiles = (p.N + 16 * RW * RG - 1) / (16 * RW * RG);
    const int grid = std::min(tiles, dev.sm_count);
    return launch_kernel(gemv_mma_kernel<WF, RG, NT, RW, SB, PK>, dim3(grid), dim3((RG + 1) * 32), smem, s, map, p);
}

template <int WF>
cudaError_t launch_mma_fmt(const DeviceInfo& dev, int M, int64_t N, int64_t K, const void* W, const void* xq,
                           float* y, bool pk, cudaStream_t s) {
    using F = MF<WF>;
    MmaParams p{};
    p.W = static_cast<const uint8_t*>(W);
    p.xq = static_cast<const uint8_t*>(xq);
    p.y = y;
    p.status = dev.status;
    p.M = M;
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.nb = static_cast<int>(K / 32);
    p.wrow = static_cast<int64_t>(p.nb) * F::BB;
    const int NT = M <= 8 ? 1 : 2;
    const int lim = std::min(dev.smem_optin, 227 * 1024);
    const TileShape T = choose_tile(F::BB, M, N, K, dev.sm_count, lim, pk);
    const MmaSmem L = mma_smem(F::BB, M, K, T.rows(), T.sb);
    p.act_pitch = L.act_pitch;
    p.stage_bytes = L.stage_bytes;
    p.smem_act = L.act;
    p.smem_scale = L.scale;
    p.smem_stage = L.stage;
    p.stages = std::min(MAX_STAGES, (lim - L.fixed) / L.stage_bytes);
    if (p.stages < 2) return cudaErrorInvalidConfiguration;
    if (pk) {
        // packed weights: each stage is one bulk copy, no tensor map
        p.ngroups = static_cast<int>((N + 15) / 16);
        const CUtensorMap none{};
        if (NT == 2) {
            if constexpr (WF == CQ_Q4_1) {
                if (T.rg == 9) return launch_mma_typed<WF, 9, 2, 2, 4, true>(dev, p, none, s);
            }
            if (T.rg == 7) return launch_mma_typed<WF, 7, 2, 2, 4, true>(dev, p, none, s);
            return T.rg == 12 ? launch_mma_typed<WF, 12, 2, 1, 4, true>(dev, p, none, s)
                              : launch_mma_typed<WF, 8, 2, 1, 4, true>(dev, p, none, s);
        }
        if (T.rg == 14) return launch_mma_typed<WF, 14, 1, 2, 4, true>(dev, p, none, s);
        return T.rw == 2 ? launch_mma_typed<WF, 7, 1, 2, 4, true>(dev, p, none, s)
                         : launch_mma_typed<WF, 8, 1, 1, 4, true>(dev, p, none, s);
    }
    tc::EncodeTiledFn enc = tc::encode_tiled_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    // Raw weights as a 2-D tensor of 2-byte elements [N rows][wrow/2]; a box is
    // SB blocks of one tile's rows.
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.wrow / 2), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.wrow)};
    const int nbox = (T.rows() + 255) / 256;
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(seg_pitch(F::BB, T.sb) / 2),
                               static_cast<cuuint32_t>(T.rows() / nbox)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(W), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (NT == 2) {
        if constexpr (WF == CQ_Q4_1) {
            if (T.rg == 9) return launch_mma_typed<WF, 9, 2, 2, 4>(dev, p, map, s);
        }
        if (T.rg == 7) {
            if constexpr (WF == CQ_Q4_1) {
                if (T.sb == 4) return launch_mma_typed<WF, 7, 2, 2, 4>(dev, p, map, s);
            }
            return launch_mma_typed<WF, 7, 2, 2, 8>(dev, p, map, s);
        }
        return T.rg == 12 ? launch_mma_typed<WF, 12, 2, 1, 8>(dev, p, map, s)
                          : launch_mma_typed<WF, 8, 2, 1, 8>(dev, p, map, s);
    }
    if (T.rg == 14) {
        if constexpr (WF == CQ_Q4_1) {
            if (T.sb == 4) return launch_mma_typed<WF, 14, 1, 2, 4>(dev, p, map, s);
        }
        return launch_mma_typed<WF, 14, 1, 2, 8>(dev, p, map, s);
    }
    return T.rw == 2 ? launch_mma_typed<WF, 7, 1, 2, 8>(dev, p, map, s) : launch_mma_typed<WF, 8, 1, 1, 8>(dev, p, map, s);
}

}  // namespace

// Shared memory the tensor-core GEMV needs for M tokens and K columns with
// the minimum of two weight stages (0 when the format has no tensor-core path).
int gemv_mma_smem(int w_fmt, int M, int64_t K) {
    if (w_fmt != CQ_Q4_0 && w_fmt != CQ_Q4_1 && w_fmt != CQ_Q8_0) return 0;
    const int bb = w_fmt == CQ_Q4_0 ? 18 : w_fmt == CQ_Q4_1 ? 20 : 34;
    const MmaSmem L = mma_smem(bb, M, K, 128, 8);
    return L.fixed + 2 * L.stage_bytes;
}

cudaError_t launch_gemv_mma(const DeviceInfo& dev, int w_fmt, int M, int64_t N, int64_t K, const void* W,
                            const void* xq, float* y, cudaStream_t s) {
    switch (w_fmt) {
    case CQ_Q4_0: return launch_mma_fmt<CQ_Q4_0>(dev, M, N, K, W, xq, y, false, s);
    case CQ_Q4_1: return launch_mma_fmt<CQ_Q4_1>(dev, M, N, K, W, xq, y, false, s);
    case CQ_Q8_0: return launch_mma_fmt<CQ_Q8_0>(dev, M, N, K, W, xq, y, false, s);
    default: return cudaErrorInvalidValue;
    }
}

int gemv_packed_smem(int w_fmt, int M, int64_t K) {
    if (w_fmt != CQ_Q4_0 && w_fmt != CQ_Q4_1 && w_fmt != CQ_Q8_0) return 0;
    const int bb = w_fmt == CQ_Q4_0 ? 18 : w_fmt == CQ_Q4_1 ? 20 : 34;
    const MmaSmem L = mma_smem(bb, M, K, 128, 4);
    return L.fixed + 2 * L.stage_bytes;
}

cudaError_t launch_gemv_packed(const DeviceInfo& dev, int w_fmt, int M, int64_t N, int64_t K, const void* Wp,
                               const void* xq, float* y, cudaStream_t s) {
    switch (w_fmt) {
    case CQ_Q4_0: return launch_mma_fmt<CQ_Q4_0>(dev, M, N, K, Wp, xq, y, true, s);
    case CQ_Q4_1: return launch_mma_fmt<CQ_Q4_1>(dev, M, N, K, Wp, xq, y, true, s);
    case CQ_Q8_0: return launch_mma_fmt<CQ_Q8_0>(dev, M, N, K, Wp, xq, y, true, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace cq
