// Routed-expert FFN projections on the tensor cores, grouped by expert.
//
// cera README "Supported models" (lfm2moe): each token routes to 4 of 32
// experts; grouping tokens by expert -- the follow-up the page names -- lets
// each expert's weights be read once for all its tokens. alice-llm "WGSL
// Shader Architecture" (swiglu_fused_q4k): gate and up share one pass.
//
// One CTA = (expert e, 128 weight rows). The expert's (token, slot) pairs,
// sorted by the routing kernel, are taken up to 64 at a time. Q4_0 weights
// stream through a ring of 2-D TMA boxes (128 rows x 8 blocks; for the up
// projection the gate and up rows of the same f land in one stage); the
// pairs' 272-byte Q8_0 activation segments arrive in the same stage, four
// rows per TMA gather4 (64 single copies per segment cost as much as the
// rest of the weight stream), then are converted to fp16 in shared memory.
// Per 32-block the integer dot is an exact fp16 mma.sync m16n8k16 product
// (two chained k-steps on the fragments of mma_frag.cuh; every partial sum is
// an integer below 2^23), and the block's scale term is accumulated as
// y = fma(d_w * d_x, isum, y) in increasing k.
//   up:   warp w computes gate and up rows f0+16w.. for the pairs; the CTA
//         then writes h = silu(g) * u (fp32) and its Q8_0 blocks hq for the
//         valid pairs into the workspace.
//   down: o = W_down[e] . hq for the pairs, written into the workspace.
#include <algorithm>

#include <cuda_fp16.h>

#include "cq_device.cuh"
#include "cq_internal.h"
#include "mma_frag.cuh"
#include "tc.cuh"

namespace cq {
namespace {

constexpr int ROWS = 128;
constexpr int SEGB = 8;              // 32-blocks per segment
constexpr int TOK = 64;              // pairs per pass (8 n-tiles)
constexpr int CONSUMERS = 8;
constexpr int THREADS = (CONSUMERS + 1) * 32;
constexpr int BOX_BYTES = ROWS * SEGB * 18;        // one matrix, one segment: 18432
constexpr int ACT_PITCH = 512 + 64;                 // bytes per token per segment (fp16) + pad:
                                                    // 36 x 16 B, so lanes' 16-byte reads miss each other's banks
constexpr int ACT_BYTES = TOK * ACT_PITCH;          // 36864
// Scale records, per (32-block b, token pair j), pitch 33 records per block
// so the converters' stores spread over banks: {d_x[2j], d_x[2j+1], bias[2j],
// bias[2j+1]}, one 16-byte load per lane and n-tile (the scales as an f32x2
// pair, the biases for the mma's C fragment). One record measured 2% faster
// than a bias quad and a separate scale pair.
constexpr int SCL_PITCH = TOK / 2 + 1;
constexpr int SCL_BYTES = (SEGB * SCL_PITCH * 16 + 127) / 128 * 128;   // 4224: keeps the stages 128-byte aligned
constexpr int RAWA = SEGB * 34;                     // one token's Q8_0 segment: 272 bytes
// The pairs' raw segments arrive four at a time (one TMA gather4 of four
// activation rows); each group of four starts on a 128-byte boundary.
constexpr int RAWG = (4 * RAWA + 127) / 128 * 128;  // 1152
constexpr int RAWA_BYTES = TOK / 4 * RAWG;          // 18432
__host__ __device__ constexpr int raw_off(int tk) { return (tk >> 2) * RAWG + (tk & 3) * RAWA; }

struct MoeMmaParams {
    const uint8_t* xq;          // up: token activations (Q8_0 [T][K]); down: hq rows (Q8_0 [P][F])
    const int* offs;            // [E+1]
    const int* order;           // [E] experts, largest first
    const int* perm;            // pairs grouped by expert
    float* out;                 // up: h [P][F]; down: o [P][Kout]
    uint8_t* hq;                // up: Q8_0 of h, [P] rows of F/32 blocks
    int* status;
    int topk;
    int rows_per_expert;        // up: F; down: K (d_model)
    int kin;                    // up: K; down: F
    int64_t xrow;               // bytes per activation row
    int stages;
};


// D = A * B + C (C given), and D += A * B.
__device__ __forceinline__ void mma16816c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                          const float4& c) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c.x), "f"(c.y), "f"(c.z), "f"(c.w));
}
__device__ __forceinline__ void mma16816acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct Smem {
    uint64_t* full;
    uint64_t* empty;
    int* pairs;        // [TOK] pair ids of the pass
    uint8_t* act;      // [TOK][ACT_PITCH] fp16 activations of one segment
    float4* sq;        // [SEGB][SCL_PITCH] scale records
    uint8_t* wst;      // [stages][stage bytes]
};

// fp16 position of chunk c (16 bytes) of block b in a token's row: chunks are
// XOR-rotated by block pair so that eight converters writing the same chunk of
// blocks 0..7, and eight readers of one block, hit eight different bank groups.
__device__ __forceinline__ int chunk_pos(int b, int c) { return 64 * b + 16 * (c ^ ((b >> 1) & 3)); }

// Converts the stage's raw Q8_0 segments (272 bytes per pair, pairs past np
// read as zero) for the first 8 * NT pairs: item = (token it / 8, block it % 8).
// Chunk c of a block is lane c's B fragments of both k-steps in the order of
// mma_frag.cuh (mf::act_frags: the Q4_0 weights' high nibbles are masked in
// place, so the k-step 1 half is scaled by 1/16), and the bias is the
// accumulator's start for the weights' BIAS + v encoding.
template <int NT>
__device__ __forceinline__ void convert_acts(const uint8_t* raw, const Smem sm, int np, int ct) {
    float* sqf = reinterpret_cast<float*>(sm.sq);
    for (int it = ct; it < 8 * NT * SEGB; it += CONSUMERS * 32) {
        const int tk = it >> 3, b = it & 7;
        uint4 ch[4] = {};
        float d = 0.0f, unused;
        int ibias = 0;
        if (tk < np) mf::act_frags<CQ_Q4_0>(raw + raw_off(tk) + b * 34, ch, d, unused, ibias);
        uint8_t* row = sm.act + tk * ACT_PITCH;
#pragma unroll
        for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(row + chunk_pos(b, c)) = ch[c];
        const int j = b * SCL_PITCH + (tk >> 1), hi = tk & 1;
        const float bias = static_cast<float>(ibias);
        sqf[4 * j + hi] = d;
        sqf[4 * j + 2 + hi] = bias;
    }
}

// One pass over the expert's K for up to 8 * NT pairs. Accumulators hold
// (pair 8n + 2t, 8n + 2t + 1) of rows g (index 0) and g + 8 (index 1); per
// 32-block, isum comes exactly out of two chained fp16 MMAs and
// y = fma(d_w * d_x, isum, y) runs two pairs per f32x2 instruction.
template <bool UP, int NT>
__device__ __forceinline__ bool run_pass(const MoeMmaParams& p, const Smem sm, int S, int nseg, int64_t& k, int np,
                                      int r0) {
    constexpr int NMAT = UP ? 2 : 1;
    constexpr int STAGE = NMAT * BOX_BYTES + RAWA_BYTES;
    const int ct = threadIdx.x, warp = ct >> 5, lane = ct & 31;
    const int g = lane >> 2, t = lane & 3;
    uint64_t ya[NT][2], yb[NT][2];
#pragma unroll
    for (int n = 0; n < NT; ++n) ya[n][0] = ya[n][1] = yb[n][0] = yb[n][1] = 0;
    for (int seg = 0; seg < nseg; ++seg, ++k) {
        const int st = static_cast<int>(k % S);
        const bool got = mbar_wait_bounded(&sm.full[st], static_cast<uint32_t>((k / S) & 1), WAIT_LIMIT_NS);
        if (!tc::named_and(2, CONSUMERS * 32, got)) {
            if (ct == 0) atomicOr(p.status, CQ_DEV_WAIT_TIMEOUT);
            return false;
        }
        const uint8_t* stage = sm.wst + st * STAGE;
        convert_acts<NT>(stage + NMAT * BOX_BYTES, sm, np, ct);
        tc::named_and(1, CONSUMERS * 32, true);
        const uint8_t* wa = stage + (16 * warp + g) * (SEGB * 18);
        // Unrolled twice for gate + up (four times measured 107 -> 114 us: a
        // longer body, instruction fetch stalls) and four times for the down
        // projection (87 -> 82 us).
#pragma unroll(UP ? 2 : 4)
        for (int b = 0; b < SEGB; ++b) {
            uint32_t fa0[4], fa1[4], fb0[4], fb1[4];
            uint64_t dwa0, dwa1, dwb0 = 0, dwb1 = 0, m_unused[2];
            constexpr int RB = SEGB * 18;     // bytes per weight row in a stage
            mf::weight_frags<CQ_Q4_0>(wa + b * 18, wa + 8 * RB + b * 18, t, fa0, fa1, dwa0, dwa1, m_unused[0],
                                      m_unused[1]);
            if constexpr (UP)
                mf::weight_frags<CQ_Q4_0>(wa + BOX_BYTES + b * 18, wa + BOX_BYTES + 8 * RB + b * 18, t, fb0, fb1,
                                          dwb0, dwb1, m_unused[0], m_unused[1]);
            const uint8_t* ab = sm.act + g * ACT_PITCH + chunk_pos(b, t);
            const float4* sq = sm.sq + b * SCL_PITCH + t;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const uint4 bv = *reinterpret_cast<const uint4*>(ab + 8 * n * ACT_PITCH);
                const float4 r4 = sq[4 * n];
                const uint64_t dx = tc::pk(r4.x, r4.y);
                const float4 bias = make_float4(r4.z, r4.w, r4.z, r4.w);
                float c[4];
                mma16816c(c, fa0, bv.x, bv.y, bias);
                mma16816acc(c, fa1, bv.z, bv.w);
                ya[n][0] = tc::fma2(tc::mul2(dwa0, dx), tc::pk(c[0], c[1]), ya[n][0]);
                ya[n][1] = tc::fma2(tc::mul2(dwa1, dx), tc::pk(c[2], c[3]), ya[n][1]);
                if constexpr (UP) {
                    mma16816c(c, fb0, bv.x, bv.y, bias);
                    mma16816acc(c, fb1, bv.z, bv.w);
                    yb[n][0] = tc::fma2(tc::mul2(dwb0, dx), tc::pk(c[0], c[1]), yb[n][0]);
                    yb[n][1] = tc::fma2(tc::mul2(dwb1, dx), tc::pk(c[2], c[3]), yb[n][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm.empty[st]);
        tc::named_and(1, CONSUMERS * 32, true);     // the fp16 tile is rewritten by the next segment
    }
    if constexpr (UP) {
        // h = silu(g) * u goes to a [pair][HS_PITCH] fp32 tile in the activation
        // tile's space (free: every consumer is past the last segment's
        // barrier). Then eight lanes per (pair, 32-row block) write the slice of
        // h and its Q8_0 block -- the same rule as the activation quantiser.
        constexpr int HS_PITCH = ROWS + 4;
        static_assert(TOK * HS_PITCH * 4 <= ACT_BYTES, "h tile does not fit");
        float* hs = reinterpret_cast<float*>(sm.act);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float a[2], u[2];
                tc::upk(ya[n][h], a[0], a[1]);
                tc::upk(yb[n][h], u[0], u[1]);
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    hs[(8 * n + 2 * t + i) * HS_PITCH + 16 * warp + g + 8 * h] =
                        __fmul_rn(__fdiv_rn(a[i], __fadd_rn(1.0f, expf(-a[i]))), u[i]);
            }
        }
        tc::named_and(1, CONSUMERS * 32, true);
        const int sub = lane & 7;
        const int64_t hq_row = static_cast<int64_t>(p.rows_per_expert / 32) * 34;
        // 4 * np items, four per warp and iteration: the trip count is warp-uniform.
        for (int it = 4 * warp + (lane >> 3); it < 4 * np; it += 4 * CONSUMERS) {
            const int tk = it >> 2, j = it & 3;
            const int pr = sm.pairs[tk];
            const float4 v = *reinterpret_cast<const float4*>(hs + tk * HS_PITCH + 32 * j + 4 * sub);
            *reinterpret_cast<float4*>(p.out + static_cast<int64_t>(pr) * p.rows_per_expert + r0 + 32 * j + 4 * sub) = v;
            float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
            const float d = q8_scale(a);
            const float id = q8_inv(d);
            const uint32_t q = (static_cast<uint32_t>(quant_q8(v.x, id)) & 0xffu) |
                               ((static_cast<uint32_t>(quant_q8(v.y, id)) & 0xffu) << 8) |
                               ((static_cast<uint32_t>(quant_q8(v.z, id)) & 0xffu) << 16) |
                               (static_cast<uint32_t>(quant_q8(v.w, id)) << 24);
            uint8_t* blk = p.hq + pr * hq_row + ((r0 >> 5) + j) * 34;
            uint16_t* q16 = reinterpret_cast<uint16_t*>(blk + 2 + 4 * sub);     // 2 mod 4: 16-bit stores
            q16[0] = static_cast<uint16_t>(q);
            q16[1] = static_cast<uint16_t>(q >> 16);
            if (sub == 0) *reinterpret_cast<__half*>(blk) = __float2half_rn(d);
        }
    } else {
        // o rows r0 + 16w + g (+8), pairs 8n + 2t (+1).
        const int f = r0 + 16 * warp + g;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float a[2];
                tc::upk(ya[n][h], a[0], a[1]);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int tk = 8 * n + 2 * t + i;
                    const int pr = tk < np ? sm.pairs[tk] : -1;
                    if (pr >= 0) p.out[static_cast<int64_t>(pr) * p.rows_per_expert + f + 8 * h] = a[i];
                }
            }
        }
    }
    return true;
}

template <bool UP>
__global__ void __launch_bounds__(THREADS, 1) moe_mma_kernel(const __grid_constant__ CUtensorMap map0,
                                                             const __grid_constant__ CUtensorMap map1,
                                                             const __grid_constant__ CUtensorMap amap,
                                                             const MoeMmaParams p) {
    pdl_trigger();
    pdl_wait();
    constexpr int NMAT = UP ? 2 : 1;
    constexpr int STAGE = NMAT * BOX_BYTES + RAWA_BYTES;      // weight boxes, then the pairs' raw segments
    extern __shared__ __align__(1024) uint8_t smem[];
    const int S = p.stages;
    Smem sm;
    sm.full = reinterpret_cast<uint64_t*>(smem);
    sm.empty = sm.full + 8;
    sm.pairs = reinterpret_cast<int*>(smem + 256);
    sm.act = smem + 1024;
    sm.sq = reinterpret_cast<float4*>(sm.act + ACT_BYTES);
    sm.wst = smem + 1024 + ACT_BYTES + SCL_BYTES;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = p.order[blockIdx.y], r0 = blockIdx.x * ROWS;
    const int beg = p.offs[e], cnt = p.offs[e + 1] - beg;
    if (cnt == 0) return;
    const int nseg = p.kin / 256;
    const int passes = (cnt + TOK - 1) / TOK;
    const int64_t steps = static_cast<int64_t>(passes) * nseg;
    const int row_base = e * p.rows_per_expert + r0;                   // row in the [E * rows] tensor

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], CONSUMERS);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == CONSUMERS) {
        // ------------------------------------------------------- producer
        // Per segment: the weight boxes (2-D TMA) and the pass's pairs'
        // 272-byte activation segments, four rows per TMA gather4.
        int seg = 0, pass = 0;
        for (int64_t k = 0; k < steps; ++k) {
            const int st = static_cast<int>(k % S);
            const int np = min(TOK, cnt - pass * TOK);
            bool ok = true;
            if (lane == 0) {
                ok = mbar_wait_bounded(&sm.empty[st], static_cast<uint32_t>(((k / S) & 1) ^ 1), WAIT_LIMIT_NS);
                if (!ok) {
                    atomicOr(p.status, CQ_DEV_WAIT_TIMEOUT);
                } else {
                    mbar_arrive_expect_tx(&sm.full[st], NMAT * BOX_BYTES + (np + 3) / 4 * 4 * RAWA);
                    uint8_t* dst = sm.wst + st * STAGE;
                    tc::tma_load_2d(dst, &map0, seg * SEGB * 9, row_base, &sm.full[st]);   // 9 = 18 bytes / 2
                    if (UP) tc::tma_load_2d(dst + BOX_BYTES, &map1, seg * SEGB * 9, row_base, &sm.full[st]);
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            uint8_t* raw = sm.wst + st * STAGE + NMAT * BOX_BYTES;
            // Four pairs per gather4; a short last group repeats its last
            // pair into slots that the conversion reads as zero.
            for (int q = lane; 4 * q < np; q += 32) {
                int r[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int pr = p.perm[beg + pass * TOK + min(4 * q + j, np - 1)];
                    r[j] = UP ? pr / p.topk : pr;
                }
                tc::tma_gather4(raw + q * RAWG, &amap, seg * (RAWA / 2), r[0], r[1], r[2], r[3], &sm.full[st]);
            }
            if (++seg == nseg) { seg = 0; ++pass; }
        }
        return;   // the producer takes no part in the consumers' named barriers
    }

    // ---------------------------------------------------------- consumers
    int64_t k = 0;
    for (int pass = 0; pass < passes; ++pass) {
        const int np = min(TOK, cnt - pass * TOK);
        if (threadIdx.x < TOK) sm.pairs[threadIdx.x] = threadIdx.x < np ? p.perm[beg + pass * TOK + threadIdx.x] : -1;
        bool ok;
        switch ((np + 7) >> 3) {
            case 1: ok = run_pass<UP, 1>(p, sm, S, nseg, k, np, r0); break;
            case 2: ok = run_pass<UP, 2>(p, sm, S, nseg, k, np, r0); break;
            case 3: ok = run_pass<UP, 3>(p, sm, S, nseg, k, np, r0); break;
            case 4: ok = run_pass<UP, 4>(p, sm, S, nseg, k, np, r0); break;
            case 5: ok = run_pass<UP, 5>(p, sm, S, nseg, k, np, r0); break;
            case 6: ok = run_pass<UP, 6>(p, sm, S, nseg, k, np, r0); break;
            case 7: ok = run_pass<UP, 7>(p, sm, S, nseg, k, np, r0); break;
            default: ok = run_pass<UP, 8>(p, sm, S, nseg, k, np, r0); break;
        }
        if (!ok) break;
        tc::named_and(1, CONSUMERS * 32, true);     // pairs[] is rewritten by the next pass
    }
}

// Q4_0 weights of all experts as one 2-D tensor of 2-byte elements:
// [E * rows][kin / 32 * 18 bytes]; box = 8 blocks x 128 rows.
bool make_map(CUtensorMap* map, const void* W, int64_t rows, int kin) {
    tc::EncodeTiledFn enc = tc::encode_tiled_fn();
    if (enc == nullptr) return false;
    const int64_t rb = static_cast<int64_t>(kin / 32) * 18;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(rb / 2), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(rb)};
    const cuuint32_t box[2] = {SEGB * 9, ROWS};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(W), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q8_0 activation rows as a 2-D tensor of 2-byte elements [rows][xrow / 2];
// box = one 272-byte segment of one row (the gather4 form takes four rows).
bool make_act_map(CUtensorMap* map, const void* X, int64_t rows, int64_t xrow) {
    tc::EncodeTiledFn enc = tc::encode_tiled_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(xrow / 2), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(xrow)};
    const cuuint32_t box[2] = {RAWA / 2, 1};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(X), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool UP>
cudaError_t launch_one(const DeviceInfo& dev, const CUtensorMap& m0, const CUtensorMap& m1, const CUtensorMap& am,
                       MoeMmaParams p, int E, cudaStream_t s) {
    const int lim = std::min(dev.smem_optin, 227 * 1024);
    const int fixed = 1024 + ACT_BYTES + SCL_BYTES;
    const int per_stage = (UP ? 2 : 1) * BOX_BYTES + RAWA_BYTES;
    p.stages = std::min(8, (lim - fixed) / per_stage);
    if (p.stages < 2) return cudaErrorInvalidConfiguration;
    const int smem = fixed + p.stages * per_stage;
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(moe_mma_kernel<UP>), lim);
    if (e != cudaSuccess) return e;
    e = launch_kernel(moe_mma_kernel<UP>, dim3(p.rows_per_expert / ROWS, E), dim3(THREADS), smem, s, m0, m1, am, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_moe_projections(const DeviceInfo& dev, int T, int K, int F, int E, int topk, const void* Wg,
                                   const void* Wu, const void* Wd, const void* xq, const int* offs, const int* order,
                                   const int* perm, float* h, const void* hq, float* o, cudaStream_t s) {
    CUtensorMap mg, mu, md;
    if (!make_map(&mg, Wg, static_cast<int64_t>(E) * F, K) || !make_map(&mu, Wu, static_cast<int64_t>(E) * F, K) ||
        !make_map(&md, Wd, static_cast<int64_t>(E) * K, F))
        return cudaErrorInvalidValue;
    MoeMmaParams up{};
    up.xq = static_cast<const uint8_t*>(xq);
    up.offs = offs;
    up.order = order;
    up.perm = perm;
    up.out = h;
    up.hq = static_cast<uint8_t*>(const_cast<void*>(hq));
    up.status = dev.status;
    up.topk = topk;
    up.rows_per_expert = F;
    up.kin = K;
    up.xrow = static_cast<int64_t>(K / 32) * 34;
    CUtensorMap ax, ah;
    if (!make_act_map(&ax, xq, T, up.xrow) ||
        !make_act_map(&ah, hq, static_cast<int64_t>(T) * topk, static_cast<int64_t>(F / 32) * 34))
        return cudaErrorInvalidValue;
    cudaError_t e = launch_one<true>(dev, mg, mu, ax, up, E, s);
    if (e != cudaSuccess) return e;
    MoeMmaParams dn = up;
    dn.xq = static_cast<const uint8_t*>(hq);
    dn.out = o;
    dn.rows_per_expert = K;
    dn.kin = F;
    dn.xrow = static_cast<int64_t>(F / 32) * 34;
    return launch_one<false>(dev, md, md, ah, dn, E, s);
}

}  // namespace cq
