// Prefill GEMM of Q4_0, Q4_1 and Q8_0 weights (x Q8_0 / Q8_1 activations)
// for any number of tokens, on mma.sync, without a workspace (cq_gemm; with a
// workspace, cq_gemm_ws runs the tensor-memory kernel of gemm_tc32.cu).
//
// cera README "Supported models": prompts are prefilled by a batched GEMM;
// cera 0.5.3 README "Breaking changes in 0.4.0": the batched and the
// per-token paths give the same bits. Each row here follows the library's
// fixed fp32 order (include/cq.h) -- c = fma(d_w * d_x, isum, c)
// [+ fma(m_w, s_x, c)] over four blocks, y = y + c per chunk -- in one
// thread per (row, token), so it equals the cq_gemv row bit for bit.
//
// One CTA = 128 weight rows x 64 tokens. Per 8-block segment a producer warp
// TMA-loads the weight box (128 rows x 8 blocks, raw GGUF bytes) and the
// tokens' raw activation blocks (64 rows x 8 blocks) into one stage of a
// ring. The consumer warps convert the activations into the CTA's B-operand
// image (fp16 fragments + a scale table); then each of the 8 takes 16 weight
// rows: per block the integer dot is an
// exact fp16 mma.sync m16n8k16 product (see mma_frag.cuh) and the scale terms
// run two tokens per f32x2 instruction. The grid walks the token tiles of one
// row tile next to each other, so a weight tile is read from DRAM once and
// from L2 by the other token tiles.
#include <algorithm>

#include <cuda_fp16.h>

#include "cq_device.cuh"
#include "cq_internal.h"
#include "mma_frag.cuh"
#include "tc.cuh"

namespace cq {
namespace {

using mf::MF;

constexpr int ROWS = 128;
constexpr int SEGB = 8;                  // 32-blocks per segment
constexpr int TOK = 64;                  // tokens per CTA (8 n-tiles)
constexpr int NT = TOK / 8;
constexpr int CONSUMERS = 8;
constexpr int THREADS = (CONSUMERS + 1) * 32;
constexpr int MAX_STAGES = 8;
// B-operand image of 64 tokens x one segment, in shared memory:
//   fp16 quants, 512 bytes per token: chunk c (16 bytes, lane t = c's B
//     fragments of both k-steps, see act_frags) of block b of token tk at
//     img_pos(tk, b, c);
//   scale table per (block b, token pair j), SCL_PITCH pairs per block:
//     {d_x, d_x', bias, bias'} as one float4 (bias = -BIAS * sum of the
//     quants) and, for Q8_1, {s_x, s_x'}.
constexpr int ACT_BYTES = TOK * SEGB * 64;            // 32768
constexpr int SCL_PITCH = TOK / 2 + 1;                // +1: converters' stores spread over banks
constexpr int SC4_BYTES = SEGB * SCL_PITCH * 16;      // 4224
constexpr int SX_BYTES = SEGB * SCL_PITCH * 8;        // 2112
__host__ __device__ constexpr int img_bytes(bool q8_1) {
    return (ACT_BYTES + SC4_BYTES + (q8_1 ? SX_BYTES : 0) + 127) / 128 * 128;
}
__host__ __device__ constexpr int wbox_bytes(int bb) { return ROWS * mf::stage_pitch(bb); }
__host__ __device__ constexpr int abox_bytes(int abb) { return TOK * SEGB * abb; }
// Shared memory ahead of the stages: barriers and the CTA's image of the
// current segment.
__host__ __device__ constexpr int fixed_bytes(bool q8_1) { return 1024 + img_bytes(q8_1); }

struct GemmMmaParams {
    float* y;
    int* status;
    int M, N;
    int nseg;               // 8-block segments per row
    int stages;
};

// Byte position of chunk c of block b of token tk in an image. Blocks swap
// places within a pair for odd tokens, so tokens g and g+1 (one 8-lane
// shared-memory phase of a fragment load) fall in different halves of the
// 128-byte bank window; chunks are XOR-rotated by block pair, so eight
// converters writing chunk c of blocks 0..7 hit eight different bank groups.
__host__ __device__ constexpr int img_pos(int tk, int b, int c) {
    return tk * (SEGB * 64) + 64 * (b ^ (tk & 1)) + 16 * (c ^ ((b >> 1) & 3));
}

// Converts one activation block (token tk of the tile, block b of the
// segment) into the image at img.
template <int WF>
__device__ __forceinline__ void put_block(uint8_t* img, const uint8_t* blk, int tk, int b) {
    using F = MF<WF>;
    uint4 ch[4];
    float d, s;
    int sum;
    mf::act_frags<WF>(blk, ch, d, s, sum);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) *reinterpret_cast<uint4*>(img + img_pos(tk, b, cc)) = ch[cc];
    float* sc4f = reinterpret_cast<float*>(img + ACT_BYTES);
    float* sx2f = reinterpret_cast<float*>(img + ACT_BYTES + SC4_BYTES);
    const int j = b * SCL_PITCH + (tk >> 1), hi = tk & 1;
    sc4f[4 * j + hi] = d;
    sc4f[4 * j + 2 + hi] = static_cast<float>(-F::BIAS * sum);
    if constexpr (WF == CQ_Q4_1) sx2f[2 * j + hi] = s;
}

template <int WF>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_mma_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap amap,
                    const GemmMmaParams p) {
    pdl_trigger();
    pdl_wait();
    using F = MF<WF>;
    constexpr int WBOX = wbox_bytes(F::BB);
    constexpr int STAGE = WBOX + abox_bytes(F::ABB);
    constexpr int PITCH = mf::stage_pitch(F::BB);
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + MAX_STAGES;
    uint8_t* img = smem + 1024;
    uint8_t* wst = smem + fixed_bytes(WF == CQ_Q4_1);
    const int S = p.stages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tok0 = blockIdx.x * TOK, r0 = blockIdx.y * ROWS;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], CONSUMERS);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == CONSUMERS) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            for (int k = 0; k < p.nseg; ++k) {
                const int st = k % S;
                if (!mbar_wait_bounded(&empty[st], static_cast<uint32_t>(((k / S) & 1) ^ 1), WAIT_LIMIT_NS)) {
                    atomicOr(p.status, CQ_DEV_WAIT_TIMEOUT);
                    break;
                }
                uint8_t* dst = wst + st * STAGE;
                mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(STAGE));
                // x counts 2-byte elements; rows past N / tokens past M read as zero
                tc::tma_load_2d(dst, &wmap, k * SEGB * F::BB / 2, r0, &full[st]);
                tc::tma_load_2d(dst + WBOX, &amap, k * SEGB * F::ABB / 2, tok0, &full[st]);
            }
        }
        return;   // the producer takes no part in the consumers' named barriers
    }

    // ---------------------------------------------------------- consumers
    const int ct = threadIdx.x, g = lane >> 2, t = lane & 3;
    uint64_t c[NT][2], y[NT][2];   // (row g | row g+8) x (token 8n+2t, 8n+2t+1)
#pragma unroll
    for (int n = 0; n < NT; ++n) y[n][0] = y[n][1] = 0;
    bool ok = true;
    for (int k = 0; k < p.nseg; ++k) {
        const int st = k % S;
        const bool got = mbar_wait_bounded(&full[st], static_cast<uint32_t>((k / S) & 1), WAIT_LIMIT_NS);
        if (!tc::named_and(2, CONSUMERS * 32, got)) {
            if (ct == 0) atomicOr(p.status, CQ_DEV_WAIT_TIMEOUT);
            ok = false;
            break;
        }
        const uint8_t* stage = wst + st * STAGE;
        // The tokens' blocks of this segment as the CTA's image (tokens past M
        // arrive as zero blocks).
        for (int it = ct; it < TOK * SEGB; it += CONSUMERS * 32)
            put_block<WF>(img, stage + WBOX + it * F::ABB, it >> 3, it & 7);
        tc::named_and(1, CONSUMERS * 32, true);
        const float4* sc4 = reinterpret_cast<const float4*>(img + ACT_BYTES);
        const float2* sx2 = reinterpret_cast<const float2*>(img + ACT_BYTES + SC4_BYTES);
        const uint8_t* rg = stage + (16 * warp + g) * PITCH;
        const uint8_t* rg8 = rg + 8 * PITCH;
#pragma unroll 1
        for (int bi = 0; bi < SEGB; ++bi) {
            uint32_t a0[4], a1[4];
            uint64_t dw0, dw1, mw0, mw1;
            mf::weight_frags<WF>(rg + bi * F::BB, rg8 + bi * F::BB, t, a0, a1, dw0, dw1, mw0, mw1);
            if ((bi & 3) == 0) {
#pragma unroll
                for (int n = 0; n < NT; ++n) c[n][0] = c[n][1] = 0;
            }
            const uint8_t* ab = img + img_pos(g, bi, t);
            const float4* s4p = sc4 + bi * SCL_PITCH + t;
            const float2* sxp = sx2 + bi * SCL_PITCH + t;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const uint4 bv = *reinterpret_cast<const uint4*>(ab + 8 * n * (SEGB * 64));
                const float4 s4 = s4p[4 * n];
                float acc[4];
                mf::mma16816c(acc, a0, bv.x, bv.y, s4.z, s4.w);
                mf::mma16816acc(acc, a1, bv.z, bv.w);
                const uint64_t dx = tc::pk(s4.x, s4.y);
                // c = fma(d_w * d_x, isum, c) per element, two tokens per instruction
                c[n][0] = tc::fma2(tc::mul2(dw0, dx), tc::pk(acc[0], acc[1]), c[n][0]);
                c[n][1] = tc::fma2(tc::mul2(dw1, dx), tc::pk(acc[2], acc[3]), c[n][1]);
                if constexpr (WF == CQ_Q4_1) {
                    const float2 s2 = sxp[4 * n];
                    const uint64_t sx = tc::pk(s2.x, s2.y);
                    c[n][0] = tc::fma2(mw0, sx, c[n][0]);
                    c[n][1] = tc::fma2(mw1, sx, c[n][1]);
                }
            }
            if ((bi & 3) == 3) {
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    y[n][0] = tc::add2(y[n][0], c[n][0]);
                    y[n][1] = tc::add2(y[n][1], c[n][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[st]);
        tc::named_and(1, CONSUMERS * 32, true);     // the image is rewritten by the next segment
    }
    if (ok) {
        // y[token][row]: rows r0 + 16w + g (+8), tokens tok0 + 8n + 2t (+1)
        const int row0 = r0 + 16 * warp + g;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int m0 = tok0 + 8 * n + 2 * t;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v[2];
                tc::upk(y[n][h], v[0], v[1]);
                const int row = row0 + 8 * h;
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    if (row < p.N && m0 + i < p.M) p.y[static_cast<int64_t>(m0 + i) * p.N + row] = v[i];
            }
        }
    }
    // Let the producer's copies in flight land before the CTA's shared memory goes.
    if (ct == 0) {
        for (int k = p.nseg > S ? p.nseg - S : 0; k < p.nseg; ++k)
            (void)mbar_wait_bounded(&full[k % S], static_cast<uint32_t>((k / S) & 1), WAIT_LIMIT_NS / 8);
    }
}

template <int WF>
cudaError_t launch_fmt(const DeviceInfo& dev, int64_t M, int64_t N, int64_t K, const void* W, const void* xq,
                       float* y, cudaStream_t s) {
    using F = MF<WF>;
    tc::EncodeTiledFn enc = tc::encode_tiled_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    const int nb = static_cast<int>(K / 32);
    const int64_t wrow = static_cast<int64_t>(nb) * F::BB, xrow = static_cast<int64_t>(nb) * F::ABB;
    // Weights [N rows][wrow / 2] and activations [M rows][xrow / 2] as 2-D
    // tensors of 2-byte elements; boxes of 8 blocks x 128 rows / 64 tokens.
    CUtensorMap wmap, amap;
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(wrow / 2), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(wrow)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(mf::stage_pitch(F::BB) / 2), ROWS};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(W), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(xrow / 2), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(xrow)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(SEGB * F::ABB / 2), TOK};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&amap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(xq), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    constexpr int STAGE = wbox_bytes(F::BB) + abox_bytes(F::ABB);
    constexpr int FIXED = fixed_bytes(WF == CQ_Q4_1);
    const int lim = std::min(dev.smem_optin, 227 * 1024);
    GemmMmaParams p{};
    p.y = y;
    p.status = dev.status;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.nseg = nb / SEGB;
    p.stages = std::min(MAX_STAGES, (lim - FIXED) / STAGE);
    if (p.stages < 2) return cudaErrorInvalidConfiguration;
    const int smem = FIXED + p.stages * STAGE;
    static int raised[64] = {};
    int devid = 0;
    cudaError_t e = cudaGetDevice(&devid);
    if (e != cudaSuccess) return e;
    if (devid >= 64 || raised[devid] < smem) {
        e = cudaFuncSetAttribute(gemm_mma_kernel<WF>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (devid < 64) raised[devid] = smem;
    }
    const int64_t row_tiles = (N + ROWS - 1) / ROWS;
    if (row_tiles > 65535) return cudaErrorInvalidValue;      // grid y limit (N above 8.4 M rows)
    return launch_kernel(gemm_mma_kernel<WF>, dim3(static_cast<unsigned>((M + TOK - 1) / TOK),
                                                   static_cast<unsigned>(row_tiles)),
                         dim3(THREADS), smem, s, wmap, amap, p);
}

}  // namespace

cudaError_t launch_gemm_mma(const DeviceInfo& dev, int w_fmt, int64_t M, int64_t N, int64_t K, const void* W,
                            const void* xq, float* y, cudaStream_t s) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    switch (w_fmt) {
    case CQ_Q4_0: return launch_fmt<CQ_Q4_0>(dev, M, N, K, W, xq, y, s);
    case CQ_Q4_1: return launch_fmt<CQ_Q4_1>(dev, M, N, K, W, xq, y, s);
    case CQ_Q8_0: return launch_fmt<CQ_Q8_0>(dev, M, N, K, W, xq, y, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace cq
