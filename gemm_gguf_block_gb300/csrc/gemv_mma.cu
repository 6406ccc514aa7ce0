// Batched GEMV for 2 <= M <= 16 tokens on the tensor cores (Q4_0, Q4_1, Q8_0).
//
// cera README "Other features" and 0.5 release notes: the speculative-decoding
// verify path projects all 1 + k positions through the LM head in one batched
// pass, so the head is read once per round; alice-llm "Batch-4 Speculative
// Decoding": weights decoded once, one accumulator set per position, and the
// batched result equal to the single-position one.
//
// Per 32-element block the integer dot is an exact fp16 tensor-core product
// (quants are small integers, exact in fp16; 32 products sum far below 2^24
// in the fp32 accumulator), mma.sync m16n8k16 twice per block. The block's
// scale terms are then applied on the CUDA cores in the library's fixed
// order (include/cq.h): c = fma(d_w * d_x, isum, c) [+ fma(m_w, s_x, c) for
// Q4_1] over four blocks, y = y + c per chunk. Every (row, token) chain lives
// in one thread, so each row equals the single-token GEMV row bit for bit.
//
// A persistent CTA (8 consumer warps of 16 rows each + 1 producer warp)
// stages the tokens' activations once as fp16 in shared memory, then streams
// 128-row weight tiles through a ring of 2-D TMA boxes (128 rows x 8 blocks).
#include <algorithm>
#include <mutex>

#include <cuda_fp16.h>

#include "cq_device.cuh"
#include "cq_internal.h"
#include "tc.cuh"

namespace cq {
namespace {

constexpr int ROWS = 128;           // rows per tile
constexpr int SEG_BLOCKS = 8;       // 32-blocks per stage (256 elements)
constexpr int NSTAGE = 4;
constexpr int CONSUMERS = 8;        // warps, 16 rows each
constexpr int THREADS = (CONSUMERS + 1) * 32;

template <int WF> struct MF;
template <> struct MF<CQ_Q4_0> { static constexpr int BB = 18, QO = 2, ABB = 34, AQO = 2; };
template <> struct MF<CQ_Q4_1> { static constexpr int BB = 20, QO = 4, ABB = 36, AQO = 4; };
template <> struct MF<CQ_Q8_0> { static constexpr int BB = 34, QO = 2, ABB = 34, AQO = 2; };

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
    int smem_act;       // offset of the staged activations
    int smem_scale;     // offset of the staged activation scales (float2 per token-block)
    int smem_stage;     // offset of the weight stages
};

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f), "f"(0.0f), "f"(0.0f),
          "f"(0.0f));
}

// Two bytes (quants of elements k, k+1) as a half2 of their integer values.
// Q4: the low (hi=false) or high nibbles, minus `off` (8 for Q4_0, 0 for Q4_1);
// Q8: the signed bytes.
template <int WF>
__device__ __forceinline__ uint32_t pair_to_half2(uint32_t two_bytes, bool hi) {
    const uint32_t p = __byte_perm(two_bytes, 0u, 0x4140);     // byte 0 -> half 0, byte 1 -> half 1
    if constexpr (WF == CQ_Q8_0) {
        return h2u(__hsub2(u2h((p ^ 0x00800080u) | 0x64006400u), u2h(0x64806480u)));   // - 1152
    } else {
        const uint32_t n = (hi ? (p >> 4) : p) & 0x000F000Fu;
        const uint32_t bias = WF == CQ_Q4_0 ? 0x64086408u : 0x64006400u;                // 1032 or 1024
        return h2u(__hsub2(u2h(n | 0x64006400u), u2h(bias)));
    }
}

template <int WF, int NT>
__global__ void __launch_bounds__(THREADS, 1) gemv_mma_kernel(const __grid_constant__ CUtensorMap wmap,
                                                              const MmaParams p) {
    using F = MF<WF>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + NSTAGE;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = (p.N + ROWS - 1) / ROWS;
    const int nseg = p.nb / SEG_BLOCKS;
    const int my_tiles = blockIdx.x < tiles ? (tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t steps = static_cast<int64_t>(my_tiles) * nseg;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], CONSUMERS);
        }
        fence_mbar_init();
    }
    // Stage the activations once: fp16 quants [token][k] (padded pitch) and
    // per-block scales (d, s) as floats; tokens >= M are zero.
    {
        __half* act = reinterpret_cast<__half*>(smem + p.smem_act);
        float2* sc = reinterpret_cast<float2*>(smem + p.smem_scale);
        const int tokens = NT * 8;
        const int total = tokens * p.nb;
        for (int i = threadIdx.x; i < total; i += blockDim.x) {
            const int m = i / p.nb, b = i - m * p.nb;
            uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            float2 ds = make_float2(0.0f, 0.0f);
            if (m < p.M) {
                const uint16_t* s = reinterpret_cast<const uint16_t*>(p.xq + (static_cast<int64_t>(m) * p.nb + b) * F::ABB);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    w[j] = static_cast<uint32_t>(s[F::AQO / 2 + 2 * j]) | (static_cast<uint32_t>(s[F::AQO / 2 + 2 * j + 1]) << 16);
                ds.x = h2f(s[0]);
                ds.y = WF == CQ_Q4_1 ? h2f(s[1]) : 0.0f;
            }
            uint32_t* dst = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(act) + m * p.act_pitch + 64 * b);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t o0 = h2u(__hsub2(u2h((__byte_perm(w[j], 0u, 0x4140) ^ 0x00800080u) | 0x64006400u), u2h(0x64806480u)));
                uint32_t o1 = h2u(__hsub2(u2h((__byte_perm(w[j], 0u, 0x4342) ^ 0x00800080u) | 0x64006400u), u2h(0x64806480u)));
                dst[2 * j] = o0;
                dst[2 * j + 1] = o1;
            }
            sc[m * p.nb + b] = ds;
        }
    }
    __syncthreads();

    if (warp == CONSUMERS) {
        // -------------------------------------------------------- producer
        if (lane == 0) {
            for (int64_t k = 0; k < steps; ++k) {
                const int st = static_cast<int>(k % NSTAGE);
                if (!mbar_wait_bounded(&empty[st], static_cast<uint32_t>(((k / NSTAGE) & 1) ^ 1), WAIT_LIMIT_NS)) {
                    atomicOr(p.status, CQ_DEV_WAIT_TIMEOUT);
                    break;
                }
                const int tile = blockIdx.x + static_cast<int>(k / nseg) * gridDim.x;
                const int seg = static_cast<int>(k % nseg);
                mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(p.stage_bytes));
                // x counts 2-byte elements of the row
                tc::tma_load_2d(smem + p.smem_stage + st * p.stage_bytes, &wmap, seg * SEG_BLOCKS * F::BB / 2,
                                tile * ROWS, &full[st]);
            }
        }
    } else {
        // -------------------------------------------------------- consumers
        const int g = lane >> 2, t = lane & 3;
        const uint8_t* act = smem + p.smem_act;
        const float2* sc = reinterpret_cast<const float2*>(smem + p.smem_scale);
        const int seg_row_bytes = SEG_BLOCKS * F::BB;
        float c[NT][4], y[NT][4];
        int64_t k = 0;
        bool ok = true;
        for (int ti = 0; ti < my_tiles && ok; ++ti) {
            const int tile = blockIdx.x + ti * gridDim.x;
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) y[n][e] = 0.0f;
            for (int seg = 0; seg < nseg; ++seg, ++k) {
                const int st = static_cast<int>(k % NSTAGE);
                if (!mbar_wait_bounded(&full[st], static_cast<uint32_t>((k / NSTAGE) & 1), WAIT_LIMIT_NS)) {
                    if (lane == 0) atomicOr(p.status, CQ_DEV_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                const uint8_t* rg = smem + p.smem_stage + st * p.stage_bytes + (16 * warp + g) * seg_row_bytes;
                const uint8_t* rg8 = rg + 8 * seg_row_bytes;
#pragma unroll 2
                for (int bi = 0; bi < SEG_BLOCKS; ++bi) {
                    const int b = seg * SEG_BLOCKS + bi;          // block index along K
                    const uint8_t* w0 = rg + bi * F::BB;
                    const uint8_t* w1 = rg8 + bi * F::BB;
                    // A fragments: k-step 0 = elements 0..15, k-step 1 = 16..31.
                    uint32_t a0[4], a1[4];
                    if constexpr (WF == CQ_Q8_0) {
                        const uint16_t* q0 = reinterpret_cast<const uint16_t*>(w0 + F::QO);
                        const uint16_t* q1 = reinterpret_cast<const uint16_t*>(w1 + F::QO);
                        a0[0] = pair_to_half2<WF>(q0[t], false);
                        a0[1] = pair_to_half2<WF>(q1[t], false);
                        a0[2] = pair_to_half2<WF>(q0[t + 4], false);
                        a0[3] = pair_to_half2<WF>(q1[t + 4], false);
                        a1[0] = pair_to_half2<WF>(q0[t + 8], false);
                        a1[1] = pair_to_half2<WF>(q1[t + 8], false);
                        a1[2] = pair_to_half2<WF>(q0[t + 12], false);
                        a1[3] = pair_to_half2<WF>(q1[t + 12], false);
                    } else {
                        const uint16_t* q0 = reinterpret_cast<const uint16_t*>(w0 + F::QO);
                        const uint16_t* q1 = reinterpret_cast<const uint16_t*>(w1 + F::QO);
                        const uint32_t r0a = q0[t], r0b = q0[t + 4], r1a = q1[t], r1b = q1[t + 4];
                        a0[0] = pair_to_half2<WF>(r0a, false);
                        a0[1] = pair_to_half2<WF>(r1a, false);
                        a0[2] = pair_to_half2<WF>(r0b, false);
                        a0[3] = pair_to_half2<WF>(r1b, false);
                        a1[0] = pair_to_half2<WF>(r0a, true);
                        a1[1] = pair_to_half2<WF>(r1a, true);
                        a1[2] = pair_to_half2<WF>(r0b, true);
                        a1[3] = pair_to_half2<WF>(r1b, true);
                    }
                    const float dw0 = h2f(*reinterpret_cast<const uint16_t*>(w0));
                    const float dw1 = h2f(*reinterpret_cast<const uint16_t*>(w1));
                    float mw0 = 0.0f, mw1 = 0.0f;
                    if constexpr (WF == CQ_Q4_1) {
                        mw0 = h2f(*reinterpret_cast<const uint16_t*>(w0 + 2));
                        mw1 = h2f(*reinterpret_cast<const uint16_t*>(w1 + 2));
                    }
                    if ((b & 3) == 0) {
#pragma unroll
                        for (int n = 0; n < NT; ++n)
#pragma unroll
                            for (int e = 0; e < 4; ++e) c[n][e] = 0.0f;
                    }
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const uint8_t* tok = act + (8 * n + g) * p.act_pitch + 64 * b + 4 * t;
                        float acc0[4], acc1[4];
                        mma16816(acc0, a0, *reinterpret_cast<const uint32_t*>(tok),
                                 *reinterpret_cast<const uint32_t*>(tok + 16));
                        mma16816(acc1, a1, *reinterpret_cast<const uint32_t*>(tok + 32),
                                 *reinterpret_cast<const uint32_t*>(tok + 48));
                        // C fragment: e=0 (row g, token 2t), e=1 (row g, 2t+1),
                        // e=2 (row g+8, 2t), e=3 (row g+8, 2t+1). The two k-steps'
                        // exact integer partials add exactly.
                        const float2 s0 = sc[(8 * n + 2 * t) * p.nb + b];
                        const float2 s1 = sc[(8 * n + 2 * t + 1) * p.nb + b];
                        const float is0 = acc0[0] + acc1[0], is1 = acc0[1] + acc1[1];
                        const float is2 = acc0[2] + acc1[2], is3 = acc0[3] + acc1[3];
                        c[n][0] = __fmaf_rn(__fmul_rn(dw0, s0.x), is0, c[n][0]);
                        c[n][1] = __fmaf_rn(__fmul_rn(dw0, s1.x), is1, c[n][1]);
                        c[n][2] = __fmaf_rn(__fmul_rn(dw1, s0.x), is2, c[n][2]);
                        c[n][3] = __fmaf_rn(__fmul_rn(dw1, s1.x), is3, c[n][3]);
                        if constexpr (WF == CQ_Q4_1) {
                            c[n][0] = __fmaf_rn(mw0, s0.y, c[n][0]);
                            c[n][1] = __fmaf_rn(mw0, s1.y, c[n][1]);
                            c[n][2] = __fmaf_rn(mw1, s0.y, c[n][2]);
                            c[n][3] = __fmaf_rn(mw1, s1.y, c[n][3]);
                        }
                    }
                    if ((b & 3) == 3) {
#pragma unroll
                        for (int n = 0; n < NT; ++n)
#pragma unroll
                            for (int e = 0; e < 4; ++e) y[n][e] = __fadd_rn(y[n][e], c[n][e]);
                    }
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&empty[st]);
            }
            if (!ok) break;
            // y[token][row]: rows 16w+g and 16w+g+8, tokens 8n+2t, 8n+2t+1
            const int r0 = tile * ROWS + 16 * warp + g;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int m0 = 8 * n + 2 * t;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = r0 + (e >= 2 ? 8 : 0), m = m0 + (e & 1);
                    if (row < p.N && m < p.M) p.y[static_cast<int64_t>(m) * p.N + row] = y[n][e];
                }
            }
        }
    }
    // Let the producer's last copies land before the CTA's shared memory goes.
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int64_t k = steps > NSTAGE ? steps - NSTAGE : 0; k < steps; ++k)
            (void)mbar_wait_bounded(&full[k % NSTAGE], static_cast<uint32_t>((k / NSTAGE) & 1), WAIT_LIMIT_NS / 8);
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* q = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) ==
                cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(q);
    });
    return fn;
}

template <int WF, int NT>
cudaError_t launch_mma_typed(const DeviceInfo& dev, MmaParams p, const CUtensorMap& map, cudaStream_t s) {
    const int smem = p.smem_stage + NSTAGE * p.stage_bytes;
    static int raised[64] = {};
    int devid = 0;
    cudaError_t e = cudaGetDevice(&devid);
    if (e != cudaSuccess) return e;
    if (devid >= 64 || raised[devid] < smem) {
        e = cudaFuncSetAttribute(gemv_mma_kernel<WF, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 std::min(dev.smem_optin, 227 * 1024));
        if (e != cudaSuccess) return e;
        if (devid < 64) raised[devid] = std::min(dev.smem_optin, 227 * 1024);
    }
    const int tiles = (p.N + ROWS - 1) / ROWS;
    const int grid = std::min(tiles, dev.sm_count);
    gemv_mma_kernel<WF, NT><<<grid, THREADS, smem, s>>>(map, p);
    return cudaGetLastError();
}

template <int WF>
cudaError_t launch_mma_fmt(const DeviceInfo& dev, int M, int64_t N, int64_t K, const void* W, const void* xq,
                           float* y, cudaStream_t s) {
    using F = MF<WF>;
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
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
    p.act_pitch = static_cast<int>(K) * 2 + 16;       // +16 bytes: tokens land on different banks
    p.stage_bytes = ROWS * SEG_BLOCKS * F::BB;
    p.smem_act = 1024;
    p.smem_scale = p.smem_act + (NT * 8 * p.act_pitch + 127) / 128 * 128;
    p.smem_stage = p.smem_scale + (NT * 8 * p.nb * 8 + 1023) / 1024 * 1024;
    // Raw weights as a 2-D tensor of 2-byte elements [N rows][wrow/2]; a box is
    // 8 blocks of 128 rows.
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.wrow / 2), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.wrow)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(SEG_BLOCKS * F::BB / 2), ROWS};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(W), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return NT == 1 ? launch_mma_typed<WF, 1>(dev, p, map, s) : launch_mma_typed<WF, 2>(dev, p, map, s);
}

}  // namespace

// Shared memory the tensor-core GEMV needs for M tokens and K columns (0 when
// the format has no tensor-core path).
int gemv_mma_smem(int w_fmt, int M, int64_t K) {
    if (w_fmt != CQ_Q4_0 && w_fmt != CQ_Q4_1 && w_fmt != CQ_Q8_0) return 0;
    const int bb = w_fmt == CQ_Q4_0 ? 18 : w_fmt == CQ_Q4_1 ? 20 : 34;
    const int NT = M <= 8 ? 1 : 2;
    const int nb = static_cast<int>(K / 32);
    const int act = (NT * 8 * (static_cast<int>(K) * 2 + 16) + 127) / 128 * 128;
    const int scale = (NT * 8 * nb * 8 + 1023) / 1024 * 1024;
    return 1024 + act + scale + NSTAGE * ROWS * SEG_BLOCKS * bb;
}

cudaError_t launch_gemv_mma(const DeviceInfo& dev, int w_fmt, int M, int64_t N, int64_t K, const void* W,
                            const void* xq, float* y, cudaStream_t s) {
    switch (w_fmt) {
    case CQ_Q4_0: return launch_mma_fmt<CQ_Q4_0>(dev, M, N, K, W, xq, y, s);
    case CQ_Q4_1: return launch_mma_fmt<CQ_Q4_1>(dev, M, N, K, W, xq, y, s);
    case CQ_Q8_0: return launch_mma_fmt<CQ_Q8_0>(dev, M, N, K, W, xq, y, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace cq
