// Decode GEMV / batched LM-head projection, 1 <= M <= 16 tokens.
//
// cera README "Quantization": integer GEMV over quantized weights with
// activations quantized to 8 bits; alice-llm "The GPU Optimization Journey"
// phases 1.5-2 (fused dequant-matvec, register reductions) and "Batch-4
// Speculative Decoding" (weights decoded once, one accumulator per token);
// cera README "Other features" (the LM head projected for all verified
// positions in one pass).
//
// Layout of the work. A row of K elements is nc = K/256 chunks (eight
// 32-blocks, or one Q4_K superblock). A warp owns "items": R consecutive rows
// (R = 32/nc when a row has fewer than 32 chunks) or, for very long rows, one
// row segment of up to SEGC chunks. An item is contiguous in memory, so one
// bulk copy (cp.async.bulk, the one-dimensional TMA engine) moves it into a
// per-warp ring of shared-memory stages; the copy for item i+S is issued as
// soon as item i has been read, so each warp keeps up to S items in flight.
// Each lane takes whole chunks of the item (task t -> row t/segc, chunk
// t%segc), unpacks nibbles in registers and forms exact int32 block dots with
// dp4a against the activations, which the CTA stages once in shared memory
// (chunk pitch padded to an odd number of 16-byte units so that the lanes'
// 128-bit loads do not collide on banks). The per-chunk fp32 values go to a
// small per-warp buffer; lane (r, m) then adds them in increasing k, which is
// the library's fixed evaluation order (see include/cq.h).
#include <algorithm>

#include "chunk_dot.cuh"
#include "cq_device.cuh"
#include "cq_internal.h"

namespace cq {
namespace {

constexpr int WPC_MAX = 16;            // warps per CTA (upper bound)
constexpr int SEGC_MAX = 64;           // chunks per segment of a long row

struct GemvParams {
    const uint8_t* W;
    const uint8_t* xq;
    float* y;
    int* status;
    int64_t N;
    int64_t row_bytes;
    int M;
    int nc;            // chunks per row
    int R;             // rows per item
    int segc;          // chunks per item segment
    int nseg;          // segments per row (R == 1 whenever nseg > 1)
    int stages;
    int stage_bytes;   // bytes reserved per stage (multiple of 128)
    int warp_bytes;    // bytes per warp region
    int act_bytes;     // bytes of the staged activations (multiple of 128)
    int tok_pitch;     // bytes between tokens in the staged activations
};

// ------------------------------------------------------------------ kernel
template <int MT> constexpr int wpc_limit() { return MT <= 4 ? WPC_MAX : WPC_MAX / 2; }

template <int WF, int MT>
__global__ void __launch_bounds__(wpc_limit<MT>() * 32) gemv_kernel(const GemvParams p) {
    using F = Fmt<WF>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wpc = blockDim.x >> 5;

    // Stage this call's activations once per CTA: token m, chunk j at
    // m * tok_pitch + j * ACP (the chunk bytes, then padding).
    {
        const int nc = p.nc;
        const int words_per_chunk = F::ACH / 4;
        const int total = p.M * nc * words_per_chunk;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(p.xq);
        for (int i = threadIdx.x; i < total; i += blockDim.x) {
            const int m = i / (nc * words_per_chunk);
            const int r = i - m * nc * words_per_chunk;
            const int j = r / words_per_chunk, w = r - j * words_per_chunk;
            *reinterpret_cast<uint32_t*>(smem + m * p.tok_pitch + j * F::ACP + 4 * w) =
                src[(static_cast<int64_t>(m) * nc + j) * words_per_chunk + w];
        }
    }
    __syncthreads();

    const int64_t groups = (p.N + p.R - 1) / p.R;
    const int64_t wtot = static_cast<int64_t>(gridDim.x) * wpc;
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * wpc + warp;
    if (wid >= groups) return;
    const int64_t nsteps = ((groups - 1 - wid) / wtot + 1) * p.nseg;

    uint8_t* region = smem + p.act_bytes + warp * p.warp_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(region);
    uint8_t* stages = region + 128;
    float* cbuf = reinterpret_cast<float*>(stages + p.stages * p.stage_bytes);
    const int S = p.stages;

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t policy = policy_evict_first();

    // Issue the copy of step k into stage k % S (lane 0 only).
    auto issue = [&](int64_t k) {
        const int64_t g = wid + (k / p.nseg) * wtot;
        const int seg = static_cast<int>(k % p.nseg);
        const int64_t row0 = g * p.R;
        uint32_t bytes;
        const uint8_t* src;
        if (p.nseg == 1) {
            const int64_t rows = min(static_cast<int64_t>(p.R), p.N - row0);
            bytes = static_cast<uint32_t>(rows * p.row_bytes);
            src = p.W + row0 * p.row_bytes;
        } else {
            const int c0 = seg * p.segc;
            const int cn = min(p.segc, p.nc - c0);
            bytes = static_cast<uint32_t>(cn * F::CH);
            src = p.W + row0 * p.row_bytes + static_cast<int64_t>(c0) * F::CH;
        }
        uint64_t* bar = &bars[k % S];
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(stages + (k % S) * p.stage_bytes, src, bytes, bar, policy);
    };

    if (lane == 0)
        for (int64_t k = 0; k < min(static_cast<int64_t>(S), nsteps); ++k) issue(k);

    float ycarry = 0.0f;
    bool failed = false;
    int64_t kfail = 0;
    for (int64_t k = 0; k < nsteps; ++k) {
        const int s = static_cast<int>(k % S);
        const uint32_t parity = static_cast<uint32_t>((k / S) & 1);
        const bool ok = mbar_wait_bounded(&bars[s], parity, WAIT_LIMIT_NS);
        if (!__all_sync(0xffffffffu, ok)) { failed = true; kfail = k; break; }

        const int64_t g = wid + (k / p.nseg) * wtot;
        const int seg = static_cast<int>(k % p.nseg);
        const int64_t row0 = g * p.R;
        const int c0 = seg * p.segc;
        const int cn = min(p.segc, p.nc - c0);
        const int rows_valid = static_cast<int>(min(static_cast<int64_t>(p.R), p.N - row0));
        const int ntasks = p.R * cn;
        const uint8_t* st = stages + s * p.stage_bytes;
        for (int t = lane; t < ntasks; t += 32) {
            const int r = t / cn, j = t - r * cn;
            if (r < rows_valid) {
                float c[MT];
                chunk_dot<WF, MT>(st + r * static_cast<int>(p.row_bytes) * (p.nseg == 1) + j * F::CH,
                                  smem + (c0 + j) * F::ACP, p.tok_pitch, p.M, c);
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    if (m < p.M) cbuf[m * ntasks + t] = c[m];
            }
        }
        __syncwarp();
        if (lane == 0 && k + S < nsteps) issue(k + S);
        // Fixed order: y = y + c over the chunks in increasing k.
        for (int q = lane; q < p.R * p.M; q += 32) {
            const int r = q / p.M, m = q - r * p.M;
            float acc = seg == 0 ? 0.0f : ycarry;
            const float* cb = cbuf + m * ntasks + r * cn;
            for (int j = 0; j < cn; ++j) acc = __fadd_rn(acc, cb[j]);
            if (seg == p.nseg - 1) {
                if (r < rows_valid) p.y[static_cast<int64_t>(m) * p.N + row0 + r] = acc;
            } else {
                ycarry = acc;
            }
        }
        __syncwarp();
    }
    if (failed) {
        // A copy never completed: record it, then give the copies still in
        // flight (bounded) time to land before the CTA's shared memory goes.
        if (lane == 0) {
            atomicOr(p.status, CQ_DEV_WAIT_TIMEOUT);
            for (int64_t k = kfail; k < min(kfail + S, nsteps); ++k)
                (void)mbar_wait_bounded(&bars[k % S], static_cast<uint32_t>((k / S) & 1), WAIT_LIMIT_NS / 8);
        }
        __syncwarp();
    }
}

template <int WF, int MT>
cudaError_t launch_typed(const DeviceInfo& dev, const GemvParams& base, int64_t groups, cudaStream_t s) {
    GemvParams p = base;
    const int smem_budget = std::min(dev.smem_optin, 227 * 1024) - 1024;
    const int per_warp_fixed = 128 + p.M * p.R * p.segc * 4;
    // Shared memory per warp for S stages; pick the largest warp count (<= 16)
    // that leaves at least two stages per warp, preferring three or four.
    int S = 4;
    int wpc = 0;
    for (; S >= 2; --S) {
        p.stages = S;
        p.warp_bytes = (per_warp_fixed + S * p.stage_bytes + 127) / 128 * 128;
        wpc = std::min(wpc_limit<MT>(), (smem_budget - p.act_bytes) / p.warp_bytes);
        if (wpc >= 4 || (S == 2 && wpc >= 1)) break;
    }
    if (wpc < 1) return cudaErrorInvalidConfiguration;
    wpc = std::min(wpc, wpc_limit<MT>());
    // Spread the groups over all SMs before stacking warps on one SM.
    const int64_t want_wpc = std::max<int64_t>(1, (groups + dev.sm_count - 1) / dev.sm_count);
    wpc = static_cast<int>(std::min<int64_t>(wpc, want_wpc));
    // Balance: every warp gets the same number of groups (give or take one).
    const int64_t wmax = static_cast<int64_t>(dev.sm_count) * wpc;
    const int64_t per_warp = (groups + wmax - 1) / wmax;
    const int64_t warps = (groups + per_warp - 1) / per_warp;
    const unsigned grid = static_cast<unsigned>((warps + wpc - 1) / wpc);
    const int smem = p.act_bytes + wpc * p.warp_bytes;
    // Raise the kernel's dynamic shared-memory limit once per device.
    static int raised[64] = {};
    int devid = 0;
    cudaError_t e = cudaGetDevice(&devid);
    if (e != cudaSuccess) return e;
    if (devid < 64 && raised[devid] < smem) {
        e = cudaFuncSetAttribute(gemv_kernel<WF, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 std::min(dev.smem_optin, 227 * 1024));
        if (e != cudaSuccess) return e;
        raised[devid] = std::min(dev.smem_optin, 227 * 1024);
    }
    gemv_kernel<WF, MT><<<grid, wpc * 32, smem, s>>>(p);
    return cudaGetLastError();
}

template <int WF>
cudaError_t launch_fmt(const DeviceInfo& dev, const GemvParams& p, int64_t groups, cudaStream_t s) {
    if (p.M <= 1) return launch_typed<WF, 1>(dev, p, groups, s);
    if (p.M <= 4) return launch_typed<WF, 4>(dev, p, groups, s);
    if (p.M <= 8) return launch_typed<WF, 8>(dev, p, groups, s);
    return launch_typed<WF, 16>(dev, p, groups, s);
}

}  // namespace

cudaError_t launch_gemv(const DeviceInfo& dev, int w_fmt, int M, int64_t N, int64_t K, const void* W,
                        const void* xq, float* y, cudaStream_t s) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    const int nc = static_cast<int>(K / CHUNK_ELEMS);
    const int ch = wchunk_bytes(w_fmt);
    const int acp = (w_fmt == CQ_Q4_1 || w_fmt == CQ_Q4_K) ? 304 : 272;
    const int ach = achunk_bytes(act_fmt_for(w_fmt));
    const int64_t row_bytes = static_cast<int64_t>(nc) * ch;
    // Token groups so that the staged activations stay within 96 KB.
    const int tok_pitch = nc * acp;
    const int max_tok = std::max(1, std::min(M, (96 * 1024) / tok_pitch));
    if (tok_pitch > 96 * 1024) return cudaErrorInvalidValue;   // K beyond the supported range
    for (int m0 = 0; m0 < M; m0 += max_tok) {
        const int mm = std::min(max_tok, M - m0);
        GemvParams p{};
        p.W = static_cast<const uint8_t*>(W);
        p.xq = static_cast<const uint8_t*>(xq) + static_cast<int64_t>(m0) * nc * ach;
        p.y = y + static_cast<int64_t>(m0) * N;
        p.status = dev.status;
        p.N = N;
        p.row_bytes = row_bytes;
        p.M = mm;
        p.nc = nc;
        if (nc <= SEGC_MAX) {
            p.R = std::max(1, 32 / nc);
            p.segc = nc;
            p.nseg = 1;
            p.stage_bytes = static_cast<int>((p.R * row_bytes + 127) / 128 * 128);
        } else {
            p.R = 1;
            p.segc = SEGC_MAX;
            p.nseg = (nc + SEGC_MAX - 1) / SEGC_MAX;
            p.stage_bytes = (SEGC_MAX * ch + 127) / 128 * 128;
        }
        p.tok_pitch = tok_pitch;
        p.act_bytes = (mm * tok_pitch + 127) / 128 * 128;
        // The y rows of this token group are [m0, m0 + mm): y stride stays N.
        const int64_t groups = (N + p.R - 1) / p.R;
        cudaError_t e;
        switch (w_fmt) {
        case CQ_Q4_0: e = launch_fmt<CQ_Q4_0>(dev, p, groups, s); break;
        case CQ_Q8_0: e = launch_fmt<CQ_Q8_0>(dev, p, groups, s); break;
        case CQ_Q4_1: e = launch_fmt<CQ_Q4_1>(dev, p, groups, s); break;
        case CQ_Q4_K: e = launch_fmt<CQ_Q4_K>(dev, p, groups, s); break;
        default: return cudaErrorInvalidValue;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace cq
