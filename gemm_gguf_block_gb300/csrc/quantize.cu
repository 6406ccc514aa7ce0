// Activation quantisation fp32 -> Q8_0 / Q8_1 / Q8_K.
//
// alice-llm docs, "Phase 4 -- i8 Dynamic Quantization + SDOT": per chunk the
// absolute maximum, a scale of amax/127, and a rounded int8 per element;
// "Computation Path (Q4_K)" step 1: Q8_K = 256 elements with an fp32 scale,
// int8 values and int16 sums of each 16 values; cera README "Quantization":
// activations quantized dynamically to Q8_0.
//
// Every decision is taken in fp32 with IEEE round-to-nearest: d = amax / 127
// (correctly rounded division), id = 1/d (correctly rounded reciprocal),
// q = roundf(x * id) (ties away from zero), clamped to [-127, 127]. The fp16
// scale is d rounded to nearest even, subnormals kept.
//
// Eight consecutive elements per lane (two 16-byte loads): four lanes per
// 32-block, a whole warp per 256-block.
#include <algorithm>

#include "cq_device.cuh"
#include "cq_internal.h"

namespace cq {
namespace {

__device__ __forceinline__ float warp_max(float a) {
#pragma unroll
    for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    return a;
}

template <int AF>
__global__ void __launch_bounds__(256) quantize32_kernel(const float* __restrict__ x, uint8_t* __restrict__ xq,
                                                         int64_t nblocks) {
    pdl_trigger();
    pdl_wait();
    constexpr int BB = AF == CQ_Q8_0 ? 34 : 36;     // block bytes
    constexpr int QOFF = AF == CQ_Q8_0 ? 2 : 4;     // offset of the quants
    const int lane = threadIdx.x & 31, sub = lane & 3;
    const int64_t wstride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    // A warp takes eight blocks at a time; the trip count is uniform across it.
    for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w * 8 < nblocks;
         w += wstride) {
        const int64_t b = w * 8 + (lane >> 2);
        const bool on = b < nblocks;
        float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
        if (on) {
            const float4* src = reinterpret_cast<const float4*>(x + b * 32 + 8 * sub);
            v0 = src[0];
            v1 = src[1];
        }
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
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
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if (on) {
            uint8_t* blk = xq + b * BB;
            if constexpr (AF == CQ_Q8_0) {      // quants at 2 mod 4: 16-bit stores
                uint16_t* q16 = reinterpret_cast<uint16_t*>(blk + QOFF + 8 * sub);
                q16[0] = static_cast<uint16_t>(packed[0]);
                q16[1] = static_cast<uint16_t>(packed[0] >> 16);
                q16[2] = static_cast<uint16_t>(packed[1]);
                q16[3] = static_cast<uint16_t>(packed[1] >> 16);
            } else {
                uint32_t* q32 = reinterpret_cast<uint32_t*>(blk + QOFF + 8 * sub);
                q32[0] = packed[0];
                q32[1] = packed[1];
            }
            if (sub == 0) {
                *reinterpret_cast<__half*>(blk) = __float2half_rn(d);
                if constexpr (AF == CQ_Q8_1)
                    *reinterpret_cast<__half*>(blk + 2) = __float2half_rn(__fmul_rn(d, static_cast<float>(sum)));
            }
        }
    }
}

__global__ void __launch_bounds__(256) quantize_q8k_kernel(const float* __restrict__ x, uint8_t* __restrict__ xq,
                                                           int64_t nblocks) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t stride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; b < nblocks; b += stride) {
        const float4* src = reinterpret_cast<const float4*>(x + b * 256 + 8 * lane);
        const float4 v0 = src[0], v1 = src[1];
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
        const float amax = warp_max(a);
        const float d = q8_scale(amax);
        const float id = q8_inv(d);
        uint32_t packed[2] = {0u, 0u};
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int q = quant_q8(v[i], id);
            sum += q;
            packed[i >> 2] |= (static_cast<uint32_t>(q) & 0xffu) << (8 * (i & 3));
        }
        uint8_t* blk = xq + b * 292;
        uint32_t* qw = reinterpret_cast<uint32_t*>(blk + 4 + 8 * lane);
        qw[0] = packed[0];
        qw[1] = packed[1];
        const int pair = sum + __shfl_xor_sync(0xffffffffu, sum, 1);   // 16 consecutive quants
        if ((lane & 1) == 0)
            *reinterpret_cast<int16_t*>(blk + 260 + lane) = static_cast<int16_t>(pair);
        if (lane == 0) *reinterpret_cast<float*>(blk) = d;
    }
}

// Self-test of the bounded wait every kernel uses: one thread waits, with
// the given limit, on an mbarrier phase that nothing completes, then sets the
// timeout bit in the status word -- the path a kernel takes when a copy never
// lands. Nothing faults and the context stays usable.
__global__ void wait_timeout_probe_kernel(uint64_t limit_ns, int* status) {
    pdl_trigger();
    pdl_wait();
    __shared__ uint64_t bar;
    mbar_init(&bar, 1);                       // one arrival expected; none comes
    fence_mbar_init();
    if (!mbar_wait_bounded(&bar, 0, limit_ns)) atomicOr(status, CQ_DEV_WAIT_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_timeout_probe(uint64_t limit_ns, int* status, cudaStream_t s) {
    return launch_kernel(wait_timeout_probe_kernel, dim3(1), dim3(1), 0, s, limit_ns, status);
}

cudaError_t launch_quantize(int act_fmt, int64_t M, int64_t K, const float* x, void* xq, cudaStream_t s) {
    const int bs = act_fmt == CQ_Q8_K ? 256 : 32;
    const int64_t nblocks = M * (K / bs);
    if (nblocks == 0) return cudaSuccess;
    const int64_t warps = act_fmt == CQ_Q8_K ? nblocks : (nblocks + 7) / 8;
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>((warps + 7) / 8, 16384));
    uint8_t* out = static_cast<uint8_t*>(xq);
    switch (act_fmt) {
    case CQ_Q8_0: return launch_kernel(quantize32_kernel<CQ_Q8_0>, dim3(grid), dim3(256), 0, s, x, out, nblocks);
    case CQ_Q8_1: return launch_kernel(quantize32_kernel<CQ_Q8_1>, dim3(grid), dim3(256), 0, s, x, out, nblocks);
    case CQ_Q8_K: return launch_kernel(quantize_q8k_kernel, dim3(grid), dim3(256), 0, s, x, out, nblocks);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace cq
