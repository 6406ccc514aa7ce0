// Routed-expert FFN (lfm2moe-style: each token picks topk of E experts).
//
// cera README "Supported models": every token routes to 4 of 32 experts and
// the block's output is the router-weighted sum of the chosen experts'
// SwiGLU FFNs; the pages note that their GPU kernels re-read an expert's
// weights once per routed token and name grouping tokens by expert as the
// follow-up. This file does that grouping: each expert's weights are read
// once per call, for all the tokens routed to it.
// alice-llm "WGSL Shader Architecture" (swiglu_fused_q4k): gate and up share
// one pass over the input.
//
// Pipeline (all asynchronous on the caller's stream, no host round trip):
//   1. route:   validate ids (range, no repeats within a token), counting-sort
//               the (token, slot) pairs by expert; stable, so deterministic.
//   2. up:      per (expert, 128 rows of F), on the tensor cores
//               (moe_mma.cu): gate and up for the expert's pairs, h =
//               silu(g) * u, then Q8_0 of h.
//   3. down:    per (expert, 128 rows of K), on the tensor cores: o = W_down . hq.
//   4. combine: y[t] = sum over slots in slot order of w * o (fma chain).
#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "cq_device.cuh"
#include "cq_internal.h"

namespace cq {

MoeLayout moe_layout(int64_t T, int64_t K, int64_t F, int64_t E, int64_t topk) {
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    MoeLayout L{};
    const size_t P = static_cast<size_t>(T * topk);
    size_t o = 0;
    L.status = o; o += 256;
    L.offs = o; o = up(o + 4 * static_cast<size_t>(E + 1));
    L.order = o; o = up(o + 4 * static_cast<size_t>(E));
    L.perm = o; o = up(o + 4 * P);
    L.valid = o; o = up(o + 4 * P);
    L.h = o; o = up(o + 4 * P * static_cast<size_t>(F));
    L.hq = o; o = up(o + P * static_cast<size_t>(F / 32 * 34));
    L.out = o; o = up(o + 4 * P * static_cast<size_t>(K));
    L.total = o;
    return L;
}

namespace {

struct MoeParams {
    const uint8_t* Wg;
    const uint8_t* Wu;
    const uint8_t* Wd;
    const int32_t* ids;
    const float* rw;
    const uint8_t* xq;
    float* y;
    uint8_t* ws;
    MoeLayout L;
    int T, K, F, E, topk;
};

__device__ __forceinline__ int* ws_status(const MoeParams& p) { return reinterpret_cast<int*>(p.ws + p.L.status); }
__device__ __forceinline__ int* ws_offs(const MoeParams& p) { return reinterpret_cast<int*>(p.ws + p.L.offs); }
__device__ __forceinline__ int* ws_perm(const MoeParams& p) { return reinterpret_cast<int*>(p.ws + p.L.perm); }
__device__ __forceinline__ int* ws_valid(const MoeParams& p) { return reinterpret_cast<int*>(p.ws + p.L.valid); }

// ------------------------------------------------------------------ route
// Pairs whose routing keys are staged in shared memory; larger batches read
// them from global memory instead.
constexpr int ROUTE_SMEM_PAIRS = 8192;

__global__ void __launch_bounds__(1024) moe_route_kernel(const MoeParams p) {
    pdl_trigger();
    pdl_wait();
    __shared__ int cnt[256];
    __shared__ int off[257];
    __shared__ int key_s[ROUTE_SMEM_PAIRS];   // expert of a valid pair, -1 for an invalid one
    const int P = p.T * p.topk;
    const bool staged = P <= ROUTE_SMEM_PAIRS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    int* valid = ws_valid(p);
    int* status = ws_status(p);
    if (tid == 0) *status = 0;   // the call's status word starts clear
    __syncthreads();
    for (int i = tid; i < P; i += blockDim.x) {
        const int t = i / p.topk, s = i - t * p.topk;
        const int e = p.ids[i];
        int flag = 0;
        if (e < 0 || e >= p.E) {
            flag = CQ_DEV_BAD_EXPERT_ID;
        } else {
            for (int s2 = 0; s2 < s; ++s2)
                if (p.ids[t * p.topk + s2] == e) flag = CQ_DEV_DUP_EXPERT_ID;
        }
        valid[i] = flag == 0;
        if (staged) key_s[i] = flag == 0 ? e : -1;
        if (flag) atomicOr(status, flag);
    }
    __syncthreads();   // valid[] and key_s[] written by this CTA: visible to it after the barrier
    auto key = [&](int i) { return staged ? key_s[i] : (valid[i] ? p.ids[i] : -1); };
    for (int e = warp; e < p.E; e += nwarps) {
        int c = 0;
        for (int base = 0; base < P; base += 32) {
            const int i = base + lane;
            c += __popc(__ballot_sync(0xffffffffu, i < P && key(i) == e));
        }
        if (lane == 0) cnt[e] = c;
    }
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int e = 0; e < p.E; ++e) { off[e] = acc; acc += cnt[e]; }
        off[p.E] = acc;
    }
    __syncthreads();
    int* offs = ws_offs(p);
    int* perm = ws_perm(p);
    for (int e = tid; e <= p.E; e += blockDim.x) offs[e] = off[e];
    // Experts by decreasing pair count (ties by id): the projection CTAs take
    // them in this order, so the largest start first and the small ones fill
    // the last wave.
    int* order = reinterpret_cast<int*>(p.ws + p.L.order);
    for (int e = tid; e < p.E; e += blockDim.x) {
        const int c = cnt[e];
        int rank = 0;
        for (int e2 = 0; e2 < p.E; ++e2) rank += (cnt[e2] > c) || (cnt[e2] == c && e2 < e);
        order[rank] = e;
    }
    for (int e = warp; e < p.E; e += nwarps) {
        int pos = off[e];
        for (int base = 0; base < P; base += 32) {
            const int i = base + lane;
            const bool hit = i < P && key(i) == e;
            const unsigned m = __ballot_sync(0xffffffffu, hit);
            if (hit) perm[pos + __popc(m & ((1u << lane) - 1u))] = i;
            pos += __popc(m);
        }
    }
}

// ---------------------------------------------------------------- combine
// y[t] = sum over the token's valid slots s, in increasing s, of rw * o; one
// CTA row per token, four consecutive outputs per thread.
__global__ void __launch_bounds__(256) moe_combine_kernel(const MoeParams p) {
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x;
    const int k = 4 * (blockIdx.y * blockDim.x + threadIdx.x);
    if (k >= p.K) return;
    const int* valid = ws_valid(p);
    const float* out = reinterpret_cast<const float*>(p.ws + p.L.out);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < p.topk; ++s) {
        const int pair = t * p.topk + s;
        if (!valid[pair]) continue;
        const float w = p.rw[pair];
        const float4 o = *reinterpret_cast<const float4*>(out + static_cast<size_t>(pair) * p.K + k);
        acc.x = __fmaf_rn(w, o.x, acc.x);
        acc.y = __fmaf_rn(w, o.y, acc.y);
        acc.z = __fmaf_rn(w, o.z, acc.z);
        acc.w = __fmaf_rn(w, o.w, acc.w);
    }
    *reinterpret_cast<float4*>(p.y + static_cast<size_t>(t) * p.K + k) = acc;
}

}  // namespace

cudaError_t launch_moe(const DeviceInfo& dev, int T, int K, int F, int E, int topk, const void* Wg,
                       const void* Wu, const void* Wd, const int32_t* ids, const float* rw, const void* xq,
                       float* y, void* ws, cudaStream_t s) {
    MoeParams p{};
    p.Wg = static_cast<const uint8_t*>(Wg);
    p.Wu = static_cast<const uint8_t*>(Wu);
    p.Wd = static_cast<const uint8_t*>(Wd);
    p.ids = ids;
    p.rw = rw;
    p.xq = static_cast<const uint8_t*>(xq);
    p.y = y;
    p.ws = static_cast<uint8_t*>(ws);
    p.L = moe_layout(T, K, F, E, topk);
    p.T = T; p.K = K; p.F = F; p.E = E; p.topk = topk;
    cudaError_t e = launch_kernel(moe_route_kernel, dim3(1), dim3(1024), 0, s, p);
    if (e != cudaSuccess) return e;
    e = launch_moe_projections(dev, T, K, F, E, topk, Wg, Wu, Wd, xq, reinterpret_cast<const int*>(p.ws + p.L.offs),
                               reinterpret_cast<const int*>(p.ws + p.L.order),
                               reinterpret_cast<const int*>(p.ws + p.L.perm), reinterpret_cast<float*>(p.ws + p.L.h),
                               p.ws + p.L.hq, reinterpret_cast<float*>(p.ws + p.L.out), s);
    if (e != cudaSuccess) return e;
    return launch_kernel(moe_combine_kernel, dim3(static_cast<unsigned>(T), static_cast<unsigned>((K / 4 + 255) / 256)),
                         dim3(256), 0, s, p);
}

}  // namespace cq

// ------------------------------------------------------ allocation-free entry
//
// cq_moe_gemv_noalloc: the routed-expert FFN for callers that cannot call
// cudaMalloc and so cannot hand the library a workspace -- for example a
// plugin whose host framework has already reserved the GPU's memory for its
// own pool and exposes no way to ask for more, or a latency-critical decode
// loop in which the device-wide synchronisation of cudaMalloc is not
// acceptable. Its scratch space is a fixed array in device memory that is part
// of this library's image: every GPU that loads libcq holds these
// CQ_MOE_NOALLOC_MAX_BYTES until the process exits.
namespace cq {
namespace {

static __device__ __align__(256) uint8_t g_moe_noalloc_scratch[CQ_MOE_NOALLOC_MAX_BYTES];

constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mutex;
uint8_t* g_noalloc_ptr[NOALLOC_MAX_DEVICES];

// Device address of the scratch array on the current device. In host code the
// array's name stands for a host-side shadow, not for device memory, so the
// address has to be asked of the runtime, once per device, with that device
// current.
cudaError_t noalloc_scratch(uint8_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_moe_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace cq

extern "C" cq_status cq_moe_gemv_noalloc(cq_format w_fmt, int64_t T, int64_t K, int64_t F, int64_t E,
                                         int64_t topk, const void* W_gate, const void* W_up, const void* W_down,
                                         const int32_t* expert_ids, const float* route_w, const void* xq,
                                         float* y, void* stream) {
    if (w_fmt != CQ_Q4_0) return CQ_ERR_UNSUPPORTED_FORMAT;
    if (T < 0 || K < 0 || F < 0 || E < 0 || topk < 0) return CQ_ERR_INVALID_ARG;
    const size_t need = cq_moe_workspace_size(T, K, F, E, topk);
    if (need == 0) return CQ_ERR_SHAPE;                       // a shape cq_moe_gemv rejects too
    if (T == 0) return CQ_OK;
    if (need > CQ_MOE_NOALLOC_MAX_BYTES) return CQ_ERR_WORKSPACE;
    if (!W_gate || !W_up || !W_down || !expert_ids || !route_w || !xq || !y) return CQ_ERR_INVALID_ARG;
    for (const void* q : {W_gate, W_up, W_down, static_cast<const void*>(expert_ids),
                          static_cast<const void*>(route_w), xq, static_cast<const void*>(y)})
        if ((reinterpret_cast<uintptr_t>(q) & 15u) != 0) return CQ_ERR_ALIGNMENT;
    cq::DeviceInfo dev;
    if (cq::device_info(&dev) != cudaSuccess) return CQ_ERR_CUDA;
    uint8_t* scratch = nullptr;
    if (cq::noalloc_scratch(&scratch) != cudaSuccess) return CQ_ERR_CUDA;
    cudaError_t e = cq::launch_moe(dev, static_cast<int>(T), static_cast<int>(K), static_cast<int>(F),
                                   static_cast<int>(E), static_cast<int>(topk), W_gate, W_up, W_down, expert_ids,
                                   route_w, xq, y, scratch, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CQ_OK : CQ_ERR_CUDA;
}

extern "C" cq_status cq_moe_noalloc_read_status(int32_t* out_code, void* stream) {
    if (out_code == nullptr) return CQ_ERR_INVALID_ARG;
    uint8_t* scratch = nullptr;
    if (cq::noalloc_scratch(&scratch) != cudaSuccess) return CQ_ERR_CUDA;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return CQ_ERR_CUDA;
    int v = 0;
    // The status word is the first section of the layout (offset 0) for every shape.
    if (cudaMemcpy(&v, scratch + cq::moe_layout(1, 256, 256, 1, 1).status, sizeof v, cudaMemcpyDeviceToHost) !=
        cudaSuccess)
        return CQ_ERR_CUDA;
    *out_code = v;
    if (v & CQ_DEV_WAIT_TIMEOUT) return CQ_ERR_TIMEOUT;
    return v ? CQ_ERR_DEVICE_STATUS : CQ_OK;
}

