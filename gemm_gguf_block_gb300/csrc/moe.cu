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
//   2. up:      per (expert, 32-row tile of F): gate and up tiles land in
//               shared memory by bulk copy; the expert's tokens stream past
//               them eight at a time; h = silu(g) * u, then Q8_0 of h.
//   3. down:    per (expert, 32-row tile of K): o = W_down . hq per pair.
//   4. combine: y[t] = sum over slots in slot order of w * o (fma chain).
#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "chunk_dot.cuh"
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
    L.perm = o; o = up(o + 4 * P);
    L.valid = o; o = up(o + 4 * P);
    L.h = o; o = up(o + 4 * P * static_cast<size_t>(F));
    L.hq = o; o = up(o + P * static_cast<size_t>(F / 32 * 34));
    L.out = o; o = up(o + 4 * P * static_cast<size_t>(K));
    L.total = o;
    return L;
}

namespace {

constexpr int TILE = 32;      // weight rows per CTA tile
constexpr int TOKG = 8;       // tokens per pass over a tile
constexpr int THREADS = 256;

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

// Copy `n` 34-byte-block rows (token rows of Q8_0) into shared memory, row i
// from src_row(i), `words` 32-bit words each, destination pitch `pitch`.
template <class RowFn>
__device__ __forceinline__ void stage_rows(uint8_t* dst, int pitch, int n, int words, RowFn src_row) {
    const int total = n * words;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int r = i / words, w = i - r * words;
        reinterpret_cast<uint32_t*>(dst + r * pitch)[w] = reinterpret_cast<const uint32_t*>(src_row(r))[w];
    }
}

// Wait (all threads) for the weight tile; on timeout flag it, give the copy a
// second bounded wait to land (so none is in flight when the CTA exits) and
// report false.
__device__ __forceinline__ bool wait_tile(uint64_t* bar, int* status) {
    const bool ok = mbar_wait_bounded(bar, 0, WAIT_LIMIT_NS);
    if (__syncthreads_and(ok)) return true;
    if (threadIdx.x == 0) {
        atomicOr(status, CQ_DEV_WAIT_TIMEOUT);
        (void)mbar_wait_bounded(bar, 0, WAIT_LIMIT_NS / 8);
    }
    __syncthreads();
    return false;
}

// ------------------------------------------------------------- gate/up + SwiGLU
__global__ void __launch_bounds__(THREADS) moe_up_kernel(const MoeParams p) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ __align__(128) uint8_t smem[];
    const int e = blockIdx.y, f0 = blockIdx.x * TILE;
    const int* offs = ws_offs(p);
    const int beg = offs[e], cnt = offs[e + 1] - beg;
    if (cnt == 0) return;
    const int nc = p.K / CHUNK_ELEMS;
    const int rowb = nc * WCHUNK_Q4_0;                 // bytes of one weight row
    const int tok_pitch = nc * ACHUNK_Q8_0;            // one Q8_0 token row
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    uint8_t* wt = smem + 128;                          // [2*TILE rows][rowb]: gate rows, then up rows
    uint8_t* xs = wt + (2 * TILE * rowb + 127) / 128 * 128;
    float* cbuf = reinterpret_cast<float*>(xs + (TOKG * tok_pitch + 127) / 128 * 128);   // [TOKG][2*TILE][nc]
    float* gu = cbuf + TOKG * 2 * TILE * nc;                                              // [TOKG][2*TILE]
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        const uint32_t half = static_cast<uint32_t>(TILE * rowb);
        mbar_arrive_expect_tx(bar, 2 * half);
        const size_t mat = static_cast<size_t>(p.F) * rowb;
        const uint64_t pol = policy_evict_first();
        bulk_g2s(wt, p.Wg + e * mat + static_cast<size_t>(f0) * rowb, half, bar, pol);
        bulk_g2s(wt + half, p.Wu + e * mat + static_cast<size_t>(f0) * rowb, half, bar, pol);
    }
    __syncthreads();
    const int* perm = ws_perm(p) + beg;
    bool have_tile = false;
    float* hbase = reinterpret_cast<float*>(p.ws + p.L.h);
    uint8_t* hqbase = p.ws + p.L.hq;
    const int hq_row = p.F / 32 * 34;
    for (int g0 = 0; g0 < cnt; g0 += TOKG) {
        const int gm = min(TOKG, cnt - g0);
        stage_rows(xs, tok_pitch, gm, tok_pitch / 4,
                   [&](int r) { return p.xq + static_cast<size_t>(perm[g0 + r] / p.topk) * tok_pitch; });
        if (!have_tile) {
            if (!wait_tile(bar, ws_status(p))) return;
            have_tile = true;
        } else {
            __syncthreads();
        }
        const int ntasks = 2 * TILE * nc;
        for (int t = threadIdx.x; t < ntasks; t += blockDim.x) {
            const int r = t / nc, j = t - r * nc;
            float c[TOKG];
            chunk_dot<CQ_Q4_0, TOKG>(wt + r * rowb + j * WCHUNK_Q4_0, xs + j * ACHUNK_Q8_0, tok_pitch, gm, c);
#pragma unroll
            for (int m = 0; m < TOKG; ++m)
                if (m < gm) cbuf[(m * 2 * TILE + r) * nc + j] = c[m];
        }
        __syncthreads();
        for (int q = threadIdx.x; q < gm * 2 * TILE; q += blockDim.x) {
            const float* cb = cbuf + q * nc;
            float acc = 0.0f;
            for (int j = 0; j < nc; ++j) acc = __fadd_rn(acc, cb[j]);
            gu[q] = acc;
        }
        __syncthreads();
        // One warp per token: lane f of the 32-row tile; h = silu(g) * u, then
        // the Q8_0 block of these 32 values (the cq_quantize_act rule).
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        if (warp < gm) {
            const int pair = perm[g0 + warp];
            const float g = gu[warp * 2 * TILE + lane];
            const float u = gu[warp * 2 * TILE + TILE + lane];
            const float silu = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
            const float h = __fmul_rn(silu, u);
            hbase[static_cast<size_t>(pair) * p.F + f0 + lane] = h;
            float amax = fabsf(h);
#pragma unroll
            for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float d = q8_scale(amax);
            const float id = q8_inv(d);
            uint8_t* blk = hqbase + static_cast<size_t>(pair) * hq_row + (f0 / 32) * 34;
            blk[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(quant_q8(h, id)));
            if (lane == 0) *reinterpret_cast<__half*>(blk) = __float2half_rn(d);
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------- down
__global__ void __launch_bounds__(THREADS) moe_down_kernel(const MoeParams p) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ __align__(128) uint8_t smem[];
    const int e = blockIdx.y, k0 = blockIdx.x * TILE;
    const int* offs = ws_offs(p);
    const int beg = offs[e], cnt = offs[e + 1] - beg;
    if (cnt == 0) return;
    const int nc = p.F / CHUNK_ELEMS;
    const int rowb = nc * WCHUNK_Q4_0;
    const int tok_pitch = nc * ACHUNK_Q8_0;            // one hq row
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    uint8_t* wt = smem + 128;
    uint8_t* xs = wt + (TILE * rowb + 127) / 128 * 128;
    float* cbuf = reinterpret_cast<float*>(xs + (TOKG * tok_pitch + 127) / 128 * 128);   // [TOKG][TILE][nc]
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        const uint32_t bytes = static_cast<uint32_t>(TILE * rowb);
        mbar_arrive_expect_tx(bar, bytes);
        const size_t mat = static_cast<size_t>(p.K) * rowb;
        bulk_g2s(wt, p.Wd + e * mat + static_cast<size_t>(k0) * rowb, bytes, bar, policy_evict_first());
    }
    __syncthreads();
    const int* perm = ws_perm(p) + beg;
    const uint8_t* hq = p.ws + p.L.hq;
    float* out = reinterpret_cast<float*>(p.ws + p.L.out);
    bool have_tile = false;
    for (int g0 = 0; g0 < cnt; g0 += TOKG) {
        const int gm = min(TOKG, cnt - g0);
        stage_rows(xs, tok_pitch, gm, tok_pitch / 4,
                   [&](int r) { return hq + static_cast<size_t>(perm[g0 + r]) * tok_pitch; });
        if (!have_tile) {
            if (!wait_tile(bar, ws_status(p))) return;
            have_tile = true;
        } else {
            __syncthreads();
        }
        const int ntasks = TILE * nc;
        for (int t = threadIdx.x; t < ntasks; t += blockDim.x) {
            const int r = t / nc, j = t - r * nc;
            float c[TOKG];
            chunk_dot<CQ_Q4_0, TOKG>(wt + r * rowb + j * WCHUNK_Q4_0, xs + j * ACHUNK_Q8_0, tok_pitch, gm, c);
#pragma unroll
            for (int m = 0; m < TOKG; ++m)
                if (m < gm) cbuf[(m * TILE + r) * nc + j] = c[m];
        }
        __syncthreads();
        for (int q = threadIdx.x; q < gm * TILE; q += blockDim.x) {
            const int m = q / TILE, r = q - m * TILE;
            const float* cb = cbuf + q * nc;
            float acc = 0.0f;
            for (int j = 0; j < nc; ++j) acc = __fadd_rn(acc, cb[j]);
            out[static_cast<size_t>(perm[g0 + m]) * p.K + k0 + r] = acc;
        }
        __syncthreads();
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

// CQ_MOE_MMA=0 runs the dp4a projections instead of the tensor-core ones (A/B runs).
bool moe_mma_enabled() {
    static const bool v = [] {
        const char* e = std::getenv("CQ_MOE_MMA");
        return !(e && e[0] == '0');
    }();
    return v;
}

size_t moe_up_smem(int K) {
    const int nc = K / CHUNK_ELEMS;
    const int rowb = nc * WCHUNK_Q4_0, tok_pitch = nc * ACHUNK_Q8_0;
    return 128 + (2 * TILE * rowb + 127) / 128 * 128 + (TOKG * tok_pitch + 127) / 128 * 128 +
           4 * (TOKG * 2 * TILE * nc + TOKG * 2 * TILE);
}
size_t moe_down_smem(int F) {
    const int nc = F / CHUNK_ELEMS;
    const int rowb = nc * WCHUNK_Q4_0, tok_pitch = nc * ACHUNK_Q8_0;
    return 128 + (TILE * rowb + 127) / 128 * 128 + (TOKG * tok_pitch + 127) / 128 * 128 + 4 * (TOKG * TILE * nc);
}

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
    if (moe_mma_enabled()) {
        e = launch_moe_projections(dev, T, K, F, E, topk, Wg, Wu, Wd, xq, reinterpret_cast<const int*>(p.ws + p.L.offs),
                                   reinterpret_cast<const int*>(p.ws + p.L.perm), reinterpret_cast<float*>(p.ws + p.L.h),
                                   p.ws + p.L.hq, reinterpret_cast<float*>(p.ws + p.L.out), s);
        if (e != cudaSuccess) return e;
    } else {
        const int smem_up = static_cast<int>(moe_up_smem(K));
        const int smem_dn = static_cast<int>(moe_down_smem(F));
        const int lim = std::min(dev.smem_optin, 227 * 1024);
        if (smem_up > lim || smem_dn > lim) return cudaErrorInvalidConfiguration;
        static int raised[64] = {};
        int devid = 0;
        if ((e = cudaGetDevice(&devid)) != cudaSuccess) return e;
        if (devid >= 64 || !raised[devid]) {
            if ((e = cudaFuncSetAttribute(moe_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lim)) !=
                cudaSuccess)
                return e;
            if ((e = cudaFuncSetAttribute(moe_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lim)) !=
                cudaSuccess)
                return e;
            if (devid < 64) raised[devid] = 1;
        }
        if ((e = launch_kernel(moe_up_kernel, dim3(F / TILE, E), dim3(THREADS), smem_up, s, p)) != cudaSuccess)
            return e;
        if ((e = launch_kernel(moe_down_kernel, dim3(K / TILE, E), dim3(THREADS), smem_dn, s, p)) != cudaSuccess)
            return e;
    }
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

