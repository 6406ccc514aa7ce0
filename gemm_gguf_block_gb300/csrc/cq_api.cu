// C ABI of libcq: argument validation and dispatch to the kernel launchers.
// Every check runs before any launch, so an error return means that nothing
// was launched and nothing was written. See include/cq.h for the contract.
#include <cstdint>
#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include <cuda_runtime.h>

#include "cq.h"
#include "cq_internal.h"

namespace {

// Status word of kernels that take no workspace (cq_gemv / cq_gemm copy waits).
__device__ int g_cq_status;

constexpr int MAX_DEVICES = 64;
std::mutex g_dev_mutex;
bool g_dev_ready[MAX_DEVICES];
cq::DeviceInfo g_dev[MAX_DEVICES];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Quantized activation rows: Q8_K rows are 292 bytes per 256 elements, so a
// token's row is only 4-byte aligned; the kernels read activations in 32-bit words.
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool is_weight_fmt(int f) {
    return f == CQ_Q4_0 || f == CQ_Q4_1 || f == CQ_Q8_0 || f == CQ_Q4_K || f == CQ_Q5_K || f == CQ_Q6_K;
}
// Q6_K rows of 210-byte superblocks meet the bulk copies' 16-byte rule only
// eight superblocks at a time: K a multiple of 2048.
bool fmt_shape_ok(int f, int64_t K) { return f != CQ_Q6_K || K % 2048 == 0; }
bool is_act_fmt(int f) { return f == CQ_Q8_0 || f == CQ_Q8_1 || f == CQ_Q8_K; }

// Largest K accepted by the single-pass kernels (activation rows staged in
// 96 KB of shared memory: 96 KB / 304 B per 256 elements).
constexpr int64_t K_MAX = 65536;

cq_status check_shape(int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return CQ_ERR_INVALID_ARG;
    if (K == 0 || K % 256 != 0 || K > K_MAX) return CQ_ERR_SHAPE;
    if (N > (int64_t(1) << 31)) return CQ_ERR_SHAPE;
    return CQ_OK;
}

}  // namespace

namespace cq {
std::atomic<int> g_weights_const{0};
bool weights_const() { return g_weights_const.load(std::memory_order_relaxed) != 0; }

std::mutex g_attr_mutex;
std::map<std::pair<int, const void*>, int> g_attr_raised;

cudaError_t raise_smem_limit(const void* kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    int& have = g_attr_raised[{dev, kernel}];
    if (have >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) have = bytes;
    return e;
}

// Library-owned stream-ordered scratch: one memory pool per device, created on
// first use, keeping up to 512 MB between calls so that steady-state
// allocations map no new memory.
std::mutex g_pool_mutex;
bool g_pool_ready[MAX_DEVICES];
cudaMemPool_t g_pool[MAX_DEVICES];

void* scratch_alloc(size_t bytes, cudaStream_t s) {
    int dev = 0;
    if (bytes == 0 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
    // No allocation while the stream is being captured into a graph: the
    // caller then takes its allocation-free path.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (cap != cudaStreamCaptureStatusNone) return nullptr;
    cudaMemPool_t pool;
    {
        std::lock_guard<std::mutex> lock(g_pool_mutex);
        if (!g_pool_ready[dev]) {
            cudaMemPoolProps props{};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            if (cudaMemPoolCreate(&g_pool[dev], &props) != cudaSuccess) {
                (void)cudaGetLastError();
                return nullptr;
            }
            uint64_t keep = uint64_t(512) << 20;
            (void)cudaMemPoolSetAttribute(g_pool[dev], cudaMemPoolAttrReleaseThreshold, &keep);
            g_pool_ready[dev] = true;
        }
        pool = g_pool[dev];
    }
    void* p = nullptr;
    if (cudaMallocFromPoolAsync(&p, bytes, pool, s) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if ((reinterpret_cast<uintptr_t>(p) & 255u) != 0) {   // the GEMM workspaces want 256-byte alignment
        (void)cudaFreeAsync(p, s);
        return nullptr;
    }
    return p;
}

cudaError_t scratch_free(void* p, cudaStream_t s) { return p != nullptr ? cudaFreeAsync(p, s) : cudaSuccess; }

cudaError_t device_info(DeviceInfo* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_dev_ready[dev]) {
        DeviceInfo d{};
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_cq_status);
        if (e != cudaSuccess) return e;
        g_dev[dev] = d;
        g_dev_ready[dev] = true;
    }
    *out = g_dev[dev];
    return cudaSuccess;
}
}  // namespace cq

extern "C" {

const char* cq_status_string(cq_status s) {
    switch (s) {
    case CQ_OK: return "ok";
    case CQ_ERR_INVALID_ARG: return "invalid argument";
    case CQ_ERR_UNSUPPORTED_FORMAT: return "unsupported format";
    case CQ_ERR_SHAPE: return "unsupported shape";
    case CQ_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case CQ_ERR_WORKSPACE: return "workspace missing or too small";
    case CQ_ERR_CUDA: return "CUDA error";
    case CQ_ERR_DEVICE_STATUS: return "device reported bad input";
    case CQ_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

cq_status cq_quantize_act(cq_format act_fmt, int64_t M, int64_t K, const float* x, void* xq, void* stream) {
    if (!is_act_fmt(act_fmt)) return CQ_ERR_UNSUPPORTED_FORMAT;
    cq_status st = check_shape(M, 1, K);
    if (st != CQ_OK) return st;
    if (M == 0) return CQ_OK;
    if (x == nullptr || xq == nullptr) return CQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq)) return CQ_ERR_ALIGNMENT;
    cudaError_t e = cq::launch_quantize(act_fmt, M, K, x, xq, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CQ_OK : CQ_ERR_CUDA;
}

cq_status cq_gemv(cq_format w_fmt, int64_t M, int64_t N, int64_t K, const void* W, const void* xq, float* y,
                  void* stream) {
    if (!is_weight_fmt(w_fmt)) return CQ_ERR_UNSUPPORTED_FORMAT;
    cq_status st = check_shape(M, N, K);
    if (st != CQ_OK) return st;
    if (M > 16 || !fmt_shape_ok(w_fmt, K)) return CQ_ERR_SHAPE;
    if (M == 0 || N == 0) return CQ_OK;
    if (W == nullptr || xq == nullptr || y == nullptr) return CQ_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned4(xq) || !aligned16(y)) return CQ_ERR_ALIGNMENT;
    cq::DeviceInfo dev;
    if (cq::device_info(&dev) != cudaSuccess) return CQ_ERR_CUDA;
    cudaError_t e = cq::launch_gemv(dev, w_fmt, static_cast<int>(M), N, K, W, xq, y, nullptr,
                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CQ_OK : CQ_ERR_CUDA;
}

size_t cq_repack_size(cq_format w_fmt, int64_t N, int64_t K) {
    if (N < 0 || K > K_MAX) return 0;
    return static_cast<size_t>(cq::repack_size(w_fmt, N, K));
}

cq_status cq_repack(cq_format w_fmt, int64_t N, int64_t K, const void* W, void* Wp, void* stream) {
    if (w_fmt != CQ_Q4_0 && w_fmt != CQ_Q4_1 && w_fmt != CQ_Q8_0) return CQ_ERR_UNSUPPORTED_FORMAT;
    cq_status st = check_shape(1, N, K);
    if (st != CQ_OK) return st;
    if (N == 0) return CQ_OK;
    if (W == nullptr || Wp == nullptr) return CQ_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(Wp)) return CQ_ERR_ALIGNMENT;
    cudaError_t e = cq::launch_repack(w_fmt, N, K, W, Wp, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CQ_OK : CQ_ERR_CUDA;
}

cq_status cq_gemv_packed(cq_format w_fmt, int64_t M, int64_t N, int64_t K, const void* Wp, const void* xq, float* y,
                         void* stream) {
    if (w_fmt != CQ_Q4_0 && w_fmt != CQ_Q4_1 && w_fmt != CQ_Q8_0) return CQ_ERR_UNSUPPORTED_FORMAT;
    cq_status st = check_shape(M, N, K);
    if (st != CQ_OK) return st;
    if (M > 16) return CQ_ERR_SHAPE;
    if (M == 0 || N == 0) return CQ_OK;
    if (Wp == nullptr || xq == nullptr || y == nullptr) return CQ_ERR_INVALID_ARG;
    if (!aligned16(Wp) || !aligned4(xq) || !aligned16(y)) return CQ_ERR_ALIGNMENT;
    cq::DeviceInfo dev;
    if (cq::device_info(&dev) != cudaSuccess) return CQ_ERR_CUDA;
    const int need = cq::gemv_packed_smem(w_fmt, static_cast<int>(M), K);
    if (need > (dev.smem_optin < 227 * 1024 ? dev.smem_optin : 227 * 1024)) return CQ_ERR_SHAPE;
    cudaError_t e = cq::launch_gemv_packed(dev, w_fmt, static_cast<int>(M), N, K, Wp, xq, y,
                                           static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CQ_OK : CQ_ERR_CUDA;
}

cq_status cq_set_option(cq_option opt, int64_t value) {
    if (opt != CQ_OPT_WEIGHTS_CONST || (value != 0 && value != 1)) return CQ_ERR_INVALID_ARG;
    cq::g_weights_const.store(static_cast<int>(value), std::memory_order_relaxed);
    return CQ_OK;
}

cq_status cq_gemv_x(cq_format w_fmt, int64_t M, int64_t N, int64_t K, const void* W, const float* x, void* xq,
                    float* y, void* stream) {
    if (!is_weight_fmt(w_fmt)) return CQ_ERR_UNSUPPORTED_FORMAT;
    cq_status st = check_shape(M, N, K);
    if (st != CQ_OK) return st;
    if (M > 16 || !fmt_shape_ok(w_fmt, K)) return CQ_ERR_SHAPE;
    if (M == 0) return CQ_OK;
    if (x == nullptr || xq == nullptr || (N > 0 && (W == nullptr || y == nullptr))) return CQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq) || (N > 0 && (!aligned16(W) || !aligned16(y)))) return CQ_ERR_ALIGNMENT;
    cq::DeviceInfo dev;
    if (cq::device_info(&dev) != cudaSuccess) return CQ_ERR_CUDA;
    cudaError_t e = cq::launch_gemv(dev, w_fmt, static_cast<int>(M), N, K, W, xq, y, x,
                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CQ_OK : CQ_ERR_CUDA;
}

cq_status cq_gemv_swiglu(cq_format w_fmt, int64_t M, int64_t F, int64_t K, const void* W_gate, const void* W_up,
                         const void* xq, float* h, void* stream) {
    if (!is_weight_fmt(w_fmt)) return CQ_ERR_UNSUPPORTED_FORMAT;
    cq_status st = check_shape(M, F, K);
    if (st != CQ_OK) return st;
    if (M < 1 || M > 16 || F < 1 || !fmt_shape_ok(w_fmt, K)) return CQ_ERR_SHAPE;
    const int64_t ce = w_fmt == CQ_Q4_K || w_fmt == CQ_Q5_K || w_fmt == CQ_Q6_K ? 256 : 128;
    if (2 * (K / ce) > 512) return CQ_ERR_SHAPE;
    if (W_gate == nullptr || W_up == nullptr || xq == nullptr || h == nullptr) return CQ_ERR_INVALID_ARG;
    if (!aligned16(W_gate) || !aligned16(W_up) || !aligned4(xq) || !aligned16(h)) return CQ_ERR_ALIGNMENT;
    cq::DeviceInfo dev;
    if (cq::device_info(&dev) != cudaSuccess) return CQ_ERR_CUDA;
    cudaError_t e = cq::launch_gemv_swiglu(dev, w_fmt, static_cast<int>(M), F, K, W_gate, W_up, xq, h,
                                           static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CQ_OK : CQ_ERR_CUDA;
}

cq_status cq_selftest_wait_timeout(int64_t limit_ns, int32_t* out_code, void* stream) {
    if (out_code == nullptr || limit_ns < 1000 || limit_ns > 1000000000) return CQ_ERR_INVALID_ARG;
    cq::DeviceInfo dev;
    if (cq::device_info(&dev) != cudaSuccess) return CQ_ERR_CUDA;
    if (cq::launch_wait_timeout_probe(static_cast<uint64_t>(limit_ns), dev.status,
                                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return CQ_ERR_CUDA;
    return cq_read_global_status(out_code, 1);
}

cq_status cq_read_global_status(int32_t* out_code, int clear) {
    if (out_code == nullptr) return CQ_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return CQ_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_cq_status, sizeof v) != cudaSuccess) return CQ_ERR_CUDA;
    if (clear) {
        const int z = 0;
        if (cudaMemcpyToSymbol(g_cq_status, &z, sizeof z) != cudaSuccess) return CQ_ERR_CUDA;
    }
    *out_code = v;
    return v ? CQ_ERR_TIMEOUT : CQ_OK;
}

}  // extern "C"

namespace {

// cq_gemm formats: Q4_K and the 32-element formats (their activation rows are
// read by TMA, so xq must be 16-byte aligned), all on tcgen05 kernels that
// take an optional workspace (cq_gemm_ws).
bool is_gemm_fmt(int f) { return f == CQ_Q4_K || f == CQ_Q4_0 || f == CQ_Q4_1 || f == CQ_Q8_0; }

// with_ws: the caller's workspace (cq_gemm_ws). Otherwise scratch = true takes
// the workspace from the library's pool when it can (cq_gemm), and false never
// allocates (cq_gemm_noalloc).
cq_status gemm_common(cq_format w_fmt, int64_t M, int64_t N, int64_t K, const void* W, const void* xq, float* y,
                      void* workspace, size_t workspace_bytes, bool with_ws, void* stream, bool scratch = false) {
    if (!is_gemm_fmt(w_fmt)) return CQ_ERR_UNSUPPORTED_FORMAT;
    cq_status st = check_shape(M, N, K);
    if (st != CQ_OK) return st;
    if (M > (int64_t(1) << 31) - 1) return CQ_ERR_SHAPE;
    if (M == 0 || N == 0) return CQ_OK;
    if (W == nullptr || xq == nullptr || y == nullptr) return CQ_ERR_INVALID_ARG;
    const size_t need = with_ws ? cq::gemm_workspace_size(w_fmt, M, K) : 0;
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return CQ_ERR_WORKSPACE;
    const bool xq_ok = w_fmt == CQ_Q4_K ? aligned4(xq) : aligned16(xq);
    if (!aligned16(W) || !xq_ok || !aligned16(y)) return CQ_ERR_ALIGNMENT;
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return CQ_ERR_ALIGNMENT;
    cq::DeviceInfo dev;
    if (cq::device_info(&dev) != cudaSuccess) return CQ_ERR_CUDA;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* ws = need > 0 ? workspace : nullptr;
    void* own = !with_ws && scratch ? cq::scratch_alloc(cq::gemm_workspace_size(w_fmt, M, K), s) : nullptr;
    if (own != nullptr) ws = own;
    const cudaError_t e = w_fmt == CQ_Q4_K ? cq::launch_gemm(dev, w_fmt, M, N, K, W, xq, y, ws, s)
                                           : cq::launch_gemm_tc32(dev, w_fmt, M, N, K, W, xq, y, ws, s);
    const cudaError_t f = cq::scratch_free(own, s);
    return e == cudaSuccess && f == cudaSuccess ? CQ_OK : CQ_ERR_CUDA;
}

}  // namespace

extern "C" {

cq_status cq_gemm(cq_format w_fmt, int64_t M, int64_t N, int64_t K, const void* W, const void* xq, float* y,
                  void* stream) {
    return gemm_common(w_fmt, M, N, K, W, xq, y, nullptr, 0, false, stream, true);
}

cq_status cq_gemm_noalloc(cq_format w_fmt, int64_t M, int64_t N, int64_t K, const void* W, const void* xq, float* y,
                          void* stream) {
    return gemm_common(w_fmt, M, N, K, W, xq, y, nullptr, 0, false, stream, false);
}

size_t cq_gemm_workspace_size(cq_format w_fmt, int64_t M, int64_t N, int64_t K) {
    if (!is_gemm_fmt(w_fmt) || check_shape(M, N, K) != CQ_OK) return 0;
    return cq::gemm_workspace_size(w_fmt, M, K);
}

cq_status cq_gemm_ws(cq_format w_fmt, int64_t M, int64_t N, int64_t K, const void* W, const void* xq, float* y,
                     void* workspace, size_t workspace_bytes, void* stream) {
    return gemm_common(w_fmt, M, N, K, W, xq, y, workspace, workspace_bytes, true, stream);
}

}  // extern "C"

extern "C" {

static cq_status moe_check_shape(int64_t T, int64_t K, int64_t F, int64_t E, int64_t topk) {
    if (T < 0 || K < 0 || F < 0 || E < 0 || topk < 0) return CQ_ERR_INVALID_ARG;
    if (K == 0 || K % 256 != 0 || K > 4096) return CQ_ERR_SHAPE;
    if (F == 0 || F % 256 != 0 || F > 8192) return CQ_ERR_SHAPE;
    if (E < 1 || E > 256 || topk < 1 || topk > E) return CQ_ERR_SHAPE;
    if (T * topk > (int64_t(1) << 20)) return CQ_ERR_SHAPE;
    return CQ_OK;
}

size_t cq_moe_workspace_size(int64_t T, int64_t K, int64_t F, int64_t E, int64_t topk) {
    if (moe_check_shape(T, K, F, E, topk) != CQ_OK) return 0;
    return cq::moe_layout(T, K, F, E, topk).total;
}

cq_status cq_moe_workspace_offsets(int64_t T, int64_t K, int64_t F, int64_t E, int64_t topk, size_t* status_off,
                                   size_t* h_off, size_t* hq_off) {
    cq_status st = moe_check_shape(T, K, F, E, topk);
    if (st != CQ_OK) return st;
    if (status_off == nullptr || h_off == nullptr || hq_off == nullptr) return CQ_ERR_INVALID_ARG;
    const cq::MoeLayout L = cq::moe_layout(T, K, F, E, topk);
    *status_off = L.status;
    *h_off = L.h;
    *hq_off = L.hq;
    return CQ_OK;
}

cq_status cq_moe_gemv(cq_format w_fmt, int64_t T, int64_t K, int64_t F, int64_t E, int64_t topk, const void* W_gate,
                      const void* W_up, const void* W_down, const int32_t* expert_ids, const float* route_w,
                      const void* xq, float* y, void* workspace, size_t workspace_bytes, void* stream) {
    if (w_fmt != CQ_Q4_0) return CQ_ERR_UNSUPPORTED_FORMAT;
    cq_status st = moe_check_shape(T, K, F, E, topk);
    if (st != CQ_OK) return st;
    if (T == 0) return CQ_OK;
    if (!W_gate || !W_up || !W_down || !expert_ids || !route_w || !xq || !y) return CQ_ERR_INVALID_ARG;
    if (workspace == nullptr || workspace_bytes < cq::moe_layout(T, K, F, E, topk).total) return CQ_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return CQ_ERR_ALIGNMENT;
    for (const void* q : {W_gate, W_up, W_down, static_cast<const void*>(expert_ids),
                          static_cast<const void*>(route_w), xq, static_cast<const void*>(y)})
        if (!aligned16(q)) return CQ_ERR_ALIGNMENT;
    cq::DeviceInfo dev;
    if (cq::device_info(&dev) != cudaSuccess) return CQ_ERR_CUDA;
    cudaError_t e = cq::launch_moe(dev, static_cast<int>(T), static_cast<int>(K), static_cast<int>(F),
                                   static_cast<int>(E), static_cast<int>(topk), W_gate, W_up, W_down, expert_ids,
                                   route_w, xq, y, workspace, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CQ_OK : CQ_ERR_CUDA;
}

cq_status cq_read_device_status(const void* workspace, int32_t* out_code, void* stream) {
    if (out_code == nullptr) return CQ_ERR_INVALID_ARG;
    if (workspace != nullptr) return cq_moe_read_status(workspace, out_code, stream);
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return CQ_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_cq_status, sizeof v) != cudaSuccess) return CQ_ERR_CUDA;
    const int z = 0;
    if (v != 0 && cudaMemcpyToSymbol(g_cq_status, &z, sizeof z) != cudaSuccess) return CQ_ERR_CUDA;
    *out_code = v;
    if (v & CQ_DEV_WAIT_TIMEOUT) return CQ_ERR_TIMEOUT;
    return v ? CQ_ERR_DEVICE_STATUS : CQ_OK;
}

cq_status cq_moe_read_status(const void* workspace, int32_t* out_code, void* stream) {
    if (workspace == nullptr || out_code == nullptr) return CQ_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return CQ_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return CQ_ERR_CUDA;
    *out_code = v;
    if (v & CQ_DEV_WAIT_TIMEOUT) return CQ_ERR_TIMEOUT;
    return v ? CQ_ERR_DEVICE_STATUS : CQ_OK;
}

}  // extern "C"
