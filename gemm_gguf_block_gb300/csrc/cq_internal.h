// Host-side launchers shared between the C-ABI translation unit and the
// kernel translation units. Arguments are validated by the caller (cq_api.cu).
#pragma once
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

namespace cq {

// Programmatic dependent launch: every kernel of the library is launched so that it may start while the previous grid in the
// stream is still running; each kernel's first act is griddepcontrol.wait
// (pdl_wait), which returns once the grids it depends on have completed and
// their memory is visible, before any global memory is read or written. The
// launch latency and the kernel's setup thus overlap the previous kernel's
// tail, with the same ordering guarantees as a plain launch.
// CQ_OPT_WEIGHTS_CONST (see include/cq.h).
bool weights_const();

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_kernel with thread-block clusters of shape `cluster` (grid a
// multiple of it in every dimension).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                  dim3 cluster, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster.x;
    attr[1].val.clusterDim.y = cluster.y;
    attr[1].val.clusterDim.z = cluster.z;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct DeviceInfo {
    int sm_count;
    int smem_optin;   // max dynamic shared memory per block (bytes)
    int* status;      // device address of the library status word
};

// Cached per-device properties; status address from cudaGetSymbolAddress.
cudaError_t device_info(DeviceInfo* out);

// Stream-ordered scratch from the library's per-device memory pool: bytes on
// `s` (256-byte aligned), or nullptr when the pool cannot supply them or the
// stream is being captured (callers then take an allocation-free path).
// scratch_free(p, s) returns it on `s` after the work queued before it.
void* scratch_alloc(size_t bytes, cudaStream_t s);
cudaError_t scratch_free(void* p, cudaStream_t s);

// Raises `kernel`'s dynamic shared-memory limit on the current device to at
// least `bytes` (cudaFuncSetAttribute), once per (device, kernel); safe to
// call from several host threads.
cudaError_t raise_smem_limit(const void* kernel, int bytes);

cudaError_t launch_quantize(int act_fmt, int64_t M, int64_t K, const float* x, void* xq, cudaStream_t s);

// Bounded-wait self-test (cq_selftest_wait_timeout).
cudaError_t launch_wait_timeout_probe(uint64_t limit_ns, int* status, cudaStream_t s);

// With x (fp32 [M][K]) non-null the activations are quantized on the way
// (cq_gemv_x): xq receives them and y is the same as from xq.
cudaError_t launch_gemv(const DeviceInfo& dev, int w_fmt, int M, int64_t N, int64_t K, const void* W,
                        const void* xq, float* y, const float* x, cudaStream_t s);

// Paired gate / up GEMV of a dense SwiGLU FFN: h = silu(Wg . xq) * (Wu . xq),
// each product as launch_gemv computes it (the dp4a kernel, any M <= 16).
cudaError_t launch_gemv_swiglu(const DeviceInfo& dev, int w_fmt, int M, int64_t F, int64_t K, const void* Wg,
                               const void* Wu, const void* xq, float* h, cudaStream_t s);

// Tensor-core batched GEMV (2 <= M <= 16; Q4_0, Q4_1, Q8_0) and the shared
// memory it needs (0 when the format has no such path).
int gemv_mma_smem(int w_fmt, int M, int64_t K);
cudaError_t launch_gemv_mma(const DeviceInfo& dev, int w_fmt, int M, int64_t N, int64_t K, const void* W,
                            const void* xq, float* y, cudaStream_t s);

// The same kernel on weights in the packed layout of cq_repack (1 <= M <= 16),
// the shared memory it needs at least, and the repack itself.
int gemv_packed_smem(int w_fmt, int M, int64_t K);
cudaError_t launch_gemv_packed(const DeviceInfo& dev, int w_fmt, int M, int64_t N, int64_t K, const void* Wp,
                               const void* xq, float* y, cudaStream_t s);
int64_t repack_size(int w_fmt, int64_t N, int64_t K);
cudaError_t launch_repack(int w_fmt, int64_t N, int64_t K, const void* W, void* Wp, cudaStream_t s);

// Prefill GEMM (any M): y rows equal the cq_gemv rows bit for bit. With a
// workspace (gemm_workspace_size bytes, 256-byte aligned) the activations are
// converted once up front instead of in every CTA.
size_t gemm_workspace_size(int w_fmt, int64_t M, int64_t K);
cudaError_t launch_gemm(const DeviceInfo& dev, int w_fmt, int64_t M, int64_t N, int64_t K, const void* W,
                        const void* xq, float* y, void* workspace, cudaStream_t s);

// Prefill GEMM of the 32-element formats (Q4_0, Q4_1, Q8_0; any M) on
// tcgen05, one tensor-memory accumulator per 32-block; y rows equal the
// cq_gemv rows bit for bit. With a workspace (gemm32_workspace_size bytes,
// 256-byte aligned) the activation operand images are built once per call;
// without one (workspace == nullptr) every CTA builds its own.
size_t gemm32_workspace_size(int w_fmt, int64_t M, int64_t K);
cudaError_t launch_gemm_tc32(const DeviceInfo& dev, int w_fmt, int64_t M, int64_t N, int64_t K, const void* W,
                             const void* xq, float* y, void* workspace, cudaStream_t s);

// Byte offsets of the routed-FFN workspace sections (each 256-byte aligned).
struct MoeLayout {
    size_t status;   // int32 status word (CQ_DEV_* bits)
    size_t offs;     // int32 [E+1]: start of each expert's pair list in perm
    size_t order;    // int32 [E]: experts by decreasing pair count (ties by id)
    size_t perm;     // int32 [T*topk]: pair indices (t*topk + s) grouped by expert
    size_t valid;    // int32 [T*topk]: 1 if the pair's expert id was accepted
    size_t h;        // fp32 [T*topk][F]: hidden activations, (token, slot) order
    size_t hq;       // Q8_0 [T*topk] rows of F/32 blocks
    size_t out;      // fp32 [T*topk][K]: per-pair down-projection outputs
    size_t total;
};
MoeLayout moe_layout(int64_t T, int64_t K, int64_t F, int64_t E, int64_t topk);

// Grouped tensor-core projections of the routed FFN: gate/up + SwiGLU into h,
// Q8_0 of h into hq, down into o (all in the caller's workspace). CTAs take
// the experts in `order` (largest first).
cudaError_t launch_moe_projections(const DeviceInfo& dev, int T, int K, int F, int E, int topk, const void* Wg,
                                   const void* Wu, const void* Wd, const void* xq, const int* offs, const int* order,
                                   const int* perm, float* h, const void* hq, float* o, cudaStream_t s);

cudaError_t launch_moe(const DeviceInfo& dev, int T, int K, int F, int E, int topk, const void* Wg,
                       const void* Wu, const void* Wd, const int32_t* ids, const float* rw, const void* xq,
                       float* y, void* ws, cudaStream_t s);

}  // namespace cq
