// Prefill GEMM entry (any M). Until the tensor-core kernel lands, tokens are
// taken sixteen at a time through the GEMV kernel, which follows the same
// fixed evaluation order, so every row is the cq_gemv row bit for bit.
#include <algorithm>

#include "cq_device.cuh"
#include "cq_internal.h"

namespace cq {

cudaError_t launch_gemm(const DeviceInfo& dev, int w_fmt, int64_t M, int64_t N, int64_t K, const void* W,
                        const void* xq, float* y, cudaStream_t s) {
    const int64_t act_row = K / CHUNK_ELEMS * achunk_bytes(act_fmt_for(w_fmt));
    for (int64_t m0 = 0; m0 < M; m0 += 16) {
        const int mm = static_cast<int>(std::min<int64_t>(16, M - m0));
        cudaError_t e = launch_gemv(dev, w_fmt, mm, N, K, W, static_cast<const uint8_t*>(xq) + m0 * act_row,
                                    y + m0 * N, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace cq
