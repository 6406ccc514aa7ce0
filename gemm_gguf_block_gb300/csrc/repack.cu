// Offline weight repack (cq_repack) into the packed layout the batched GEMV
// streams: cera README, "Qualcomm Hexagon" -> "Accelerated Kernels" (Q4_0 /
// Q8_0 weights repacked into tiles once, at load); alice-llm docs, "Phase 6 ->
// Block-Packed Weight Layout" (rows interleaved so that one load serves
// several rows).
//
// The layout (include/cq.h): rows in groups of 16, K in segments of 4 blocks;
// unit (group G, segment s) of 64 * BB bytes at byte (s * ceil(N/16) + G) *
// 64 * BB, segment-major so that a tile of consecutive groups is one contiguous
// copy. Inside a unit: the 16 rows' scale fields of the 4 blocks, then per
// (half h, row r, lane t) the quant words 16h + 4t .. 16h + 4t + 3 of blocks
// 0..3 as one aligned 16-byte piece -- the four bytes an mma.sync fragment
// lane t takes from each block (mma_frag.cuh), so one 16-byte load gives a lane
// its quants of four blocks. Rows at or past N are zero.
#include <cstdint>

#include "cq.h"
#include "cq_internal.h"

namespace cq {
namespace {

template <int WF> struct RepackFmt;
template <> struct RepackFmt<CQ_Q4_0> { static constexpr int BB = 18, QO = 2, SC = 2, HALVES = 1; };
template <> struct RepackFmt<CQ_Q4_1> { static constexpr int BB = 20, QO = 4, SC = 4, HALVES = 1; };
template <> struct RepackFmt<CQ_Q8_0> { static constexpr int BB = 34, QO = 2, SC = 2, HALVES = 2; };

// Four bytes at any byte address (the GGUF blocks of 18 and 34 bytes are only
// 2-byte aligned).
__device__ __forceinline__ uint32_t ld_bytes4(const uint8_t* p) {
    return static_cast<uint32_t>(p[0]) | static_cast<uint32_t>(p[1]) << 8 | static_cast<uint32_t>(p[2]) << 16 |
           static_cast<uint32_t>(p[3]) << 24;
}

// One CTA of 64 threads per unit at a time: thread (r, t) = (row of the
// group, lane) writes that row's lane-t quant pieces and block t's scale field.
template <int WF>
__global__ void __launch_bounds__(64) repack_kernel(const uint8_t* __restrict__ W, uint8_t* __restrict__ P, int64_t N,
                                                    int64_t wrow, int64_t ngroups, int64_t units) {
    using R = RepackFmt<WF>;
    constexpr int UNIT = 64 * R::BB, QUANTS = 64 * R::SC;
    const int r = threadIdx.x >> 2, t = threadIdx.x & 3;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int64_t s = u / ngroups, G = u - s * ngroups;
        const int64_t row = 16 * G + r;
        uint8_t* dst = P + u * UNIT;
        const uint8_t* seg = row < N ? W + row * wrow + 4 * s * R::BB : nullptr;
#pragma unroll
        for (int h = 0; h < R::HALVES; ++h)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t v = seg ? ld_bytes4(seg + j * R::BB + R::QO + 16 * h + 4 * t) : 0u;
                *reinterpret_cast<uint32_t*>(dst + QUANTS + h * 1024 + ((4 * r + t) * 4 + j) * 4) = v;
            }
        uint8_t* sc = dst + r * 4 * R::SC + t * R::SC;
#pragma unroll
        for (int i = 0; i < R::SC; ++i) sc[i] = seg ? seg[t * R::BB + i] : 0;
    }
}

template <int WF>
cudaError_t launch_repack_fmt(int64_t N, int64_t K, const void* W, void* Wp, cudaStream_t s) {
    using R = RepackFmt<WF>;
    const int64_t ngroups = (N + 15) / 16, units = ngroups * (K / 128);
    const int64_t grid = units < 65536 ? units : 65536;
    repack_kernel<WF><<<static_cast<unsigned>(grid), 64, 0, s>>>(static_cast<const uint8_t*>(W),
                                                                  static_cast<uint8_t*>(Wp), N, K / 32 * R::BB,
                                                                  ngroups, units);
    return cudaGetLastError();
}

}  // namespace

int64_t repack_size(int w_fmt, int64_t N, int64_t K) {
    const int64_t bb = w_fmt == CQ_Q4_0 ? 18 : w_fmt == CQ_Q4_1 ? 20 : w_fmt == CQ_Q8_0 ? 34 : 0;
    if (bb == 0 || N < 0 || K <= 0 || K % 256 != 0) return 0;
    return (N + 15) / 16 * (K / 128) * 64 * bb;
}

cudaError_t launch_repack(int w_fmt, int64_t N, int64_t K, const void* W, void* Wp, cudaStream_t s) {
    switch (w_fmt) {
    case CQ_Q4_0: return launch_repack_fmt<CQ_Q4_0>(N, K, W, Wp, s);
    case CQ_Q4_1: return launch_repack_fmt<CQ_Q4_1>(N, K, W, Wp, s);
    case CQ_Q8_0: return launch_repack_fmt<CQ_Q8_0>(N, K, W, Wp, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace cq
