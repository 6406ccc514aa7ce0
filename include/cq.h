/*
 * cq.h -- GGUF block-quantized GEMV / GEMM / routed-expert FFN on NVIDIA GB300.
 *
 * y = W . x where W is stored in a GGUF block format and x is quantized at run
 * time to the paired 8-bit format:
 *
 *     weight format   activation format   block
 *     Q4_0            Q8_0                32 elements
 *     Q8_0            Q8_0                32 elements
 *     Q4_1            Q8_1                32 elements
 *     Q4_K            Q8_K                256 elements
 *     Q5_K            Q8_K                256 elements (GEMV only)
 *     Q6_K            Q8_K                256 elements (GEMV only)
 *
 * Sources (web pages on GGUF inference engines; sections by name):
 *   cera README "Quantization" (weight types; activations quantized to Q8_0
 *   for an integer GEMV); alice-llm docs "Quantization Block Specs" (Q4_K and
 *   Q8_0 block layouts), "Computation Path (Q4_K)" (Q8_K activations and the
 *   Q4_K x Q8_K integer formula), "Phase 4 -- i8 Dynamic Quantization + SDOT"
 *   (per-chunk amax/127 quantisation); cera 0.5 release notes and README
 *   "Other features" (batched LM-head projection over verified positions;
 *   Q4_1 decode matching the batched prefill GEMM bit for bit); cera README
 *   "Supported models" (lfm2moe: 4-of-32 routed experts, grouping tokens by
 *   expert as the follow-up); alice-llm "WGSL Shader Architecture" (fused
 *   gate+up SwiGLU); alice-llm "Quantization Block Specs" (Q6_K = ql[128] +
 *   qh[64] + scales[16] + d per 256 elements), "aarch64 NEON Quantized Matvec
 *   Bench" (qh's bit pairs feed the four quadrants) and cera README (the
 *   tied Q6_K embedding as the LM head). Q6_K element i: half h = i/128,
 *   quadrant q = (i%128)/32, l = i%32; low four bits in ql[64h + l + 32(q&1)]
 *   (low nibble for q < 2, high for q >= 2), high two bits in qh[32h + l]
 *   bits 2q, 2q+1; value = d * (int8)scales[i/16] * (q6 - 32). Q5_K = d +
 *   dmin + scales[12] + qh[32] + qs[128] ("Quantization Block Specs"): Q4_K's
 *   nibbles, scales and mins with bit 4 of element i in qh[i%32], bit i/32.
 *
 * Conventions for every call:
 *   - All data pointers are DEVICE pointers owned by the caller, 16-byte
 *     aligned, except quantized activations (xq) passed to cq_gemv, and to
 *     cq_gemm with Q4_K weights, which need 4-byte alignment (a Q8_K row is
 *     292 bytes per 256 elements). The library never allocates, frees or synchronises on these
 *     paths; every call is asynchronous on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) on the current device.
 *   - Matrices are row-major. A weight row holds the K/blk blocks of one
 *     output row contiguously (GGUF order); activations are M rows of blocks;
 *     outputs are fp32 [M][N] (token-major).
 *   - K must be a positive multiple of 256 (2048 for Q6_K, whose 210-byte
 *     superblocks reach a 16-byte boundary every eight). N == 0 or M == 0 is
 *     a valid no-op.
 *   - Arguments are validated before any launch: an error status means
 *     nothing was launched and nothing was written.
 *   - Results are deterministic and do not depend on the launch shape: each
 *     output is accumulated in one fixed fp32 order (below), so a row of a
 *     multi-token call equals the single-token call bit for bit, and cq_gemv
 *     and cq_gemm agree bit for bit.
 *
 * Fixed fp32 evaluation order (the contract behind the bitwise equalities):
 *   isum = exact int32 dot of the block's quants.
 *   Q4_0/Q8_0 block:  c = fma(D(d_w) * D(d_x), (float)isum, c)
 *   Q4_1 block:       c = fma(D(d_w) * D(d_x), (float)isum, c);
 *                     c = fma(D(m_w), D(s_x), c)
 *   Q4_0/Q4_1/Q8_0: blocks are taken in chunks of four (128 elements); c
 *   starts at 0 for every chunk and takes the chunk's blocks in increasing k;
 *   then y = y + c over the chunks in increasing k, starting from y = 0.
 *   Q4_K, per superblock in increasing k, from y = 0:
 *                     S_j = int dot of sub-block j, isum_sc = sum_j sc_j S_j,
 *                     isum_m = sum_j m_j (bsum_2j + bsum_2j+1),
 *                     t = fma(D(d), (float)isum_sc, -(D(dmin) * (float)isum_m)),
 *                     y = fma(d_x, t, y).
 *   Q5_K: as Q4_K, with the five-bit quants.
 *   Q6_K, per superblock in increasing k, from y = 0:
 *                     S_j = int dot of sub-block j (16 elements) of (q6 - 32)
 *                     with q8, isum = sum_j sc_j S_j, t = D(d) * (float)isum,
 *                     y = fma(d_x, t, y).
 *   Every operation rounds to nearest.
 */
#ifndef CQ_H
#define CQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Block formats, numbered as the GGML tensor-type ids. */
typedef enum {
    CQ_Q4_0 = 2,
    CQ_Q4_1 = 3,
    CQ_Q8_0 = 8,
    CQ_Q8_1 = 9,
    CQ_Q4_K = 12,
    CQ_Q5_K = 13,
    CQ_Q6_K = 14,
    CQ_Q8_K = 15
} cq_format;

typedef enum {
    CQ_OK = 0,
    CQ_ERR_INVALID_ARG = 1,        /* NULL pointer or a negative size */
    CQ_ERR_UNSUPPORTED_FORMAT = 2, /* a format (pairing) this call does not take */
    CQ_ERR_SHAPE = 3,              /* K not a positive multiple of 256, M out of range, too large */
    CQ_ERR_ALIGNMENT = 4,          /* a pointer not aligned as the call requires */
    CQ_ERR_WORKSPACE = 5,          /* workspace missing or smaller than required */
    CQ_ERR_CUDA = 6,               /* a CUDA runtime call or launch failed */
    CQ_ERR_DEVICE_STATUS = 7,      /* a kernel reported bad input (see the status word) */
    CQ_ERR_TIMEOUT = 8             /* a bounded device wait gave up (see the status word) */
} cq_status;

/* Device status word bits (written by kernels, read by the cq_read_* calls). */
#define CQ_DEV_BAD_EXPERT_ID   0x1 /* an expert id outside [0, E): that (token, slot) is skipped */
#define CQ_DEV_DUP_EXPERT_ID   0x2 /* an expert id repeated within a token: the repeat is skipped */
#define CQ_DEV_WAIT_TIMEOUT    0x4 /* a copy-completion wait ran out of iterations */

/*
 * Activation quantisation (alice-llm "Phase 4 -- i8 Dynamic Quantization";
 * cera "Quantization"; alice-llm "Computation Path (Q4_K)" step 1).
 * x: fp32 [M][K] -> xq: M rows of act_fmt blocks, per block (all in fp32):
 *   amax = max|x_i|; d = amax / 127; q_i = round-half-away(x_i * (1/d)),
 *   clamped to [-127, 127] (q = 0 when d = 0).
 *   Q8_0 (34 B / 32): fp16(d), q[32].
 *   Q8_1 (36 B / 32): fp16(d), fp16(d * sum q), q[32].
 *   Q8_K (292 B / 256): fp32 d, q[256], int16 bsum[16] (sums of 16 quants).
 * x must be finite. xq must hold M * K/blk * bytes(blk).
 */
cq_status cq_quantize_act(cq_format act_fmt, int64_t M, int64_t K, const float* x, void* xq,
                          void* stream);

/*
 * Decode GEMV and batched LM-head projection, 1 <= M <= 16 tokens
 * (cera "Other features": the verify path projects all 1+k positions in one
 * batched pass so the head is read once; alice-llm "Batch-4 Speculative
 * Decoding": weights decoded once, one accumulator set per token).
 * w_fmt in {Q4_0, Q8_0, Q4_1, Q4_K, Q5_K, Q6_K}; xq in the paired activation format.
 * W: N rows of K/blk blocks. y: fp32 [M][N]. M > 16 returns CQ_ERR_SHAPE.
 */
cq_status cq_gemv(cq_format w_fmt, int64_t M, int64_t N, int64_t K, const void* W, const void* xq,
                  float* y, void* stream);

/*
 * cq_quantize_act followed by cq_gemv, as one call: x (fp32 [M][K], DEVICE,
 * 16-byte aligned) is quantized to the activation format paired with w_fmt
 * and written to xq (16-byte aligned, M rows of blocks, byte for byte what
 * cq_quantize_act writes), and y = W . xq as cq_gemv computes it, bit for bit.
 * For one token the quantisation happens inside the GEMV kernel (each CTA
 * quantizes the row it needs; the first also writes xq), which takes a
 * launch and a dependency off the decode path. M <= 16; N == 0 only
 * quantizes. Errors as cq_gemv.
 */
cq_status cq_gemv_x(cq_format w_fmt, int64_t M, int64_t N, int64_t K, const void* W, const float* x,
                    void* xq, float* y, void* stream);

/*
 * Gate and up projections of a dense SwiGLU FFN in one pass, and their
 * combination (alice-llm docs "WGSL Shader Architecture": swiglu_fused_q4k;
 * "The GPU Optimization Journey", phase 4: gate and up read in one pass):
 *   g = W_gate . xq,  u = W_up . xq   (each exactly as cq_gemv computes it)
 *   h[m][f] = silu(g) * u = g / (1 + exp(-g)) * u   (fp32: RN divide,
 *             RN add, RN multiply; exp is CUDA's expf)
 * w_fmt in {Q4_0, Q8_0, Q4_1, Q4_K, Q5_K, Q6_K}; xq in the paired activation format;
 * W_gate, W_up: F rows of K/blk blocks each (16-byte aligned); h: fp32
 * [M][F] (16-byte aligned). 1 <= M <= 16 (else CQ_ERR_SHAPE); F >= 1;
 * K a positive multiple of 256 with 2 * K / 128 <= 512 chunks (K <= 32768;
 * Q4_K, Q5_K, Q6_K: K <= 65536). Errors as cq_gemv. g and u never leave the kernel: one
 * launch reads both matrices, combines the two sums of each (row, token) and
 * writes only h.
 */
cq_status cq_gemv_swiglu(cq_format w_fmt, int64_t M, int64_t F, int64_t K, const void* W_gate,
                         const void* W_up, const void* xq, float* h, void* stream);

/*
 * Offline weight repack for the batched decode path (cera README "Qualcomm
 * Hexagon" -> "Accelerated Kernels": weights repacked into tiles once, at
 * load; alice-llm docs "Phase 6 -> Block-Packed Weight Layout": rows
 * interleaved so that one load serves several rows; ggml's "repacked" CPU
 * kernels). w_fmt in {Q4_0, Q4_1, Q8_0}; W: N rows of K/32 blocks (GGUF
 * order), DEVICE, 16-byte aligned; Wp: cq_repack_size(w_fmt, N, K) bytes of
 * DEVICE memory, 16-byte aligned, owned by the caller (0 from cq_repack_size
 * for another format or a K that is not a positive multiple of 256).
 *
 * The packed layout, byte for byte (BB = 18, 20, 34 bytes per block):
 *   - rows in groups of 16 (G = 0 .. ceil(N/16) - 1; rows >= N are zero),
 *     K in segments of 4 blocks (s = 0 .. K/128 - 1);
 *   - the unit (G, s) is 64 * BB bytes at byte (s * ceil(N/16) + G) * 64 * BB
 *     (segment-major: the units of one segment for consecutive groups are
 *     one contiguous range);
 *   - inside a unit, for row r = 0..15 of the group: the scale fields of
 *     blocks j = 0..3 of the segment, in block order (Q4_1: d then m, 4 bytes
 *     per block, 16 per row; Q4_0 / Q8_0: d, 2 bytes per block, 8 per row);
 *   - then, at 64 * (4 or 2) bytes, for half h (Q8_0: 0 and 1; Q4_0 / Q4_1: 0),
 *     row r, lane t = 0..3, block j = 0..3: bytes 16h + 4t .. 16h + 4t + 3 of
 *     block j's quant array (4 bytes each; 16 bytes per (h, r, t)).
 * Total ceil(N/16) * 16 * K/32 * BB bytes: the GGUF bytes plus the zero rows.
 * Asynchronous on `stream`; W is not modified. Errors: CQ_ERR_UNSUPPORTED_FORMAT,
 * CQ_ERR_SHAPE (as cq_gemv), CQ_ERR_INVALID_ARG, CQ_ERR_ALIGNMENT, CQ_ERR_CUDA.
 */
size_t cq_repack_size(cq_format w_fmt, int64_t N, int64_t K);
cq_status cq_repack(cq_format w_fmt, int64_t N, int64_t K, const void* W, void* Wp, void* stream);

/*
 * cq_gemv on repacked weights: Wp as cq_repack wrote it from an N x K matrix
 * W of w_fmt (Q4_0, Q4_1, Q8_0), 16-byte aligned. y equals cq_gemv(W) bit for
 * bit (the same fixed order). 1 <= M <= 16 (M > 16: CQ_ERR_SHAPE). The
 * kernel keeps the tokens' activations in shared memory: CQ_ERR_SHAPE when
 * they and two weight stages do not fit, which every format avoids for K up
 * to 10752 at M <= 8 and up to 5376 at M <= 16. Each stage of the
 * weight stream is one contiguous bulk copy, and each lane reads its quants of
 * four blocks in one 16-byte load instead of one or three loads per block.
 * Errors as cq_gemv.
 */
cq_status cq_gemv_packed(cq_format w_fmt, int64_t M, int64_t N, int64_t K, const void* Wp, const void* xq,
                         float* y, void* stream);

/*
 * Prefill GEMM, any M >= 0 (cera README "Supported models": batched-GEMM
 * prefill; alice-llm "Computation Path (Q4_K)"). Same operands and result as
 * cq_gemv; each row equals the cq_gemv result for that token bit for bit.
 * w_fmt: Q4_K or Q4_0 / Q4_1 / Q8_0 (tcgen05 paths; cera
 * 0.5.3 README "Breaking changes in 0.4.0" holds a Q4_1 decode equal to
 * the batched prefill bit for bit). For Q4_0 / Q4_1 / Q8_0
 * the activation rows are read by TMA, so xq must be 16-byte aligned
 * (CQ_ERR_ALIGNMENT otherwise). M < 2^31. Other formats return
 * CQ_ERR_UNSUPPORTED_FORMAT.
 * Memory: the activation workspace of cq_gemm_ws (cq_gemm_workspace_size
 * bytes) comes from a memory pool the library owns, one per device, created
 * on first use and keeping up to 512 MB between calls. It is allocated
 * (cudaMallocFromPoolAsync) and freed (cudaFreeAsync) on `stream`, around the
 * kernels. While `stream` is being captured into a graph, or when the pool
 * cannot supply the bytes, the call runs cq_gemm_noalloc's kernels instead:
 * same bits either way. cq_gemv routes Q4_K calls here from 7 tokens (8 for
 * matrices of fewer than 8192 rows) when the pool supplies the workspace, and
 * from 9 (11) tokens without it.
 */
cq_status cq_gemm(cq_format w_fmt, int64_t M, int64_t N, int64_t K, const void* W, const void* xq,
                  float* y, void* stream);

/*
 * cq_gemm that never allocates: every CTA converts the activations of its
 * token tile itself instead of reading them once converted from a workspace
 * (slower: Q4_K 512 x 14336 x 4096 157.7 us against about 104 us). Same
 * arguments, errors and bits as cq_gemm.
 */
cq_status cq_gemm_noalloc(cq_format w_fmt, int64_t M, int64_t N, int64_t K, const void* W, const void* xq,
                          float* y, void* stream);

/*
 * cq_gemm with a caller-owned device workspace: the quantized activations are
 * converted once, into the workspace, to the tensor-core operand layout,
 * instead of in every weight tile. Same result, bit for bit, as cq_gemm.
 * cq_gemm_workspace_size returns the bytes needed (0 for an unsupported
 * format or shape): ceil(M/128) * (K/256) * 70144 for Q4_K;
 * ceil(M/64) * (K/128) * 17408 for Q4_0 and Q8_0 (Q8_0 activations) and
 * ceil(M/64) * (K/128) * 18432 for Q4_1 (Q8_1 activations). The workspace
 * must be 256-byte aligned; it is scratch (no state is kept between calls),
 * and two calls that may overlap on the GPU need separate workspaces.
 * Errors as cq_gemm, plus CQ_ERR_WORKSPACE (NULL or too small) and
 * CQ_ERR_ALIGNMENT for a misaligned workspace.
 */
size_t cq_gemm_workspace_size(cq_format w_fmt, int64_t M, int64_t N, int64_t K);
cq_status cq_gemm_ws(cq_format w_fmt, int64_t M, int64_t N, int64_t K, const void* W, const void* xq,
                     float* y, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Routed-expert FFN (cera README "Supported models", lfm2moe; grouping tokens
 * by expert so each expert's weights are read once per call).
 * For token t and slot s: e = expert_ids[t][s] (distinct within a token),
 *   g = W_gate[e] . xq[t],  u = W_up[e] . xq[t]        (F outputs each)
 *   h = silu(g) * u = g / (1 + exp(-g)) * u              (fp32)
 *   hq = Q8_0(h) (the cq_quantize_act rule)
 *   o = W_down[e] . hq                                   (K outputs)
 *   y[t] = route_w[t][0] * o_0, then y[t] = fma(route_w[t][s], o_s, y[t])
 *          for s = 1..topk-1 in slot order.
 * w_fmt: Q4_0. W_gate, W_up: [E][F rows][K]; W_down: [E][K rows][F];
 * xq: Q8_0 [T][K]; expert_ids: int32 [T][topk]; route_w: fp32 [T][topk];
 * y: fp32 [T][K]. K and F positive multiples of 256; 1 <= topk <= E <= 256.
 * workspace: device memory of at least cq_moe_workspace_size(...) bytes,
 * 256-byte aligned, owned by the caller; its status word is cleared by the
 * call. Ids outside [0, E) or repeated within a token are skipped and flagged
 * in the status word (CQ_DEV_*): read it with cq_moe_read_status.
 */
size_t cq_moe_workspace_size(int64_t T, int64_t K, int64_t F, int64_t E, int64_t topk);

cq_status cq_moe_gemv(cq_format w_fmt, int64_t T, int64_t K, int64_t F, int64_t E, int64_t topk,
                      const void* W_gate, const void* W_up, const void* W_down,
                      const int32_t* expert_ids, const float* route_w, const void* xq, float* y,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * Allocation-free variant of cq_moe_gemv. The pages have no counterpart: this
 * is for callers that cannot call cudaMalloc and so cannot supply a
 * workspace -- a plugin whose host framework owns all device memory through
 * its own pool, or a latency-critical loop that cannot afford the device-wide
 * synchronisation of an allocation. The caller still passes every input and
 * the output; the scratch space is a fixed array of CQ_MOE_NOALLOC_MAX_BYTES
 * in the library's device image, held on every GPU that loads the library
 * until the process exits, and shared by every call of this function.
 * - Same arguments, arithmetic and results as cq_moe_gemv (without the
 *   workspace arguments); the array keeps the previous call's contents, and
 *   the call clears what must start at zero (its status word) itself.
 * - Shapes whose cq_moe_workspace_size exceeds CQ_MOE_NOALLOC_MAX_BYTES return
 *   CQ_ERR_WORKSPACE before any launch; shapes cq_moe_gemv rejects return
 *   CQ_ERR_SHAPE. It calls no cudaMalloc, cudaFree or other allocating routine.
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 * - Calls whose executions overlap on the GPU (two streams, or two host
 *   threads on one device) race on the shared array: serialise them.
 * - Expert-id errors are still skipped as in cq_moe_gemv; their status word
 *   lives in the shared array: read it with cq_moe_noalloc_read_status.
 */
#define CQ_MOE_NOALLOC_MAX_BYTES (24u << 20)
cq_status cq_moe_gemv_noalloc(cq_format w_fmt, int64_t T, int64_t K, int64_t F, int64_t E, int64_t topk,
                              const void* W_gate, const void* W_up, const void* W_down,
                              const int32_t* expert_ids, const float* route_w, const void* xq, float* y,
                              void* stream);

/* Synchronises `stream`, then copies the status word of the last
 * cq_moe_gemv_noalloc call on the current device (CQ_DEV_* bits; 0 if none
 * ran) to *out_code; the next call clears it. Return values as for
 * cq_moe_read_status. Allocates nothing. */
cq_status cq_moe_noalloc_read_status(int32_t* out_code, void* stream);

/*
 * Byte offsets inside the MoE workspace, for inspection by tests: the status
 * word (int32), the hidden activations h (fp32 [T*topk][F], in (token, slot)
 * order) and their Q8_0 quantisation hq ([T*topk] rows of F/32 blocks).
 */
cq_status cq_moe_workspace_offsets(int64_t T, int64_t K, int64_t F, int64_t E, int64_t topk,
                                   size_t* status_off, size_t* h_off, size_t* hq_off);

/* Synchronises `stream`, then copies the MoE workspace status word to *out_code.
 * Returns CQ_ERR_DEVICE_STATUS if any CQ_DEV_* bit is set, else CQ_OK. */
cq_status cq_moe_read_status(const void* workspace, int32_t* out_code, void* stream);

/*
 * The status read-out of the boundary: synchronises `stream`, then copies a
 * device status word to *out_code.
 * - workspace != NULL: the status word of a cq_moe_gemv workspace (as
 *   cq_moe_read_status); the next cq_moe_gemv on that workspace clears it.
 * - workspace == NULL: the library's own status word (as
 *   cq_read_global_status with clear = 1: read, then zeroed).
 * Returns CQ_ERR_TIMEOUT if CQ_DEV_WAIT_TIMEOUT is set, CQ_ERR_DEVICE_STATUS
 * if any other CQ_DEV_* bit is set, else CQ_OK; CQ_ERR_INVALID_ARG for a null
 * out_code, CQ_ERR_CUDA if the synchronisation or the copy fails.
 */
cq_status cq_read_device_status(const void* workspace, int32_t* out_code, void* stream);

/* Synchronises the current device, then reads (and, if clear != 0, zeroes) the
 * library's own status word, used by kernels that take no workspace (a copy
 * wait that timed out in cq_gemv / cq_gemm). CQ_ERR_TIMEOUT if set. */
cq_status cq_read_global_status(int32_t* out_code, int clear);

const char* cq_status_string(cq_status s);

/*
 * Self-test of the bounded waits (no counterpart on the pages): launches one
 * thread that waits, with a limit of limit_ns (1e3 .. 1e9 ns), on an mbarrier
 * phase that nothing completes -- as a kernel whose copy never lands would --
 * then reads and clears the library status word like cq_read_global_status.
 * Expected result: CQ_ERR_TIMEOUT with CQ_DEV_WAIT_TIMEOUT in *out_code, and
 * a device that keeps working. Synchronises the current device.
 */
cq_status cq_selftest_wait_timeout(int64_t limit_ns, int32_t* out_code, void* stream);

/*
 * Library-wide options (process-wide, all devices; set them before the calls
 * they should affect, not while calls are being issued from other threads).
 *
 * CQ_OPT_WEIGHTS_CONST (default 0): 1 is the caller's promise that no weight
 * buffer passed to cq_gemv is written by work that may still be in flight on
 * the stream of the call (the weights of an inference model). The GEMV then
 * starts streaming its weight tiles while the preceding kernel in the stream
 * is still finishing, and waits for that kernel only before it reads the
 * activations or writes its output. With 0, every kernel waits for the
 * preceding one before touching any global memory.
 *
 * Returns CQ_ERR_INVALID_ARG for an unknown option or value.
 */
typedef enum { CQ_OPT_WEIGHTS_CONST = 1 } cq_option;
cq_status cq_set_option(cq_option opt, int64_t value);

#ifdef __cplusplus
}
#endif
#endif /* CQ_H */
