"""cq_gemv / cq_gemm on the GPU against the CPU oracle.

* Random GGUF weights and activations, every format, M = 1..16 tokens, ragged
  N, K from one chunk to multi-segment rows: |y - y_ref| <= 2e-5 * sum|terms|.
* Exact-arithmetic inputs (power-of-two scales, partial sums far below 2^24):
  every fp32 evaluation order is exact, so y must equal the oracle bit for bit
  -- this pins the integer block dots themselves through the real kernels.
* Each row of a multi-token call equals the single-token call bit for bit, and
  cq_gemm rows equal cq_gemv rows bit for bit (the fixed evaluation order).
"""
import numpy as np
import pytest

from gemm_gguf_block_gb300 import synth
from helpers import W_NAMES, assert_within, cq_built, dev, torch_cuda

pytestmark = pytest.mark.gpu

FMTS = [2, 3, 8, 12]
SHAPES = [(1, 256), (33, 512), (100, 768), (257, 2048), (64, 8448), (40, 16640)]


def _case(orc, wfmt, N, K, M, seed):
    rng = np.random.default_rng(seed)
    W = synth.GEN[W_NAMES[wfmt]](rng, N, K)
    x = rng.standard_normal((M, K)).astype(np.float32)
    xq = orc.quantize(orc.ACT_FOR[wfmt], x)
    return W, xq


@pytest.mark.parametrize("wfmt", FMTS)
@pytest.mark.parametrize("N,K", SHAPES)
def test_gemv_matches_oracle(orc, wfmt, N, K):
    torch = torch_cuda()
    cq = cq_built()
    W, xq = _case(orc, wfmt, N, K, 16, seed=wfmt * 7919 + N * 31 + K)
    y_ref, at = orc.matmul(wfmt, W, xq, K)
    Wd, xd = dev(torch, W), dev(torch, xq)
    y1 = np.stack([cq.gemv_t(Wd, xd[m:m + 1], wfmt, K).cpu().numpy()[0] for m in range(16)])
    assert_within(y1, y_ref, at, what=f"fmt {wfmt} M=1")
    for M in (2, 3, 5, 8, 11, 16):
        yM = cq.gemv_t(Wd, xd[:M], wfmt, K).cpu().numpy()
        assert np.array_equal(yM.view(np.uint32), y1[:M].view(np.uint32)), f"M={M} rows differ from M=1"


def _exact_case(wfmt, N, K, M, rng):
    """Weights with scales 2^-8 (and mins / offsets on the same grid), activations
    x = q * 2^-6 with |q| <= 127 and one 127 per block, so d_x = 2^-6 exactly."""
    nb = K // 32
    if wfmt == 2:
        W = synth.pack_q4_0(np.full((N, nb), 0x1C00, np.uint16), rng.integers(0, 16, (N, K)))
    elif wfmt == 8:
        W = synth.pack_q8_0(np.full((N, nb), 0x1C00, np.uint16), rng.integers(-127, 128, (N, K)))
    elif wfmt == 3:
        m = (rng.integers(-16, 17, (N, nb)) * 2.0 ** -8).astype(np.float16).view(np.uint16)
        W = synth.pack_q4_1(np.full((N, nb), 0x1C00, np.uint16), m, rng.integers(0, 16, (N, K)))
    else:
        ns = K // 256
        W = synth.pack_q4_k(np.full((N, ns), 0x1C00, np.uint16), np.full((N, ns), 0x1800, np.uint16),
                            rng.integers(0, 16, (N, ns, 8)), rng.integers(0, 16, (N, ns, 8)),
                            rng.integers(0, 16, (N, K)))
    q = rng.integers(-127, 128, (M, K))
    bs = 256 if wfmt == 12 else 32
    q.reshape(M, K // bs, bs)[:, :, 0] = 127
    x = (q * 2.0 ** -6).astype(np.float32)
    return W, x


@pytest.mark.parametrize("wfmt", FMTS)
@pytest.mark.parametrize("N,K,M", [(37, 512, 3), (300, 1024, 1), (64, 2048, 16)])
def test_gemv_exact_arithmetic(orc, wfmt, N, K, M):
    torch = torch_cuda()
    cq = cq_built()
    rng = np.random.default_rng(wfmt * 101 + K)
    W, x = _exact_case(wfmt, N, K, M, rng)
    xd = dev(torch, x)
    xq = cq.quantize_act_t(xd, cq.ACT_FOR[wfmt])
    xq_np = xq.cpu().numpy()
    assert np.array_equal(xq_np, orc.quantize(orc.ACT_FOR[wfmt], x))
    y_ref, at = orc.matmul(wfmt, W, xq_np, K)
    # Every term is a multiple of 2^-15; with sum|terms| < 2^(24-15) any fp32
    # evaluation order is exact, so the results must agree exactly.
    assert at.max() < 2.0 ** 9, "test precondition: partial sums must stay exact in fp32"
    y = cq.gemv_t(dev(torch, W), xq, wfmt, K).cpu().numpy()
    assert np.array_equal(y.astype(np.float64), y_ref)
    y2 = cq.gemm_t(dev(torch, W), xq, wfmt, K).cpu().numpy()
    assert np.array_equal(y2.astype(np.float64), y_ref)
    y3 = cq.gemm_ws_t(dev(torch, W), xq, wfmt, K).cpu().numpy()
    assert np.array_equal(y3.astype(np.float64), y_ref)


@pytest.mark.parametrize("wfmt", FMTS)
@pytest.mark.parametrize("M,N,K", [(1, 33, 256), (17, 100, 512), (64, 257, 2048), (65, 129, 768),
                                   (130, 96, 4096), (200, 300, 1024), (300, 200, 512), (700, 130, 256)])
def test_gemm_rows_equal_gemv(orc, wfmt, M, N, K):
    """cq_gemm (tcgen05 kernels for Q4_K and for the 32-element formats) against
    the oracle; cq_gemm_ws and cq_gemm_noalloc (the kernels that convert the
    activations in every CTA) give its bits; each row against the single-token
    cq_gemv bit for bit;
    M and N ragged against the 64-token / 128-row tiles. For Q4_K the token
    tile counts 1, 2, 3 and 6 cover single CTAs (odd counts) and CTA pairs
    sharing the weight conversion (even counts, one and three pairs)."""
    torch = torch_cuda()
    cq = cq_built()
    W, xq = _case(orc, wfmt, N, K, M, seed=wfmt * 31 + M + N + K)
    Wd, xd = dev(torch, W), dev(torch, xq)
    y = cq.gemm_t(Wd, xd, wfmt, K).cpu().numpy()
    y_ref, at = orc.matmul(wfmt, W, xq, K)
    assert_within(y, y_ref, at, what=f"gemm fmt {wfmt}")
    y_ws = cq.gemm_ws_t(Wd, xd, wfmt, K).cpu().numpy()
    assert np.array_equal(y.view(np.uint32), y_ws.view(np.uint32)), "cq_gemm_ws differs from cq_gemm"
    y_na = cq.gemm_noalloc_t(Wd, xd, wfmt, K).cpu().numpy()
    assert np.array_equal(y.view(np.uint32), y_na.view(np.uint32)), "cq_gemm_noalloc differs from cq_gemm"
    for m in sorted({0, 1, M // 2, M - 1} & set(range(M))):
        y1 = cq.gemv_t(Wd, xd[m:m + 1], wfmt, K).cpu().numpy()[0]
        assert np.array_equal(y[m].view(np.uint32), y1.view(np.uint32)), f"row {m}"
    if M >= 16:
        y16 = cq.gemv_t(Wd, xd[:16], wfmt, K).cpu().numpy()
        assert np.array_equal(y[:16].view(np.uint32), y16.view(np.uint32)), "batched GEMV rows differ"


@pytest.mark.parametrize("N,Ms", [(8200, (6, 7, 8, 9)), (300, (7, 8, 10, 11))])
def test_q4k_many_token_gemv_route(orc, N, Ms):
    """cq_gemv sends Q4_K calls with many tokens to the prefill GEMM (with the
    library's pooled workspace from M = 7 when N >= 8192 and from M = 8 below;
    without one from M = 9 and M = 11): both sides of each switch give the
    single-token rows bit for bit and agree with the oracle."""
    torch = torch_cuda()
    cq = cq_built()
    K = 1024
    W, xq = _case(orc, 12, N, K, 16, seed=N)
    Wd, xd = dev(torch, W), dev(torch, xq)
    y1 = np.stack([cq.gemv_t(Wd, xd[m:m + 1], 12, K).cpu().numpy()[0] for m in range(max(Ms))])
    for M in Ms:
        yM = cq.gemv_t(Wd, xd[:M], 12, K).cpu().numpy()
        assert np.array_equal(yM.view(np.uint32), y1[:M].view(np.uint32)), f"M={M} rows differ from M=1"
    y_ref, at = orc.matmul(12, W, xq[:max(Ms)], K)
    assert_within(y1, y_ref, at, what=f"q4_k {N}x{K}")


@pytest.mark.parametrize("wfmt", FMTS)
def test_zero_scales_and_empty(orc, wfmt):
    torch = torch_cuda()
    cq = cq_built()
    N, K, M = 50, 1024, 4
    W, xq = _case(orc, wfmt, N, K, M, seed=5)
    bs, bb = orc.BLOCK[wfmt]
    Wz = W.copy().reshape(N, K // bs, bb)
    Wz[:, :, 0:2] = 0
    if wfmt in (3, 12):
        Wz[:, :, 2:4] = 0
    y = cq.gemv_t(dev(torch, Wz.reshape(N, -1)), dev(torch, xq), wfmt, K).cpu().numpy()
    assert np.all(y == 0)
    # N = 0 and M = 0 are no-ops that touch nothing
    out = torch.full((4,), 7.0, device="cuda")
    assert cq.cq_gemv(wfmt, 0, N, K, dev(torch, W).data_ptr(), 0, out.data_ptr()) == cq.OK
    assert cq.cq_gemv(wfmt, M, 0, K, 0, dev(torch, xq).data_ptr(), out.data_ptr()) == cq.OK
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


def test_output_guard_bytes(orc):
    """Writes stay inside y: guard values around a ragged output survive."""
    torch = torch_cuda()
    cq = cq_built()
    N, K, M = 77, 2048, 3
    W, xq = _case(orc, 8, N, K, M, seed=9)
    buf = torch.full((M * N + 64,), 12345.0, device="cuda")
    y = buf[32:32 + M * N].view(M, N)
    assert y.data_ptr() % 16 == 0
    cq.gemv_t(dev(torch, W), dev(torch, xq), 8, K, out=y)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:32] == 12345.0) and np.all(b[32 + M * N:] == 12345.0)
    y_ref, at = orc.matmul(8, W, xq, K)
    assert_within(y.cpu().numpy(), y_ref, at)


def test_no_device_status(orc):
    torch_cuda()
    cq = cq_built()
    st, code = cq.cq_read_global_status(1)
    assert st == cq.OK and code == 0


def test_weights_const_option_same_bits(orc):
    """Prefetching weights ahead of the dependency wait changes no result: a
    chain of quantise -> GEMV calls, each GEMV's activation produced by the
    kernel right before it, gives the same bits with the option on and off."""
    torch = torch_cuda()
    cq = cq_built()
    rng = np.random.default_rng(7)
    shapes = [(4096, 4096), (1024, 4096), (2048, 8192)]
    Ws = [dev(torch, synth.gen_q8_0(rng, N, K)) for N, K in shapes]
    xs = [dev(torch, rng.standard_normal((1, K)).astype(np.float32)) for _, K in shapes]

    def run():
        outs = []
        for W, x, (N, K) in zip(Ws, xs, shapes):
            xq = cq.quantize_act_t(x, cq.Q8_0)
            outs.append(cq.gemv_t(W, xq, cq.Q8_0, K))
        torch.cuda.synchronize()
        return [o.cpu().numpy() for o in outs]

    try:
        assert cq.cq_set_option(cq.OPT_WEIGHTS_CONST, 0) == cq.OK
        a = run()
        assert cq.cq_set_option(cq.OPT_WEIGHTS_CONST, 1) == cq.OK
        b = run()
    finally:
        cq.cq_set_option(cq.OPT_WEIGHTS_CONST, 0)
    for u, v in zip(a, b):
        assert np.array_equal(u.view(np.uint32), v.view(np.uint32))


@pytest.mark.parametrize("wfmt", FMTS)
@pytest.mark.parametrize("N,K", [(33, 512), (100, 768), (257, 2048), (64, 8448)])
@pytest.mark.parametrize("M", [1, 3, 16])
def test_gemv_x_equals_quantize_then_gemv(orc, wfmt, N, K, M):
    """cq_gemv_x writes the bytes cq_quantize_act writes and the y cq_gemv computes, bit for bit."""
    torch = torch_cuda()
    cq = cq_built()
    rng = np.random.default_rng(N * 7 + K + M)
    W = dev(torch, synth.GEN[W_NAMES[wfmt]](rng, N, K))
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[0, :32] = 0.0                                  # an all-zero block
    xd = dev(torch, x)
    y, xq = cq.gemv_x_t(W, xd, wfmt)
    xq_ref = cq.quantize_act_t(xd, cq.ACT_FOR[wfmt])
    y_ref = cq.gemv_t(W, xq_ref, wfmt, K)
    assert np.array_equal(xq.cpu().numpy(), xq_ref.cpu().numpy())
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_ref.cpu().numpy().view(np.uint32))
    assert np.array_equal(xq.cpu().numpy(), orc.quantize(orc.ACT_FOR[wfmt], x))


def test_gemv_x_quantize_only():
    torch = torch_cuda()
    cq = cq_built()
    x = dev(torch, np.random.default_rng(3).standard_normal((2, 1024)).astype(np.float32))
    xq = torch.zeros((2, cq.row_bytes(cq.Q8_0, 1024)), dtype=torch.uint8, device="cuda")
    assert cq.cq_gemv_x(cq.Q4_0, 2, 0, 1024, None, x.data_ptr(), xq.data_ptr(), None,
                        torch.cuda.current_stream().cuda_stream) == cq.OK
    assert torch.equal(xq, cq.quantize_act_t(x, cq.Q8_0))


def test_bounded_wait_times_out_and_device_keeps_working(orc):
    """The bounded wait every kernel uses gives up after its limit and reports
    CQ_DEV_WAIT_TIMEOUT (no fault, no hang); a GEMV afterwards is still right."""
    torch = torch_cuda()
    cq = cq_built()
    st, code = cq.cq_selftest_wait_timeout(50_000_000)          # 50 ms
    assert st == cq.ERR_TIMEOUT and code & cq.DEV_WAIT_TIMEOUT
    st, code = cq.cq_read_global_status(clear=0)
    assert st == cq.OK and code == 0                            # the self-test cleared it
    W, xq = _case(orc, 8, 100, 512, 1, seed=9)
    y = cq.gemv_t(dev(torch, W), dev(torch, xq), 8, 512).cpu().numpy()
    y_ref, at = orc.matmul(8, W, xq, 512)
    assert_within(y, y_ref, at, what="after timeout")


@pytest.mark.parametrize("wfmt", FMTS)
def test_gemv_largest_k(orc, wfmt):
    """K at the library's limit (65536): rows split into many segments."""
    torch = torch_cuda()
    cq = cq_built()
    N, K = 20, 65536
    W, xq = _case(orc, wfmt, N, K, 2, seed=17)
    y = cq.gemv_t(dev(torch, W), dev(torch, xq), wfmt, K).cpu().numpy()
    y_ref, at = orc.matmul(wfmt, W, xq, K)
    assert_within(y, y_ref, at, what=f"K={K}")
    y1 = cq.gemv_t(dev(torch, W), dev(torch, xq[1:2]), wfmt, K).cpu().numpy()[0]
    assert np.array_equal(y[1].view(np.uint32), y1.view(np.uint32))


@pytest.mark.parametrize("wfmt", [2, 3, 8])
@pytest.mark.parametrize("tail", ["ragged", "empty_box"])
def test_batched_gemv_long_tiles(orc, wfmt, tail):
    """Row counts that make the batched tensor-core GEMV take its long tiles
    (448 rows of 14 warps x 32 for up to 8 tokens with Q4_1, 224 rows of 7 x 32
    for Q4_0, 192 rows of 12 x 16 for up to 16 tokens): one tile of 448 rows
    per SM, the last one ragged, or with its second 224-row box wholly past N.
    Sampled rows against the oracle, every row of M = 2..16 bit for bit equal
    to M = 1."""
    torch = torch_cuda()
    cq = cq_built()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N = sms * 448 - 37 if tail == "ragged" else (sms - 1) * 448 + 100
    K = 512
    W, xq = _case(orc, wfmt, N, K, 16, seed=wfmt * 31 + N)
    Wd, xd = dev(torch, W), dev(torch, xq)
    single = np.stack([cq.gemv_t(Wd, xd[m:m + 1], wfmt, K).cpu().numpy()[0] for m in range(16)])
    idx = np.unique(np.concatenate([np.arange(0, 500), np.arange(N - 700, N),
                                    np.linspace(0, N - 1, 200).astype(np.int64)]))
    y_ref, at = orc.matmul(wfmt, W[idx], xq, K)
    assert_within(single[:, idx], y_ref, at, what=f"fmt {wfmt} N={N} M=1")
    for M in (2, 4, 8, 9, 16):
        yM = cq.gemv_t(Wd, xd[:M], wfmt, K).cpu().numpy()
        assert np.array_equal(yM.view(np.uint32), single[:M].view(np.uint32)), f"M={M} rows differ from M=1"


@pytest.mark.parametrize("wfmt,M,N,K", [(12, 130, 300, 1024), (12, 9, 8200, 512), (2, 70, 200, 512)])
def test_gemm_under_graph_capture(orc, wfmt, M, N, K):
    """cq_gemm (and cq_gemv's Q4_K route to it at M = 9) captured into a CUDA
    graph: the library's pool is not used while the stream is capturing, so the
    graph holds the allocation-free kernels; its replay gives the bits of the
    eager call, which took its workspace from the pool."""
    torch = torch_cuda()
    cq = cq_built()
    W, xq = _case(orc, wfmt, N, K, M, seed=wfmt * 5 + M + N)
    Wd, xd = dev(torch, W), dev(torch, xq)
    call = (lambda out: cq.gemv_t(Wd, xd, wfmt, K, out=out)) if M <= 16 else \
        (lambda out: cq.gemm_t(Wd, xd, wfmt, K, out=out))
    y_eager = call(None).clone()
    cq.gemm_noalloc_t(Wd, xd, wfmt, K)        # the allocation-free kernels' attributes set outside capture
    torch.cuda.synchronize()
    y = torch.zeros_like(y_eager)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(y)
    for _ in range(2):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy().view(np.uint32), y_eager.cpu().numpy().view(np.uint32))
