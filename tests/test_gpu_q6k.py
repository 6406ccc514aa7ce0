"""Q6_K weights (x Q8_K) through cq_gemv, cq_gemv_x and cq_gemv_swiglu
against the oracle.

* Random weights, M = 1..16, ragged N, K from one item of whole rows to
  many segments (K up to the 65536 limit): |y - y_ref| <= 2e-5 * sum|terms|,
  and each row of a multi-token call equal to the single-token call bit
  for bit.
* Exact-arithmetic inputs (d = 2^-8, small scales, activations on a 2^-6
  grid): every fp32 evaluation order is exact, so y equals the oracle bit for
  bit -- the six-bit unpack and the integer sub-block dots through the kernel.
* The fused quantise (cq_gemv_x) and the paired SwiGLU call take Q6_K too.
"""
import numpy as np
import pytest

from gemm_gguf_block_gb300 import synth
from helpers import TOL, assert_within, cq_built, dev, torch_cuda

pytestmark = pytest.mark.gpu

Q6K = 14


@pytest.mark.parametrize("N,K", [(1, 2048), (33, 2048), (257, 4096), (100, 14336), (40, 16384), (20, 65536)])
def test_q6k_matches_oracle(orc, N, K):
    torch = torch_cuda()
    cq = cq_built()
    rng = np.random.default_rng(N * 13 + K)
    W = synth.gen_q6_k(rng, N, K)
    x = rng.standard_normal((16, K)).astype(np.float32)
    xq = orc.quantize(orc.Q8_K, x)
    Wd, xd = dev(torch, W), dev(torch, xq)
    y_ref, at = orc.matmul(Q6K, W, xq, K)
    y1 = np.stack([cq.gemv_t(Wd, xd[m:m + 1], Q6K, K).cpu().numpy()[0] for m in range(16)])
    assert_within(y1, y_ref, at, what=f"q6_k {N}x{K} M=1")
    for M in (2, 5, 16):
        yM = cq.gemv_t(Wd, xd[:M], Q6K, K).cpu().numpy()
        assert np.array_equal(yM.view(np.uint32), y1[:M].view(np.uint32)), f"M={M} rows differ from M=1"


@pytest.mark.parametrize("N,K,M", [(37, 2048, 3), (300, 4096, 1)])
def test_q6k_exact_arithmetic(orc, N, K, M):
    torch = torch_cuda()
    cq = cq_built()
    rng = np.random.default_rng(K + M)
    ns = K // 256
    W = synth.pack_q6_k(np.full((N, ns), 0x1C00, np.uint16), rng.integers(-2, 3, (N, ns, 16)),
                        rng.integers(0, 64, (N, K)))
    q = rng.integers(-127, 128, (M, K))
    q.reshape(M, ns, 256)[:, :, 0] = 127
    x = (q * 2.0 ** -6).astype(np.float32)
    xq = cq.quantize_act_t(dev(torch, x), cq.Q8_K)
    xq_np = xq.cpu().numpy()
    assert np.array_equal(xq_np, orc.quantize(orc.Q8_K, x))
    y_ref, at = orc.matmul(Q6K, W, xq_np, K)
    # terms are multiples of 2^-14; below 2^10 in sum every fp32 order is exact
    assert at.max() < 2.0 ** 10, "test precondition: partial sums must stay exact in fp32"
    y = cq.gemv_t(dev(torch, W), xq, Q6K, K).cpu().numpy()
    assert np.array_equal(y.astype(np.float64), y_ref)


@pytest.mark.parametrize("M", [1, 3])
def test_q6k_gemv_x_equals_quantize_then_gemv(orc, M):
    torch = torch_cuda()
    cq = cq_built()
    rng = np.random.default_rng(M)
    N, K = 70, 4096
    W = dev(torch, synth.gen_q6_k(rng, N, K))
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[0, :256] = 0.0                                  # an all-zero superblock
    xd = dev(torch, x)
    y, xq = cq.gemv_x_t(W, xd, Q6K)
    xq_ref = cq.quantize_act_t(xd, cq.Q8_K)
    y_ref = cq.gemv_t(W, xq_ref, Q6K, K)
    assert np.array_equal(xq.cpu().numpy(), xq_ref.cpu().numpy())
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_ref.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("F,K,M", [(45, 2048, 1), (64, 14336, 4)])
def test_q6k_swiglu(orc, F, K, M):
    torch = torch_cuda()
    cq = cq_built()
    rng = np.random.default_rng(F + K)
    Wg, Wu = synth.gen_q6_k(rng, F, K), synth.gen_q6_k(rng, F, K)
    x = rng.standard_normal((M, K)).astype(np.float32)
    xq = orc.quantize(orc.Q8_K, x)
    tg, tu, txq = dev(torch, Wg), dev(torch, Wu), dev(torch, xq)
    h = cq.gemv_swiglu_t(tg, tu, txq, Q6K, K).cpu().numpy().astype(np.float64)
    g = np.stack([cq.gemv_t(tg, txq[m:m + 1], Q6K, K).cpu().numpy()[0] for m in range(M)]).astype(np.float64)
    u = np.stack([cq.gemv_t(tu, txq[m:m + 1], Q6K, K).cpu().numpy()[0] for m in range(M)]).astype(np.float64)
    want = g / (1.0 + np.exp(-g)) * u
    assert np.all(np.abs(h - want) <= 1e-6 * np.abs(want) + 1e-30)
    h_ref, aux = orc.swiglu(Q6K, Wg, Wu, xq, K)
    gg, uu = aux[..., 0], aux[..., 1]
    bound = 1.1 * TOL * aux[..., 2] * (np.abs(uu) + TOL * aux[..., 3]) + \
        np.abs(gg / (1.0 + np.exp(-gg))) * TOL * aux[..., 3] + 1e-6 * np.abs(h_ref) + 1e-30
    assert np.all(np.abs(h - h_ref) <= bound)
