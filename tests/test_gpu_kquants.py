"""Q5_K and Q6_K weights (x Q8_K) through cq_gemv, cq_gemv_x and
cq_gemv_swiglu against the oracle.

* Random weights, M = 1..16, ragged N, K from one item of whole rows to
  many segments (K up to the 65536 limit): |y - y_ref| <= 2e-5 * sum|terms|,
  and each row of a multi-token call equal to the single-token call bit
  for bit.
* Exact-arithmetic inputs (d = 2^-8, small scales, activations on a 2^-6
  grid): every fp32 evaluation order is exact, so y equals the oracle bit for
  bit -- the five- and six-bit unpacks and the integer sub-block dots
  through the kernel.
* The fused quantise (cq_gemv_x) and the paired SwiGLU call take them too.
"""
import numpy as np
import pytest

from gemm_gguf_block_gb300 import synth
from helpers import TOL, assert_within, cq_built, dev, torch_cuda

# silu of a large negative g: exp(-g) overflows to inf and g / inf = -0, as intended
pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore:overflow encountered in exp")]

Q5K, Q6K = 13, 14
GEN = {Q5K: synth.gen_q5_k, Q6K: synth.gen_q6_k}
SHAPES = [(1, 2048), (33, 2048), (257, 4096), (100, 14336), (40, 16384), (20, 65536)]


@pytest.mark.parametrize("N,K", SHAPES + [(64, 256), (17, 768)])
@pytest.mark.parametrize("wfmt", [Q5K, Q6K])
def test_kquant_matches_oracle(orc, wfmt, N, K):
    if wfmt == Q6K and K % 2048:
        pytest.skip("Q6_K takes K % 2048 == 0")
    torch = torch_cuda()
    cq = cq_built()
    rng = np.random.default_rng(N * 13 + K + wfmt)
    W = GEN[wfmt](rng, N, K)
    x = rng.standard_normal((16, K)).astype(np.float32)
    xq = orc.quantize(orc.Q8_K, x)
    Wd, xd = dev(torch, W), dev(torch, xq)
    y_ref, at = orc.matmul(wfmt, W, xq, K)
    y1 = np.stack([cq.gemv_t(Wd, xd[m:m + 1], wfmt, K).cpu().numpy()[0] for m in range(16)])
    assert_within(y1, y_ref, at, what=f"fmt {wfmt} {N}x{K} M=1")
    for M in (2, 5, 16):
        yM = cq.gemv_t(Wd, xd[:M], wfmt, K).cpu().numpy()
        assert np.array_equal(yM.view(np.uint32), y1[:M].view(np.uint32)), f"M={M} rows differ from M=1"


@pytest.mark.parametrize("N,K,M", [(37, 2048, 3), (300, 4096, 1)])
@pytest.mark.parametrize("wfmt", [Q5K, Q6K])
def test_kquant_exact_arithmetic(orc, wfmt, N, K, M):
    torch = torch_cuda()
    cq = cq_built()
    rng = np.random.default_rng(K + M + wfmt)
    ns = K // 256
    if wfmt == Q6K:
        W = synth.pack_q6_k(np.full((N, ns), 0x1C00, np.uint16), rng.integers(-2, 3, (N, ns, 16)),
                            rng.integers(0, 64, (N, K)))
    else:
        # d = 2^-8, dmin = 2^-9, scales / mins < 4
        W = synth.pack_q5_k(np.full((N, ns), 0x1C00, np.uint16), np.full((N, ns), 0x1800, np.uint16),
                            rng.integers(0, 4, (N, ns, 8)), rng.integers(0, 4, (N, ns, 8)),
                            rng.integers(0, 32, (N, K)))
    q = rng.integers(-127, 128, (M, K))
    q.reshape(M, ns, 256)[:, :, 0] = 127
    x = (q * 2.0 ** -6).astype(np.float32)
    xq = cq.quantize_act_t(dev(torch, x), cq.Q8_K)
    xq_np = xq.cpu().numpy()
    assert np.array_equal(xq_np, orc.quantize(orc.Q8_K, x))
    y_ref, at = orc.matmul(wfmt, W, xq_np, K)
    # terms are multiples of 2^-14 (Q6_K) or 2^-15 (the Q5_K mins); below
    # 2^24 grid steps in sum every fp32 order is exact
    step = 14 if wfmt == Q6K else 15
    assert at.max() < 2.0 ** (24 - step), "test precondition: partial sums must stay exact in fp32"
    y = cq.gemv_t(dev(torch, W), xq, wfmt, K).cpu().numpy()
    assert np.array_equal(y.astype(np.float64), y_ref)


@pytest.mark.parametrize("M", [1, 3])
@pytest.mark.parametrize("wfmt", [Q5K, Q6K])
def test_kquant_gemv_x_equals_quantize_then_gemv(orc, wfmt, M):
    torch = torch_cuda()
    cq = cq_built()
    rng = np.random.default_rng(M + wfmt)
    N, K = 70, 4096
    W = dev(torch, GEN[wfmt](rng, N, K))
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[0, :256] = 0.0                                  # an all-zero superblock
    xd = dev(torch, x)
    y, xq = cq.gemv_x_t(W, xd, wfmt)
    xq_ref = cq.quantize_act_t(xd, cq.Q8_K)
    y_ref = cq.gemv_t(W, xq_ref, wfmt, K)
    assert np.array_equal(xq.cpu().numpy(), xq_ref.cpu().numpy())
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_ref.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("F,K,M", [(45, 2048, 1), (64, 14336, 4)])
@pytest.mark.parametrize("wfmt", [Q5K, Q6K])
def test_kquant_swiglu(orc, wfmt, F, K, M):
    torch = torch_cuda()
    cq = cq_built()
    rng = np.random.default_rng(F + K + wfmt)
    Wg, Wu = GEN[wfmt](rng, F, K), GEN[wfmt](rng, F, K)
    x = rng.standard_normal((M, K)).astype(np.float32)
    xq = orc.quantize(orc.Q8_K, x)
    tg, tu, txq = dev(torch, Wg), dev(torch, Wu), dev(torch, xq)
    h = cq.gemv_swiglu_t(tg, tu, txq, wfmt, K).cpu().numpy().astype(np.float64)
    g = np.stack([cq.gemv_t(tg, txq[m:m + 1], wfmt, K).cpu().numpy()[0] for m in range(M)]).astype(np.float64)
    u = np.stack([cq.gemv_t(tu, txq[m:m + 1], wfmt, K).cpu().numpy()[0] for m in range(M)]).astype(np.float64)
    want = g / (1.0 + np.exp(-g)) * u
    assert np.all(np.abs(h - want) <= 1e-6 * np.abs(want) + 1e-30)
    h_ref, aux = orc.swiglu(wfmt, Wg, Wu, xq, K)
    gg, uu = aux[..., 0], aux[..., 1]
    bound = 1.1 * TOL * aux[..., 2] * (np.abs(uu) + TOL * aux[..., 3]) + \
        np.abs(gg / (1.0 + np.exp(-gg))) * TOL * aux[..., 3] + 1e-6 * np.abs(h_ref) + 1e-30
    assert np.all(np.abs(h - h_ref) <= bound)
