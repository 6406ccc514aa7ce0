"""cq_repack and cq_gemv_packed on the GPU.

* The repacked bytes equal the oracle's repack (a byte permutation: bit-exact),
  for every format, with ragged N (zero padding rows) and multi-segment K.
* cq_gemv_packed against the oracle on the original weights (2e-5 * sum|terms|)
  and bit for bit against cq_gemv on the original weights, for M = 1..16, on
  small and ragged shapes, on row counts that take the long tiles, and on the
  full Q4_1 LM head; K at the largest value the kernel takes, and the shape
  error just beyond it.
"""
import numpy as np
import pytest

from gemm_gguf_block_gb300 import synth
from helpers import W_NAMES, assert_within, cq_built, dev, torch_cuda

pytestmark = pytest.mark.gpu

FMTS = [2, 3, 8]


def _case(orc, wfmt, N, K, M, seed):
    rng = np.random.default_rng(seed)
    W = synth.GEN[W_NAMES[wfmt]](rng, N, K)
    x = rng.standard_normal((M, K)).astype(np.float32)
    xq = orc.quantize(orc.ACT_FOR[wfmt], x)
    return W, xq


@pytest.mark.parametrize("wfmt", FMTS)
@pytest.mark.parametrize("N,K", [(1, 256), (17, 512), (300, 1024), (64, 8448)])
def test_repack_bytes_equal_oracle(orc, wfmt, N, K):
    torch = torch_cuda()
    cq = cq_built()
    W, _ = _case(orc, wfmt, N, K, 1, seed=wfmt * 13 + N + K)
    Wp = cq.repack_t(dev(torch, W), wfmt, K).cpu().numpy()
    ref = orc.repack(wfmt, W, K)
    assert Wp.size == ref.size == cq.cq_repack_size(wfmt, N, K)
    assert np.array_equal(Wp, ref)


def _check_packed(orc, cq, torch, wfmt, N, K, Ms, seed, idx=None):
    W, xq = _case(orc, wfmt, N, K, max(Ms), seed)
    Wd, xd = dev(torch, W), dev(torch, xq)
    Wp = cq.repack_t(Wd, wfmt, K)
    rows = slice(None) if idx is None else idx
    y_ref, at = orc.matmul(wfmt, W if idx is None else W[idx], xq, K)
    for M in Ms:
        yp = cq.gemv_packed_t(Wp, xd[:M], wfmt, N, K).cpu().numpy()
        yg = cq.gemv_t(Wd, xd[:M], wfmt, K).cpu().numpy()
        assert np.array_equal(yp.view(np.uint32), yg.view(np.uint32)), f"fmt {wfmt} M={M}: packed != cq_gemv"
        assert_within(yp[:, rows], y_ref[:M], at[:M], what=f"fmt {wfmt} N={N} K={K} M={M} packed")


@pytest.mark.parametrize("wfmt", FMTS)
@pytest.mark.parametrize("N,K", [(1, 256), (33, 512), (300, 1024), (257, 2048)])
def test_gemv_packed_small(orc, wfmt, N, K):
    torch = torch_cuda()
    cq = cq_built()
    _check_packed(orc, cq, torch, wfmt, N, K, (1, 2, 3, 5, 8, 9, 16), seed=wfmt * 7 + N * 3 + K)


@pytest.mark.parametrize("wfmt", FMTS)
def test_gemv_packed_long_tiles(orc, wfmt):
    """One tile of 224 rows (up to 8 tokens) or 192 rows (up to 16) per SM and
    more; the last tile's groups past N are not copied."""
    torch = torch_cuda()
    cq = cq_built()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N, K = sms * 224 * 2 - 37, 512
    idx = np.unique(np.concatenate([np.arange(0, 300), np.arange(N - 500, N),
                                    np.linspace(0, N - 1, 200).astype(np.int64)]))
    _check_packed(orc, cq, torch, wfmt, N, K, (1, 4, 8, 12, 16), seed=wfmt + 5, idx=idx)


@pytest.mark.parametrize("wfmt", FMTS)
def test_gemv_packed_largest_k(orc, wfmt):
    """The largest K the kernel takes for every format (10752 at M <= 8, 5376 at
    M <= 16) runs; the next step past a format's limit is a shape error."""
    torch = torch_cuda()
    cq = cq_built()
    _check_packed(orc, cq, torch, wfmt, 40, 10752, (1, 8), seed=wfmt + 11)
    _check_packed(orc, cq, torch, wfmt, 40, 5376, (16,), seed=wfmt + 12)
    limit8 = {2: 11776, 3: 11008, 8: 10752}[wfmt]
    limit16 = {2: 5888, 3: 5376, 8: 5376}[wfmt]
    for M, K in ((8, limit8 + 256), (16, limit16 + 256)):
        Wp = torch.zeros(cq.cq_repack_size(wfmt, 16, K), dtype=torch.uint8, device="cuda")
        xq = torch.zeros((M, cq.row_bytes(cq.ACT_FOR[wfmt], K)), dtype=torch.uint8, device="cuda")
        y = torch.empty((M, 16), dtype=torch.float32, device="cuda")
        st = cq.cq_gemv_packed(wfmt, M, 16, K, Wp.data_ptr(), xq.data_ptr(), y.data_ptr(), 0)
        assert st == cq.ERR_SHAPE, (M, K, st)


def test_gemv_packed_lm_head(orc):
    """The full Q4_1 LM head, 128256 x 4096: every row of M = 1, 4, 8, 16 on the
    packed weights equals cq_gemv on the GGUF weights bit for bit; sampled rows
    against the oracle."""
    torch = torch_cuda()
    cq = cq_built()
    W, x = synth.lm_head_q4_1(0)
    N, K = W.shape[0], x.shape[1]
    Wd = dev(torch, W)
    Wp = cq.repack_t(Wd, cq.Q4_1, K)
    xq = cq.quantize_act_t(dev(torch, x), cq.Q8_1)
    idx = np.unique(np.concatenate([[0, 1, 15, 16, 223, 224, N // 2, N - 17, N - 16, N - 1],
                                    np.linspace(0, N - 1, 40).astype(np.int64)]))
    y_ref, at = orc.matmul(cq.Q4_1, W[idx], xq.cpu().numpy(), K)
    for M in (1, 4, 8, 16):
        yp = cq.gemv_packed_t(Wp, xq[:M], cq.Q4_1, N, K).cpu().numpy()
        yg = cq.gemv_t(Wd, xq[:M], cq.Q4_1, K).cpu().numpy()
        assert np.array_equal(yp.view(np.uint32), yg.view(np.uint32)), f"M={M}"
        assert_within(yp[:, idx], y_ref[:M], at[:M], what=f"lm head packed M={M}")


def test_packed_empty_calls():
    torch = torch_cuda()
    cq = cq_built()
    assert cq.cq_gemv_packed(cq.Q4_1, 0, 8, 256, 0, 0, 0, 0) == cq.OK
    assert cq.cq_gemv_packed(cq.Q4_1, 4, 0, 256, 0, 0, 0, 0) == cq.OK
    assert cq.cq_repack(cq.Q4_1, 0, 256, 0, 0, 0) == cq.OK
    torch.cuda.synchronize()
