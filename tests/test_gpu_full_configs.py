"""The full-size workloads, called as the benchmark calls them, against the
oracle on sampled outputs.

* Q4_0 2048 x 2048 decode GEMV: every row (small enough for the oracle).
* Q8_0 decode suite at Llama-3-8B shapes: the whole GEMV on the GPU with its
  in-step activation quantisation (byte-equal to the oracle's); the oracle
  on a spread of rows of each matrix, including the first and last tiles.
* Q4_K prefill GEMM, M=512 N=14336 K=4096: cq_gemm and cq_gemm_ws over the
  whole problem; the oracle on sampled weight rows for all 512 tokens; the two
  calls equal bit for bit, and sampled tokens equal to their cq_gemv rows.
* Q4_0 / Q4_1 / Q8_0 prefill GEMM, M=512 N=14336 K=4096: sampled rows
  against the oracle, sampled tokens equal to their cq_gemv rows.
* Q4_1 LM head 128256 x 4096 at M = 1, 4, 8, 16: the oracle on sampled rows;
  every row of an M>1 call bitwise equal to the M=1 call of that position.
* Q6_K tied-embedding LM head 128256 x 2048 at M = 1 and 4, the same checks.
"""
import numpy as np
import pytest

from gemm_gguf_block_gb300 import synth
from helpers import assert_within, cq_built, dev, torch_cuda

pytestmark = pytest.mark.gpu


def _rows(N, n_spread=40):
    """Rows to check: both ends, tile boundaries near the start, and a spread."""
    fixed = [0, 1, 2, 127, 128, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1]
    spread = np.linspace(0, N - 1, n_spread).astype(np.int64)
    return np.unique(np.clip(np.concatenate([fixed, spread]), 0, N - 1))


def _oracle_rows(orc, wfmt, W, xq, K, idx):
    y, at = orc.matmul(wfmt, W[idx], xq, K)
    return y, at


def test_decode_q4_0_2048_all_rows(orc):
    torch = torch_cuda()
    cq = cq_built()
    W, x = synth.decode_q4_0_small(0)
    K = x.shape[1]
    xq = cq.quantize_act_t(dev(torch, x), cq.Q8_0)
    assert np.array_equal(xq.cpu().numpy(), orc.quantize(orc.Q8_0, x))
    y = cq.gemv_t(dev(torch, W), xq, cq.Q4_0, K).cpu().numpy()
    y_ref, at = orc.matmul(cq.Q4_0, W, xq.cpu().numpy(), K)
    assert_within(y, y_ref, at, what="q4_0 2048")


@pytest.mark.parametrize("layer", range(len(synth.DECODE_SUITE_Q8_0)))
def test_decode_q8_0_suite_sampled(orc, layer):
    torch = torch_cuda()
    cq = cq_built()
    N, K = synth.DECODE_SUITE_Q8_0[layer]
    W, x = synth.decode_q8_0_layer(0, layer, N, K)
    xq = cq.quantize_act_t(dev(torch, x), cq.Q8_0)
    xq_np = xq.cpu().numpy()
    assert np.array_equal(xq_np, orc.quantize(orc.Q8_0, x)), "in-step quantisation"
    y = cq.gemv_t(dev(torch, W), xq, cq.Q8_0, K).cpu().numpy()
    idx = _rows(N)
    y_ref, at = _oracle_rows(orc, cq.Q8_0, W, xq_np, K, idx)
    assert_within(y[:, idx], y_ref, at, what=f"q8_0 {N}x{K}")


def test_prefill_gemm_sampled(orc):
    torch = torch_cuda()
    cq = cq_built()
    W, x = synth.prefill_q4_k(0)
    M, K = x.shape
    N = W.shape[0]
    xq = cq.quantize_act_t(dev(torch, x), cq.Q8_K)
    xq_np = xq.cpu().numpy()
    assert np.array_equal(xq_np, orc.quantize(orc.Q8_K, x))
    Wd = dev(torch, W)
    y = cq.gemm_t(Wd, xq, cq.Q4_K, K).cpu().numpy()
    y_ws = cq.gemm_ws_t(Wd, xq, cq.Q4_K, K).cpu().numpy()
    assert np.array_equal(y.view(np.uint32), y_ws.view(np.uint32)), "cq_gemm_ws differs from cq_gemm"
    idx = _rows(N, 24)
    y_ref, at = _oracle_rows(orc, cq.Q4_K, W, xq_np, K, idx)
    assert_within(y[:, idx], y_ref, at, what="q4_k gemm")
    for m in (0, 1, 127, 128, 300, M - 1):
        y1 = cq.gemv_t(Wd, xq[m:m + 1], cq.Q4_K, K).cpu().numpy()[0]
        assert np.array_equal(y[m].view(np.uint32), y1.view(np.uint32)), f"token {m}: gemm row != gemv row"


@pytest.mark.parametrize("fmt", ["q4_0", "q4_1", "q8_0"])
def test_prefill_gemm_32_sampled(orc, fmt):
    """The prefill GEMM of a 32-element format at M=512 N=14336 K=4096, with and
    without a workspace."""
    torch = torch_cuda()
    cq = cq_built()
    wfmt = cq.FMT[fmt]
    W, x = synth.prefill_32(fmt, 0)
    M, K = x.shape
    N = W.shape[0]
    xq = cq.quantize_act_t(dev(torch, x), cq.ACT_FOR[wfmt])
    xq_np = xq.cpu().numpy()
    assert np.array_equal(xq_np, orc.quantize(orc.ACT_FOR[wfmt], x))
    Wd = dev(torch, W)
    y = cq.gemm_t(Wd, xq, wfmt, K).cpu().numpy()
    y_ws = cq.gemm_ws_t(Wd, xq, wfmt, K).cpu().numpy()
    assert np.array_equal(y.view(np.uint32), y_ws.view(np.uint32)), "cq_gemm_ws differs from cq_gemm"
    idx = _rows(N, 24)
    y_ref, at = _oracle_rows(orc, wfmt, W, xq_np, K, idx)
    assert_within(y[:, idx], y_ref, at, what=f"{fmt} gemm")
    for m in (0, 1, 63, 64, 300, M - 1):
        y1 = cq.gemv_t(Wd, xq[m:m + 1], wfmt, K).cpu().numpy()[0]
        assert np.array_equal(y[m].view(np.uint32), y1.view(np.uint32)), f"token {m}: gemm row != gemv row"


def test_lm_head_q4_1_batched(orc):
    torch = torch_cuda()
    cq = cq_built()
    W, x = synth.lm_head_q4_1(0)
    K = x.shape[1]
    N = W.shape[0]
    Wd = dev(torch, W)
    xq = cq.quantize_act_t(dev(torch, x), cq.Q8_1)
    xq_np = xq.cpu().numpy()
    assert np.array_equal(xq_np, orc.quantize(orc.Q8_1, x))
    single = [cq.gemv_t(Wd, xq[m:m + 1], cq.Q4_1, K).cpu().numpy()[0] for m in range(16)]
    idx = _rows(N)
    y_ref, at = _oracle_rows(orc, cq.Q4_1, W, xq_np, K, idx)
    assert_within(np.stack(single)[:, idx], y_ref, at, what="q4_1 lm head")
    for M in (4, 8, 16):
        y = cq.gemv_t(Wd, xq[:M], cq.Q4_1, K).cpu().numpy()
        for m in range(M):
            assert np.array_equal(y[m].view(np.uint32), single[m].view(np.uint32)), f"M={M} row {m}"


def test_lm_head_q6_k(orc):
    torch = torch_cuda()
    cq = cq_built()
    W, x = synth.lm_head_q6_k(0)
    K = x.shape[1]
    N = W.shape[0]
    Wd = dev(torch, W)
    xq = cq.quantize_act_t(dev(torch, x), cq.Q8_K)
    xq_np = xq.cpu().numpy()
    assert np.array_equal(xq_np, orc.quantize(orc.Q8_K, x))
    single = [cq.gemv_t(Wd, xq[m:m + 1], cq.Q6_K, K).cpu().numpy()[0] for m in range(4)]
    idx = _rows(N)
    y_ref, at = _oracle_rows(orc, cq.Q6_K, W, xq_np, K, idx)
    assert_within(np.stack(single)[:, idx], y_ref, at, what="q6_k lm head")
    y = cq.gemv_t(Wd, xq[:4], cq.Q6_K, K).cpu().numpy()
    for m in range(4):
        assert np.array_equal(y[m].view(np.uint32), single[m].view(np.uint32)), f"M=4 row {m}"
