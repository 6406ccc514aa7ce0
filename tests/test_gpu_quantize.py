"""Activation quantisation on the GPU vs the oracle: byte-exact."""
import numpy as np
import pytest

from helpers import cq_built, dev, torch_cuda

pytestmark = pytest.mark.gpu


def _inputs(rng, M, K):
    x = rng.standard_normal((M, K))
    if M >= 4:
        x[1] *= 1e-6                              # fp16-subnormal scales
        x[2] *= 3e3
        x[3, : K // 2] = 0.0                      # all-zero blocks
    x = x.astype(np.float32)
    # exact ties: a block whose amax is 127 gives d = 1 and x * (1/d) = x
    if K >= 64:
        x[0, :32] = np.array([127, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5] + [3.5] * 24, np.float32)
    return x


@pytest.mark.parametrize("afmt", [8, 9, 15])
@pytest.mark.parametrize("M,K", [(1, 256), (4, 2048), (7, 4096), (2, 14336), (5, 768)])
def test_quantize_bytes(orc, afmt, M, K):
    torch = torch_cuda()
    cq = cq_built()
    rng = np.random.default_rng(1000 * afmt + K + M)
    x = _inputs(rng, M, K)
    got = cq.quantize_act_t(dev(torch, x), afmt).cpu().numpy()
    want = orc.quantize(afmt, x)
    assert got.shape == want.shape
    assert np.array_equal(got, want), np.argwhere(got != want)[:5]


def test_quantize_large_batch(orc):
    """512 x 4096 (the prefill workload's activation shape) to Q8_K, byte-exact."""
    torch = torch_cuda()
    cq = cq_built()
    from gemm_gguf_block_gb300 import synth
    x = synth.gen_x(synth.stream(0, 3, 1), 512, 4096)
    got = cq.quantize_act_t(dev(torch, x), cq.Q8_K).cpu().numpy()
    assert np.array_equal(got, orc.quantize(orc.Q8_K, x))
