"""cq_gemv_swiglu (gate and up projections of a dense SwiGLU FFN in one
launch) against the oracle, and against silu(g) * u formed from cq_gemv's own
g and u.

Shapes cover every way the kernel splits a paired row: whole rows several to
an item (small K), a gate/up boundary on a segment edge (K = 4096 at 128
elements per chunk), a boundary inside a segment (K = 14336), one Q4_K item
per row pair (K = 4096), ragged F, and M from 1 to 16.
"""
import numpy as np
import pytest

from gemm_gguf_block_gb300 import synth
from helpers import TOL, W_NAMES, cq_built, dev, torch_cuda

# silu of a large negative g: exp(-g) overflows to inf and g / inf = -0, as intended
pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore:overflow encountered in exp")]

CASES = [(2, 37, 256), (8, 300, 256), (8, 130, 4096), (8, 64, 14336), (3, 129, 4096), (12, 77, 4096),
         (12, 40, 2048), (2, 96, 2048), (3, 33, 768)]


def _silu_mul(g, u):
    return g / (1.0 + np.exp(-g)) * u


def _bound(aux):
    """|dh| from the g, u bounds (TOL * sum|terms| each) carried through
    silu(g) * u: |d silu/dg| <= 1.1, plus the fp32 rounding of the four steps."""
    g, u, ag, au = aux[..., 0], aux[..., 1], aux[..., 2], aux[..., 3]
    dg, du = TOL * ag, TOL * au
    s = np.abs(g / (1.0 + np.exp(-g)))
    return 1.1 * dg * (np.abs(u) + du) + s * du + 1e-6 * np.abs(_silu_mul(g, u)) + 1e-30


@pytest.mark.parametrize("wfmt,F,K", CASES)
@pytest.mark.parametrize("M", [1, 3, 16])
def test_swiglu_matches_oracle_and_gemv(orc, wfmt, F, K, M):
    torch = torch_cuda()
    cq = cq_built()
    rng = np.random.default_rng(wfmt * 1009 + F * 31 + K + M)
    Wg = synth.GEN[W_NAMES[wfmt]](rng, F, K)
    Wu = synth.GEN[W_NAMES[wfmt]](rng, F, K)
    x = rng.standard_normal((M, K)).astype(np.float32)
    xq = orc.quantize(orc.ACT_FOR[wfmt], x)
    tg, tu, txq = dev(torch, Wg), dev(torch, Wu), dev(torch, xq)
    h = cq.gemv_swiglu_t(tg, tu, txq, wfmt, K).cpu().numpy().astype(np.float64)

    h_ref, aux = orc.swiglu(wfmt, Wg, Wu, xq, K)
    err = np.abs(h - h_ref)
    bound = _bound(aux)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3g}"

    # g and u inside the kernel are cq_gemv's: the fused result is silu(g) * u of
    # those values up to the fp32 rounding of the combination.
    g = np.stack([cq.gemv_t(tg, txq[m:m + 1], wfmt, K).cpu().numpy()[0] for m in range(M)]).astype(np.float64)
    u = np.stack([cq.gemv_t(tu, txq[m:m + 1], wfmt, K).cpu().numpy()[0] for m in range(M)]).astype(np.float64)
    want = _silu_mul(g, u)
    assert np.all(np.abs(h - want) <= 1e-6 * np.abs(want) + 1e-30)

