"""Routed-expert FFN on the GPU against the CPU oracle.

The hidden activations are re-quantized to Q8_0 between the projections, so
an fp32 h that sits within its rounding error of a quantisation boundary may
legitimately land on either side. The checks therefore go in tiers:

1. h (read from the workspace) within the propagated bound of the exact h:
   TOL * (|silu'(g)| |u| sum|g terms| + |silu(g)| sum|u terms|) plus a few
   fp32 ulps for the silu evaluation.
2. hq (read from the workspace) equals the oracle's Q8_0(h) except at
   elements the oracle itself marks ambiguous: a quant whose x/d lies within
   the tier-1 bound of a rounding boundary, or a whole block whose fp16 scale
   could round either way.
3. y within TOL * sum|terms| plus, per output, the largest change those
   ambiguous elements could make (one quantisation step each, times the down
   weight and the router weight).

Beside tier 2, the down projection and the combine are checked on their own:
the oracle recomputes them from the GPU's own hq bytes (oracle_moe_down), and
y must then lie within TOL * sum|terms| with no allowance at all.
"""
import numpy as np
import pytest

from gemm_gguf_block_gb300 import synth
from helpers import TOL, cq_built, dev, torch_cuda

# silu of a large negative g: exp(-g) overflows to inf and g / inf = -0, as intended
pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore:overflow encountered in exp")]

U32 = 2.0 ** -24


def _q4_0_abs_dequant(W):
    """|value| of every element of Q4_0 rows: [rows, K]."""
    rows = W.shape[0]
    blk = W.reshape(rows, -1, 18)
    d = np.abs(blk[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64))
    qs = blk[:, :, 2:18]
    q = np.concatenate([qs & 15, qs >> 4], axis=2).astype(np.int64) - 8
    return (d[:, :, None] * np.abs(q)).reshape(rows, -1)


def _ambiguity(h, gu, F):
    """Per (pair, element): may the GPU's Q8_0 decision differ from the oracle's?
    Returns (mask [P, F] bool, step [P, F] float)."""
    g, u, ag, au = gu[..., 0], gu[..., 1], gu[..., 2], gu[..., 3]
    sig = 1.0 / (1.0 + np.exp(-g))
    silu = g * sig
    dsilu = np.abs(sig * (1.0 + g * (1.0 - sig)))
    bound = TOL * (dsilu * np.abs(u) * ag + np.abs(silu) * au) + 8 * U32 * np.abs(h) + 1e-30
    P = h.shape[0]
    hb = h.reshape(P, F // 32, 32)
    bb = bound.reshape(P, F // 32, 32)
    amax = np.abs(hb).max(axis=2)
    dmax = np.abs(bb).max(axis=2)
    lo = (np.maximum(amax - dmax, 0) / 127).astype(np.float32).astype(np.float16)
    hi = ((amax + dmax) / 127).astype(np.float32).astype(np.float16)
    d_amb = lo != hi
    d = (amax / 127).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(d[..., None] > 0, hb / d[..., None], 0.0)
        tb = np.where(d[..., None] > 0, bb / d[..., None], 0.0)
    frac = np.abs(t - np.floor(t) - 0.5)
    q_amb = frac <= tb + 3e-5
    mask = q_amb | d_amb[..., None]
    step = np.broadcast_to((hi.astype(np.float64) * 1.001)[..., None], hb.shape)
    return mask.reshape(P, F), step.reshape(P, F)


def _run(orc, T, E, topk, K, F, seed, token_sample=None):
    torch = torch_cuda()
    cq = cq_built()
    if (T, E, topk, K, F) == (256, 32, 4, 2048, 1792):
        Wg, Wu, Wd, ids, rw, x = synth.moe_ffn(seed)
    else:
        rng = np.random.default_rng(seed)
        Wg = np.stack([synth.gen_q4_0(rng, F, K) for _ in range(E)])
        Wu = np.stack([synth.gen_q4_0(rng, F, K) for _ in range(E)])
        Wd = np.stack([synth.gen_q4_0(rng, K, F) for _ in range(E)])
        ids, rw = synth.gen_routing(rng, T, E, topk)
        x = rng.standard_normal((T, K)).astype(np.float32)
    xq = orc.quantize(orc.Q8_0, x)
    y, ws = cq.moe_t(dev(torch, Wg), dev(torch, Wu), dev(torch, Wd), dev(torch, ids), dev(torch, rw),
                     dev(torch, xq), K, F)
    st, code = cq.cq_moe_read_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == cq.OK and code == 0
    st, so, ho, qo = cq.cq_moe_workspace_offsets(T, K, F, E, topk)
    wsn = ws.cpu().numpy()
    P = T * topk
    h_gpu = wsn[ho:ho + 4 * P * F].view(np.float32).reshape(T, topk, F)
    hq_gpu = wsn[qo:qo + P * (F // 32) * 34].reshape(T, topk, -1)
    y = y.cpu().numpy()
    tok = np.arange(T) if token_sample is None else token_sample
    r = orc.moe(Wg, Wu, Wd, ids[tok], rw[tok], xq[tok], K, F)
    return dict(Wd=Wd, ids=ids[tok], rw=rw[tok], y=y[tok], h=h_gpu[tok], hq=hq_gpu[tok], r=r, orc=orc)


def _check(c, K, F):
    r = c["r"]
    T, topk = c["ids"].shape
    P = T * topk
    h_ref = r["h"].reshape(P, F)
    gu = r["gu_aux"].reshape(P, F, 4)
    mask, step = _ambiguity(h_ref, gu, F)
    # tier 1: hidden activations
    g, u, ag, au = gu[..., 0], gu[..., 1], gu[..., 2], gu[..., 3]
    sig = 1.0 / (1.0 + np.exp(-g))
    bound = TOL * (np.abs(sig * (1 + g * (1 - sig))) * np.abs(u) * ag + np.abs(g * sig) * au) \
        + 8 * U32 * np.abs(h_ref) + 1e-30
    err = np.abs(c["h"].reshape(P, F).astype(np.float64) - h_ref)
    assert np.all(err <= bound), f"h: {np.sum(err > bound)} outside the bound"
    # tier 2: the hidden quantisation differs only where the oracle allows it
    hq_ref = r["hq"].reshape(P, F // 32, 34)
    hq = c["hq"].reshape(P, F // 32, 34)
    d_diff = np.any(hq[:, :, :2] != hq_ref[:, :, :2], axis=2)
    q_diff = (hq[:, :, 2:].view(np.int8) != hq_ref[:, :, 2:].view(np.int8)).reshape(P, F)
    mb = mask.reshape(P, F // 32, 32)
    assert np.all(mb.all(axis=2)[d_diff]), "a scale differs in a block the oracle holds unambiguous"
    assert np.all(mask[q_diff]), "a quant differs at an element the oracle holds unambiguous"
    dq = np.abs(hq[:, :, 2:].view(np.int8).astype(int) - hq_ref[:, :, 2:].view(np.int8).astype(int))
    assert np.all(dq[~d_diff] <= 1)
    # tier 3: outputs, with the allowance of the ambiguous elements
    allow = np.zeros((T, K))
    ids, rw = c["ids"], c["rw"]
    for t in range(T):
        for s in range(topk):
            pi = t * topk + s
            if not mask[pi].any():
                continue
            absWd = _q4_0_abs_dequant(c["Wd"][ids[t, s]])
            allow[t] += abs(float(rw[t, s])) * (absWd @ (mask[pi] * step[pi]))
    err = np.abs(c["y"].astype(np.float64) - r["y"])
    bound = TOL * r["y_abs"] + allow * 1.01
    assert np.all(err <= bound), f"y: {np.sum(err > bound)} outside the bound"
    _check_down(c, K, F)
    return int(q_diff.sum()), int(mask.sum())


def _check_down(c, K, F, valid=None):
    """Down projection + combine against the oracle run on the GPU's own hq bytes:
    within TOL * sum|terms|, no allowance."""
    y2, ya2 = c["orc"].moe_down(c["Wd"], c["ids"], c["rw"], c["hq"], K, F, valid)
    err = np.abs(c["y"].astype(np.float64) - y2)
    bound = TOL * ya2
    assert np.all(err <= bound), f"y from the GPU's hq: {np.sum(err > bound)} outside TOL * sum|terms|"


def test_moe_small(orc):
    c = _run(orc, T=24, E=8, topk=3, K=512, F=768, seed=11)
    _check(c, 512, 768)


def test_moe_many_pairs_per_expert(orc):
    """More routed pairs per expert than one pass of the grouped kernels takes
    (64): 192 tokens, 4 experts, top-2 -> ~96 pairs per expert, two passes;
    also an expert with no pairs at all (5 experts, ids drawn from 4)."""
    torch = torch_cuda()
    cq = cq_built()
    T, E, topk, K, F = 192, 5, 2, 512, 512
    rng = np.random.default_rng(21)
    Wg = np.stack([synth.gen_q4_0(rng, F, K) for _ in range(E)])
    Wu = np.stack([synth.gen_q4_0(rng, F, K) for _ in range(E)])
    Wd = np.stack([synth.gen_q4_0(rng, K, F) for _ in range(E)])
    ids = np.stack([rng.permutation(4)[:topk] for _ in range(T)]).astype(np.int32)   # expert 4 unused
    rw = rng.random((T, topk)).astype(np.float32)
    x = rng.standard_normal((T, K)).astype(np.float32)
    xq = orc.quantize(orc.Q8_0, x)
    y, ws = cq.moe_t(dev(torch, Wg), dev(torch, Wu), dev(torch, Wd), dev(torch, ids), dev(torch, rw),
                     dev(torch, xq), K, F)
    st, code = cq.cq_moe_read_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == cq.OK and code == 0
    assert np.bincount(ids.ravel(), minlength=E).max() > 64
    st, so, ho, qo = cq.cq_moe_workspace_offsets(T, K, F, E, topk)
    wsn = ws.cpu().numpy()
    P = T * topk
    c = dict(Wd=Wd, ids=ids, rw=rw, y=y.cpu().numpy(), orc=orc,
             h=wsn[ho:ho + 4 * P * F].view(np.float32).reshape(T, topk, F),
             hq=wsn[qo:qo + P * (F // 32) * 34].reshape(T, topk, -1),
             r=orc.moe(Wg, Wu, Wd, ids, rw, xq, K, F))
    _check(c, K, F)


def test_moe_config_sampled(orc):
    """The routed-FFN workload (256 tokens, 32 experts, top-4, 2048/1792, Q4_0):
    the GPU runs the whole batch; the oracle checks a sample of 12 tokens."""
    sample = np.array([0, 1, 17, 63, 64, 100, 128, 170, 200, 229, 254, 255])
    c = _run(orc, T=256, E=32, topk=4, K=2048, F=1792, seed=0, token_sample=sample)
    _check(c, 2048, 1792)


def test_moe_bad_ids_flagged(orc):
    torch = torch_cuda()
    cq = cq_built()
    T, E, topk, K, F = 8, 4, 2, 256, 256
    rng = np.random.default_rng(3)
    Wg = np.stack([synth.gen_q4_0(rng, F, K) for _ in range(E)])
    Wu = np.stack([synth.gen_q4_0(rng, F, K) for _ in range(E)])
    Wd = np.stack([synth.gen_q4_0(rng, K, F) for _ in range(E)])
    ids, rw = synth.gen_routing(rng, T, E, topk)
    xq = orc.quantize(orc.Q8_0, rng.standard_normal((T, K)).astype(np.float32))
    for bad, bit in ((lambda a: a.__setitem__((2, 1), 7), cq.DEV_BAD_EXPERT_ID),
                     (lambda a: a.__setitem__((3, 1), a[3, 0]), cq.DEV_DUP_EXPERT_ID),
                     (lambda a: a.__setitem__((0, 0), -1), cq.DEV_BAD_EXPERT_ID)):
        ids2 = ids.copy()
        bad(ids2)
        y, ws = cq.moe_t(dev(torch, Wg), dev(torch, Wu), dev(torch, Wd), dev(torch, ids2), dev(torch, rw),
                         dev(torch, xq), K, F)
        st, code = cq.cq_moe_read_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == cq.ERR_DEVICE_STATUS and code & bit
        assert cq.cq_read_device_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == (st, code)
        st, so, ho, qo = cq.cq_moe_workspace_offsets(T, K, F, E, topk)
        wsn = ws.cpu().numpy()
        P = T * topk
        h_gpu = wsn[ho:ho + 4 * P * F].view(np.float32).reshape(T, topk, F)
        hq_gpu = wsn[qo:qo + P * (F // 32) * 34].reshape(T, topk, -1)
        yy = y.cpu().numpy()
        # every token, the skipped pair left out: down + combine from the GPU's own hq
        valid = np.array([[0 <= ids2[t, s] < E and ids2[t, s] not in ids2[t, :s] for s in range(topk)]
                          for t in range(T)], np.int32)
        _check_down(dict(orc=orc, Wd=Wd, ids=np.where(valid, ids2, 0), rw=rw, hq=hq_gpu, y=yy), K, F, valid)
        # the tokens without a bad id: the full tiered check against the oracle
        ok_t = [t for t in range(T) if valid[t].all()]
        r = orc.moe(Wg, Wu, Wd, ids2[ok_t], rw[ok_t], xq[ok_t], K, F)
        _check(dict(orc=orc, Wd=Wd, ids=ids2[ok_t], rw=rw[ok_t], y=yy[ok_t], h=h_gpu[ok_t], hq=hq_gpu[ok_t], r=r),
               K, F)
    # a clean call afterwards reports a clear status
    y, ws = cq.moe_t(dev(torch, Wg), dev(torch, Wu), dev(torch, Wd), dev(torch, ids), dev(torch, rw),
                     dev(torch, xq), K, F)
    assert cq.cq_moe_read_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == (cq.OK, 0)
