"""Pins of the CPU oracle against things other than itself.

Each check is chosen so that a plausible slip in the oracle (a swapped nibble,
a dropped min term, a wrong sign, a transposed operand, a half-even instead of
half-away rounding) fails at least one of them:

* IEEE binary16 decode/encode against numpy's own float16 over all 65536 bit
  patterns and a set of edge values (a library routine).
* Hand-written block fixtures (tests/golden/blocks.txt) and hand-worked
  quantisation examples (tests/golden/quantize.txt).
* Closed forms: constant-nibble blocks, one-hot activations, zero scales.
* Brute force on tiny inputs: dequantize every element and sum the products in
  exact rational arithmetic; the oracle's block formula must agree to within
  the fp64 rounding of its own sum.
* Quantizer invariants: |q| <= 127, the amax element hits +-127, the
  reconstruction error is at most half a step, Q8_K block sums equal the sums.
* Offline repack: byte offsets worked out by hand from the packed layout's
  definition, and an inverse written as array reshapes that must give back
  the weights exactly, with zero padding rows.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from gemm_gguf_block_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _records(name):
    recs, cur = [], None
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "name":
            cur = {"name": rest, "value": []}
        elif key == "end":
            recs.append(cur)
            cur = None
        elif key == "value":
            i, v = rest.split()
            cur["value"].append((int(i), float(v)))
        else:
            cur[key] = rest
    return recs


# ------------------------------------------------------------------ binary16
def test_half_decode_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got) & (got > 0), np.isinf(ref) & (ref > 0))


def test_half_encode_matches_numpy(orc):
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(0.01),
        rng.standard_normal(5000).astype(np.float32) * np.float32(1e-6),   # fp16 subnormals
        rng.standard_normal(5000).astype(np.float32) * np.float32(3e4),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 1 + 2.0 ** -11,
                  1 + 3 * 2.0 ** -11, 2049.0, 2051.0], dtype=np.float32),
    ])
    ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([orc.float_to_half(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------- block decoding
FMT = {"q4_0": 2, "q4_1": 3, "q8_0": 8, "q4_k": 12, "q5_k": 13, "q6_k": 14}


@pytest.mark.parametrize("rec", _records("blocks.txt"), ids=lambda r: r["name"])
def test_block_fixture(orc, rec):
    fmt = FMT[rec["fmt"]]
    raw = np.array([int(b, 16) for b in rec["bytes"].split()], np.uint8)
    assert raw.size == orc.BLOCK[fmt][1]
    if "values" in rec:
        want = [float(v) for v in rec["values"].split()]
        got = [orc.weight_value(fmt, raw, k) for k in range(len(want))]
        assert got == want
    for k, v in rec["value"]:
        assert orc.weight_value(fmt, raw, k) == v
    if "scalemin" in rec:
        sm = [int(v) for v in rec["scalemin"].split()]
        for j in range(8):
            assert orc.q4k_scale_min(raw[4:16].tobytes(), j) == (sm[2 * j], sm[2 * j + 1])     # Q4_K and Q5_K


def test_generator_packs_fixture_layouts():
    """The input generator's packing reproduces the hand-written fixture bytes."""
    recs = {r["name"]: r for r in _records("blocks.txt")}
    raw = np.array([int(b, 16) for b in recs["q4_k_scales"]["bytes"].split()], np.uint8)
    sm = [int(v) for v in recs["q4_k_scales"]["scalemin"].split()]
    sc = np.array(sm[0::2]).reshape(1, 1, 8)
    mn = np.array(sm[1::2]).reshape(1, 1, 8)
    qs = np.arange(128)
    q = np.zeros(256, int)
    for g in range(4):
        q[64 * g:64 * g + 32] = qs[32 * g:32 * g + 32] & 15
        q[64 * g + 32:64 * g + 64] = qs[32 * g:32 * g + 32] >> 4
    packed = synth.pack_q4_k(np.array([[0x3C00]], np.uint16), np.array([[0x3800]], np.uint16), sc, mn,
                             q.reshape(1, 256))
    assert np.array_equal(packed[0], raw)
    raw40 = np.array([int(b, 16) for b in recs["q4_0_basic"]["bytes"].split()], np.uint8)
    lo = [0, 2, 4, 6, 8, 10, 12, 14, 1, 3, 5, 7, 9, 11, 13, 15]
    hi = [1, 3, 5, 7, 9, 11, 13, 15, 0, 2, 4, 6, 8, 10, 12, 14]
    packed = synth.pack_q4_0(np.array([[0x3800]], np.uint16), np.array([lo + hi]))
    assert np.array_equal(packed[0], raw40)
    # Q6_K: ql[i] = i, every qh byte 0xe4, scales[j] = j - 8, d = 1.0, worked
    # back into six-bit quants element by element from the fixture's layout.
    raw6 = np.array([int(b, 16) for b in recs["q6_k_quadrants"]["bytes"].split()], np.uint8)
    q6 = np.zeros(256, int)
    for i in range(256):
        h, qd, l = i // 128, (i % 128) // 32, i % 32
        b = 64 * h + l + 32 * (qd & 1)
        q6[i] = (b & 15 if qd < 2 else b >> 4) | (qd << 4)
    packed = synth.pack_q6_k(np.array([[0x3C00]], np.uint16), (np.arange(16) - 8).reshape(1, 1, 16),
                             q6.reshape(1, 256))
    assert np.array_equal(packed[0], raw6)
    # Q5_K: the q4_k_scales scales, qs[i] = i, qh[l] = l (l < 16) or 0xff
    raw5 = np.array([int(b, 16) for b in recs["q5_k_fifth_bit"]["bytes"].split()], np.uint8)
    qh = [l if l < 16 else 0xFF for l in range(32)]
    q5 = q.copy()
    for e in range(256):
        q5[e] |= ((qh[e % 32] >> (e // 32)) & 1) << 4
    packed = synth.pack_q5_k(np.array([[0x3C00]], np.uint16), np.array([[0x3800]], np.uint16), sc, mn,
                             q5.reshape(1, 256))
    assert np.array_equal(packed[0], raw5)


def test_q4k_scale_packing_roundtrip(orc):
    """Every (scale, min) pair 0..63 x 0..63 survives pack (generator) -> unpack (oracle) in every slot."""
    allsc = np.repeat(np.arange(64), 64)
    allmn = np.tile(np.arange(64), 64)
    for j in range(8):
        rng = np.random.default_rng(j)
        sc = rng.integers(0, 64, size=(4096, 1, 8))
        mn = rng.integers(0, 64, size=(4096, 1, 8))
        sc[:, 0, j] = allsc
        mn[:, 0, j] = allmn
        z = np.zeros((4096, 1), np.uint16)
        packed = synth.pack_q4_k(z, z, sc, mn, np.zeros((4096, 256), int))
        for r in range(0, 4096, 97):   # a spread-out sample keeps this quick
            for jj in range(8):
                assert orc.q4k_scale_min(packed[r, 4:16].tobytes(), jj) == (sc[r, 0, jj], mn[r, 0, jj])


# --------------------------------------------------------------- quantizers
def _quant_records():
    return _records("quantize.txt")


@pytest.mark.parametrize("rec", _quant_records(), ids=lambda r: r["name"])
def test_quantize_fixture(orc, rec):
    x = np.array([float(v) for v in rec["x"].split()], np.float64)
    if "xscale" in rec:
        x = x * 2.0 ** int(rec["xscale"])
    x = x.astype(np.float32).reshape(1, 32)
    q = np.array([int(v) for v in rec["q"].split()], np.int8)
    d16, s16 = int(rec["d16"], 16), int(rec["s16"], 16)
    b0 = orc.quantize(orc.Q8_0, x)[0]
    assert int(b0[0]) | (int(b0[1]) << 8) == d16
    assert np.array_equal(b0[2:].view(np.int8), q)
    b1 = orc.quantize(orc.Q8_1, x)[0]
    assert int(b1[0]) | (int(b1[1]) << 8) == d16
    assert int(b1[2]) | (int(b1[3]) << 8) == s16
    assert np.array_equal(b1[4:].view(np.int8), q)


def test_quantize_q8k_unit_scale(orc):
    """amax = 127 gives d = 1.0f stored as fp32; q = x for integer x; bsums are the sums."""
    x = np.zeros((1, 256), np.float32)
    x[0, 0] = 127
    x[0, 1:] = (np.arange(1, 256) % 7) - 3
    b = orc.quantize(orc.Q8_K, x)[0]
    assert b[:4].tobytes() == np.float32(1.0).tobytes()
    q = b[4:260].view(np.int8)
    assert np.array_equal(q, x[0].astype(np.int8))
    bs = b[260:292].view("<i2")
    assert np.array_equal(bs, q.astype(int).reshape(16, 16).sum(1))


@pytest.mark.parametrize("afmt", [8, 9, 15])
def test_quantize_invariants(orc, afmt):
    rng = np.random.default_rng(afmt)
    K = 1024
    x = np.concatenate([rng.standard_normal((6, K)), rng.standard_normal((2, K)) * 1e-6,
                        rng.standard_normal((2, K)) * 300]).astype(np.float32)
    x[7, 256:512] = 0.0   # an all-zero block
    xq = orc.quantize(afmt, x)
    bs = 32 if afmt != 15 else 256
    bb = orc.BLOCK[afmt][1]
    for m in range(x.shape[0]):
        for b in range(K // bs):
            blk = xq[m, b * bb:(b + 1) * bb]
            if afmt == 15:
                d = float(blk[:4].view(np.float32)[0])
                q = blk[4:260].view(np.int8).astype(int)
                assert np.array_equal(blk[260:].view("<i2"), q.reshape(16, 16).sum(1))
            else:
                d16 = np.frombuffer(blk[:2].tobytes(), np.float16)[0]
                off = 2 if afmt == 8 else 4
                q = blk[off:off + 32].view(np.int8).astype(int)
                d = float(np.float32(np.abs(x[m, b * bs:(b + 1) * bs]).max()) / np.float32(127))
                assert np.float16(np.float32(d)) == d16
            xs = x[m, b * bs:(b + 1) * bs].astype(np.float64)
            amax = np.abs(xs).max()
            assert np.abs(q).max() <= 127
            if amax == 0:
                assert d == 0 and not q.any()
                continue
            assert np.abs(q).max() == 127
            step = amax / 127
            # reconstruction within half a step, allowing the fp32 rounding of d and x/d
            assert np.all(np.abs(xs - step * q) <= step * (0.5 + 1e-5))
            if afmt == 9:
                s16 = np.frombuffer(blk[2:4].tobytes(), np.float16)[0]
                dd = np.float32(amax) / np.float32(127)
                assert s16 == np.float16(np.float32(dd) * np.float32(q.sum()))


# ------------------------------------------------------------- closed forms
def _q8_bytes(d_bits, q):
    return synth.pack_q8_0(np.array([d_bits], np.uint16), np.array([q]))


def test_constant_nibble_q4_0(orc):
    """q == c everywhere: y = sum_b d_w (c - 8) d_x sum(q_x) (exact in fp64)."""
    rng = np.random.default_rng(1)
    K, N = 512, 5
    nb = K // 32
    for c in (0, 3, 8, 15):
        dw = synth._f16_bits(np.abs(rng.standard_normal((N, nb))) * 0.01)
        W = synth.pack_q4_0(dw, np.full((N, K), c))
        x = rng.standard_normal((1, K)).astype(np.float32)
        xq = orc.quantize(orc.Q8_0, x)
        y, _ = orc.matmul(orc.Q4_0, W, xq, K)
        blocks = xq[0].reshape(nb, 34)
        dx = blocks[:, :2].copy().view(np.float16).astype(np.float64)[:, 0]
        sq = blocks[:, 2:].view(np.int8).astype(np.int64).sum(1)
        want = [sum(Fraction(float(np.float16(dw[n, b].view(np.float16)))) * (c - 8)
                    * Fraction(float(dx[b])) * int(sq[b]) for b in range(nb)) for n in range(N)]
        for n in range(N):
            assert abs(Fraction(y[0, n]) - want[n]) <= abs(want[n]) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)


@pytest.mark.parametrize("wfmt", [2, 3, 8, 12, 13, 14])
def test_one_hot_activation(orc, wfmt):
    """x = e_k: the block holding k has d_x = fp16(1/127) (Q8_K: fp32 1/127), q_k = 127 and
    all other quants 0, so y_n = d_x * 127 * W[n,k] exactly -- plus, for Q4_1, the offset
    term m_w * s_x of that block, and for Q4_K, nothing else since mins multiply sum(q)=127
    inside the value formula."""
    rng = np.random.default_rng(wfmt)
    K, N = 512, 7
    W = synth.GEN[{2: "q4_0", 3: "q4_1", 8: "q8_0", 12: "q4_k", 13: "q5_k", 14: "q6_k"}[wfmt]](rng, N, K)
    afmt = orc.ACT_FOR[wfmt]
    for k in (0, 31, 100, 511):
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        xq = orc.quantize(afmt, x)
        y, _ = orc.matmul(wfmt, W, xq, K)
        dx = float(np.float32(1.0) / np.float32(127))
        if afmt != orc.Q8_K:
            dx = float(np.float16(dx))
        for n in range(N):
            wv = orc.weight_value(wfmt, W[n], k)
            if wfmt == 3:
                # value = d q + m: the m part enters through s = fp16(d_x * 127)
                blk = W[n, (k // 32) * 20:(k // 32) * 20 + 20]
                m = float(blk[2:4].copy().view(np.float16)[0])
                s = float(np.float16(np.float32(dx) * np.float32(127)))
                want = (wv - m) * dx * 127 + m * s
            else:
                want = wv * dx * 127
            assert y[0, n] == pytest.approx(want, rel=1e-14, abs=1e-300)


@pytest.mark.parametrize("wfmt", [2, 3, 8, 12, 13, 14])
def test_zero_scales_give_zero(orc, wfmt):
    rng = np.random.default_rng(3)
    K, N = 512, 4
    W = synth.GEN[{2: "q4_0", 3: "q4_1", 8: "q8_0", 12: "q4_k", 13: "q5_k", 14: "q6_k"}[wfmt]](rng, N, K)
    bs, bb = orc.BLOCK[wfmt]
    Wz = W.copy().reshape(N, K // bs, bb)
    if wfmt == 14:
        Wz[:, :, 208:210] = 0           # Q6_K: d is the last field
    else:
        Wz[:, :, 0:2] = 0               # d
    if wfmt in (3, 12, 13):
        Wz[:, :, 2:4] = 0               # m / dmin
    x = rng.standard_normal((2, K)).astype(np.float32)
    xq = orc.quantize(orc.ACT_FOR[wfmt], x)
    y, at = orc.matmul(wfmt, Wz.reshape(N, -1), xq, K)
    assert np.all(y == 0) and np.all(at == 0)


# -------------------------------------------------------- brute force (exact)
def _exact_dot(orc, wfmt, wrow, xrow, K):
    afmt = orc.ACT_FOR[wfmt]
    return sum(Fraction(orc.weight_value(wfmt, wrow, k)) * Fraction(orc.act_value(afmt, xrow, k))
               for k in range(K))


@pytest.mark.parametrize("wfmt", [2, 3, 8, 12, 13, 14])
def test_brute_force_tiny(orc, wfmt):
    """Dequantize every element and sum exactly; compare with the block formula.

    For Q4_1 the block formula uses the activation's stored block sum s = fp16(d_x sum q)
    for the offset term, so the exact reference replaces m_w d_x sum(q_x) by m_w s_x."""
    rng = np.random.default_rng(100 + wfmt)
    K, N, M = 512, 6, 3
    W = synth.GEN[{2: "q4_0", 3: "q4_1", 8: "q8_0", 12: "q4_k", 13: "q5_k", 14: "q6_k"}[wfmt]](rng, N, K)
    x = rng.standard_normal((M, K)).astype(np.float32)
    afmt = orc.ACT_FOR[wfmt]
    xq = orc.quantize(afmt, x)
    y, at = orc.matmul(wfmt, W, xq, K)
    for m in range(M):
        for n in range(N):
            want = _exact_dot(orc, wfmt, W[n], xq[m], K)
            if wfmt == 3:
                for b in range(K // 32):
                    wb = W[n, b * 20:b * 20 + 20]
                    xb = xq[m, b * 36:b * 36 + 36]
                    mw = Fraction(float(wb[2:4].copy().view(np.float16)[0]))
                    dx = Fraction(float(xb[0:2].copy().view(np.float16)[0]))
                    sx = Fraction(float(xb[2:4].copy().view(np.float16)[0]))
                    sq = int(xb[4:].view(np.int8).astype(int).sum())
                    want += mw * (sx - dx * sq)
            err = abs(Fraction(y[m, n]) - want)
            assert err <= Fraction(at[m, n]) * Fraction(64, 2 ** 53), (m, n, float(err))


def test_rows_independent_of_batch(orc):
    """Row n of a batched call equals the single-token call bit for bit."""
    rng = np.random.default_rng(5)
    K, N = 1024, 9
    W = synth.gen_q4_1(rng, N, K)
    x = rng.standard_normal((4, K)).astype(np.float32)
    xq = orc.quantize(orc.Q8_1, x)
    y4, _ = orc.matmul(orc.Q4_1, W, xq, K)
    for m in range(4):
        y1, _ = orc.matmul(orc.Q4_1, W, xq[m:m + 1], K)
        assert np.array_equal(y1[0], y4[m])


# -------------------------------------------------------------------- MoE
def _tiny_moe(seed=0, T=3, E=4, topk=2, K=256, F=256):
    rng = np.random.default_rng(seed)
    Wg = np.stack([synth.gen_q4_0(rng, F, K) for _ in range(E)])
    Wu = np.stack([synth.gen_q4_0(rng, F, K) for _ in range(E)])
    Wd = np.stack([synth.gen_q4_0(rng, K, F) for _ in range(E)])
    ids, rw = synth.gen_routing(rng, T, E, topk)
    x = rng.standard_normal((T, K)).astype(np.float32)
    return Wg, Wu, Wd, ids, rw, x


def test_moe_brute_force(orc):
    """Routed FFN against an element-wise dequantize-and-sum evaluation of every step
    (exact rationals for the contractions, math.exp for silu, the pinned quantizer for h)."""
    K = F = 256
    Wg, Wu, Wd, ids, rw, x = _tiny_moe(K=K, F=F)
    xq = orc.quantize(orc.Q8_0, x)
    r = orc.moe(Wg, Wu, Wd, ids, rw, xq, K, F)
    T, topk = ids.shape
    for t in range(T):
        acc = [Fraction(0)] * K
        for s in range(topk):
            e = ids[t, s]
            g = [float(_exact_dot(orc, 2, Wg[e, f], xq[t], K)) for f in range(F)]
            u = [float(_exact_dot(orc, 2, Wu[e, f], xq[t], K)) for f in range(F)]
            h = [gi / (1.0 + math.exp(-gi)) * ui for gi, ui in zip(g, u)]
            np.testing.assert_allclose(r["h"][t, s], h, rtol=1e-13, atol=1e-300)
            hq = orc.quantize(orc.Q8_0, np.array([h], np.float32))
            assert np.array_equal(hq[0], r["hq"][t, s])
            for k in range(K):
                acc[k] += Fraction(float(rw[t, s])) * _exact_dot(orc, 2, Wd[e, k], hq[0], F)
        want = np.array([float(a) for a in acc])
        assert np.all(np.abs(r["y"][t] - want) <= r["y_abs"][t] * 1e-13)


def test_moe_down_brute_force(orc):
    """The routed FFN from given hidden quantisations on (oracle_moe_down): every
    pair's down projection of arbitrary Q8_0 rows, dequantized element by element
    and summed in exact rationals, weighted and combined over the token's valid
    slots; a pair marked invalid contributes nothing."""
    K = F = 256
    _, _, Wd, ids, rw, _ = _tiny_moe(seed=4, K=K, F=F)
    T, topk = ids.shape
    rng = np.random.default_rng(44)
    hq = orc.quantize(orc.Q8_0, rng.standard_normal((T * topk, F)).astype(np.float32))
    valid = np.ones((T, topk), np.int32)
    valid[1, 0] = 0
    y, ya = orc.moe_down(Wd, ids, rw, hq, K, F, valid)
    for t in range(T):
        acc = [Fraction(0)] * K
        for s in range(topk):
            if not valid[t, s]:
                continue
            for k in range(K):
                acc[k] += Fraction(float(rw[t, s])) * _exact_dot(orc, 2, Wd[ids[t, s], k], hq[t * topk + s], F)
        want = np.array([float(a) for a in acc])
        assert np.all(np.abs(y[t] - want) <= ya[t] * 1e-13)
    # the skipped pair: token 1's output is its other slot's alone
    y1, _ = orc.moe_down(Wd, ids[1:2, 1:], rw[1:2, 1:], hq[3:4], K, F)
    assert np.array_equal(y1[0], y[1])


def test_moe_down_continues_moe(orc):
    """Fed the whole routed FFN's own hidden quantisation, the second half gives
    the same outputs and bounds bit for bit (one definition, one arithmetic)."""
    K, F = 256, 512
    Wg, Wu, Wd, ids, rw, x = _tiny_moe(seed=5, K=K, F=F)
    xq = orc.quantize(orc.Q8_0, x)
    r = orc.moe(Wg, Wu, Wd, ids, rw, xq, K, F)
    y, ya = orc.moe_down(Wd, ids, rw, r["hq"], K, F)
    assert np.array_equal(y, r["y"]) and np.array_equal(ya, r["y_abs"])
    bad = ids.copy()
    bad[0, 0] = Wd.shape[0]
    with pytest.raises(ValueError):
        orc.moe_down(Wd, bad, rw, r["hq"], K, F)


def test_moe_router_weight_linearity_and_slot_order(orc):
    K = F = 256
    Wg, Wu, Wd, ids, rw, x = _tiny_moe(seed=1, K=K, F=F)
    xq = orc.quantize(orc.Q8_0, x)
    a = orc.moe(Wg, Wu, Wd, ids, rw, xq, K, F)["y"]
    b = orc.moe(Wg, Wu, Wd, ids, rw * np.float32(2), xq, K, F)["y"]
    assert np.array_equal(b, 2 * a)                     # power-of-two scaling is exact
    c = orc.moe(Wg, Wu, Wd, ids[:, ::-1].copy(), rw[:, ::-1].copy(), xq, K, F)["y"]
    np.testing.assert_allclose(c, a, rtol=1e-12, atol=1e-300)


def test_moe_zero_up_gives_zero(orc):
    K = F = 256
    Wg, Wu, Wd, ids, rw, x = _tiny_moe(seed=2, K=K, F=F)
    Wu = Wu.reshape(Wu.shape[0], F, K // 32, 18).copy()
    Wu[..., 0:2] = 0
    xq = orc.quantize(orc.Q8_0, x)
    r = orc.moe(Wg, Wu.reshape(Wg.shape), Wd, ids, rw, xq, K, F)
    assert np.all(r["h"] == 0) and np.all(r["y"] == 0)


def test_moe_rejects_bad_ids(orc):
    K = F = 256
    Wg, Wu, Wd, ids, rw, x = _tiny_moe(seed=3, K=K, F=F)
    xq = orc.quantize(orc.Q8_0, x)
    bad = ids.copy()
    bad[1, 1] = bad[1, 0]
    with pytest.raises(ValueError):
        orc.moe(Wg, Wu, Wd, bad, rw, xq, K, F)
    bad = ids.copy()
    bad[0, 0] = Wg.shape[0]
    with pytest.raises(ValueError):
        orc.moe(Wg, Wu, Wd, bad, rw, xq, K, F)


# ------------------------------------------------------------- dense SwiGLU
def _fmt_name(wfmt):
    return {2: "q4_0", 3: "q4_1", 8: "q8_0", 12: "q4_k"}[wfmt]


@pytest.mark.parametrize("wfmt", [2, 3, 8, 12])
def test_swiglu_brute_force(orc, wfmt):
    """h = silu(g) * u with g, u from an element-wise dequantize-and-sum (exact
    rationals) evaluation, silu from math.exp; the gate goes through silu, the
    up projection does not (a swapped pair fails: silu(u) * g != silu(g) * u)."""
    rng = np.random.default_rng(200 + wfmt)
    K, F, M = 512, 5, 2
    Wg = synth.GEN[_fmt_name(wfmt)](rng, F, K)
    Wu = synth.GEN[_fmt_name(wfmt)](rng, F, K)
    x = rng.standard_normal((M, K)).astype(np.float32)
    xq = orc.quantize(orc.ACT_FOR[wfmt], x)
    h, aux = orc.swiglu(wfmt, Wg, Wu, xq, K)
    for m in range(M):
        for f in range(F):
            g = float(_exact_dot(orc, wfmt, Wg[f], xq[m], K))
            u = float(_exact_dot(orc, wfmt, Wu[f], xq[m], K))
            if wfmt == 3:
                # the block formula's offset term uses the stored s_x (see test_brute_force_tiny)
                g, u = aux[m, f, 0], aux[m, f, 1]
            assert aux[m, f, 0] == pytest.approx(g, rel=1e-12, abs=1e-12)
            assert aux[m, f, 1] == pytest.approx(u, rel=1e-12, abs=1e-12)
            assert h[m, f] == pytest.approx(g / (1.0 + math.exp(-g)) * u, rel=1e-12, abs=1e-300)


def test_swiglu_odd_part_identity(orc):
    """silu(g) - silu(-g) = g for every g. Negating every Q8_0 gate quant negates g
    exactly, so h(W_gate) - h(-W_gate) = g * u -- a property of the definition
    that a sign slip in silu or a dropped factor breaks."""
    rng = np.random.default_rng(7)
    K, F, M = 768, 9, 3
    Wg = synth.GEN["q8_0"](rng, F, K)
    Wu = synth.GEN["q8_0"](rng, F, K)
    blocks = Wg.reshape(F, K // 32, 34).copy()
    q = blocks[:, :, 2:].view(np.int8)
    neg = blocks.copy()
    neg[:, :, 2:] = (-q.astype(np.int16)).astype(np.int8).view(np.uint8)     # |q| <= 127: exact
    x = rng.standard_normal((M, K)).astype(np.float32)
    xq = orc.quantize(orc.Q8_0, x)
    h1, aux = orc.swiglu(orc.Q8_0, Wg, Wu, xq, K)
    h2, aux2 = orc.swiglu(orc.Q8_0, neg.reshape(F, -1), Wu, xq, K)
    assert np.array_equal(aux2[..., 0], -aux[..., 0])
    gu = aux[..., 0] * aux[..., 1]
    np.testing.assert_allclose(h1 - h2, gu, rtol=1e-12, atol=1e-12 * np.abs(gu).max())


@pytest.mark.parametrize("which", ["gate", "up"])
def test_swiglu_zero_scales_give_zero(orc, which):
    """Zero gate scales give g = 0 and silu(0) = 0; zero up scales give u = 0."""
    rng = np.random.default_rng(11)
    K, F = 512, 6
    Wg = synth.GEN["q4_k"](rng, F, K)
    Wu = synth.GEN["q4_k"](rng, F, K)
    target = (Wg if which == "gate" else Wu).reshape(F, K // 256, 144)
    target[:, :, 0:4] = 0                # d and dmin
    x = rng.standard_normal((2, K)).astype(np.float32)
    xq = orc.quantize(orc.Q8_K, x)
    h, _ = orc.swiglu(orc.Q4_K, Wg, Wu, xq, K)
    assert np.all(h == 0)


# ------------------------------------------------------------ offline repack
# The packed layout is the library's own (include/cq.h, cq_repack): units of
# 16 rows x 4 blocks, segment-major; per row the blocks' scale fields, then per
# (half, row, lane t, block j) the quant bytes 16h + 4t .. 16h + 4t + 3.

def _identity_rows(N, row_bytes):
    """Weight bytes that name their own position: (7 n + 3 b + 1) mod 251."""
    n = np.arange(N)[:, None]
    b = np.arange(row_bytes)[None, :]
    return ((7 * n + 3 * b + 1) % 251).astype(np.uint8)


def test_repack_hand_offsets(orc):
    """Byte offsets worked out by hand from the layout definition."""
    W = _identity_rows(17, 160)                  # Q4_1, K = 256: 8 blocks of 20 bytes
    P = orc.repack(orc.Q4_1, W, 256)
    assert P.size == 2 * 2 * 1280                # 2 groups x 2 segments x 64 * 20
    assert list(P[0:4]) == list(W[0, 0:4])       # row 0, block 0: d, m
    assert list(P[24:28]) == list(W[1, 40:44])   # row 1, block 2: at 1*16 + 2*4
    assert list(P[364:368]) == list(W[1, 72:76]) # row 1, lane 2, block 3: 256 + ((1*4+2)*4+3)*4
    assert list(P[1280:1284]) == list(W[16, 0:4])            # group 1 (row 16), segment 0
    assert not P[1280 + 16:1280 + 256].any()                 # rows 17..31: no scales
    assert not P[1280 + 256 + 64:2560].any()                 # rows 17..31: no quants
    assert list(P[2560:2564]) == list(W[0, 80:84])           # group 0, segment 1: block 4
    W8 = _identity_rows(16, 272)                 # Q8_0, K = 256: 8 blocks of 34 bytes
    P8 = orc.repack(orc.Q8_0, W8, 256)
    assert P8.size == 2 * 2176
    assert list(P8[26:28]) == list(W8[3, 34:36])             # row 3, block 1: d at 3*8 + 1*2
    assert list(P8[1328:1332]) == list(W8[2, 30:34])         # half 1, row 2, lane 3, block 0
    W4 = _identity_rows(3, 144)                  # Q4_0, K = 256
    P4 = orc.repack(orc.Q4_0, W4, 256)
    assert P4.size == 2 * 1152
    assert list(P4[148:152]) == list(W4[0, 24:28])           # row 0, lane 1, block 1: 128 + 5*4
    assert list(P4[22:24]) == list(W4[2, 54:56])             # row 2, block 3: d at 2*8 + 3*2


def _unpack(fmt, P, N, K):
    """Inverse of the layout, written as array reshapes (scatter form)."""
    bb = {2: 18, 3: 20, 8: 34}[fmt]
    sb = 4 if fmt == 3 else 2
    halves = 2 if fmt == 8 else 1
    ng, ns = (N + 15) // 16, K // 128
    U = P.reshape(ns, ng, 64 * bb)
    scales = U[:, :, :64 * sb].reshape(ns, ng, 16, 4, sb)
    quants = U[:, :, 64 * sb:].reshape(ns, ng, halves, 16, 4, 4, 4)          # s, G, h, r, t, j, byte
    quants = quants.transpose(1, 3, 0, 5, 2, 4, 6).reshape(ng * 16, ns * 4, halves * 16)
    scales = scales.transpose(1, 2, 0, 3, 4).reshape(ng * 16, ns * 4, sb)
    blocks = np.concatenate([scales, quants], axis=2)                        # row, block, bytes
    assert blocks.shape[2] == bb
    return blocks.reshape(ng * 16, K // 32 * bb)


@pytest.mark.parametrize("fmt", [2, 3, 8])
@pytest.mark.parametrize("N,K", [(1, 256), (15, 512), (16, 256), (33, 768)])
def test_repack_inverse_roundtrip(orc, fmt, N, K):
    """Unpacking by the inverse reshapes gives back W; padding rows are zero."""
    rng = np.random.default_rng(fmt * 100 + N + K)
    W = rng.integers(0, 256, (N, orc.row_bytes(fmt, K)), dtype=np.uint8)
    P = orc.repack(fmt, W, K)
    assert P.size == (N + 15) // 16 * 16 * orc.row_bytes(fmt, K)
    Wb = _unpack(fmt, P, N, K)
    assert np.array_equal(Wb[:N], W)
    assert not Wb[N:].any()


def test_repack_rejects(orc):
    assert orc.repack_size(orc.Q4_K, 16, 256) == -1
    assert orc.repack_size(orc.Q4_0, 16, 128) == -1
    assert orc.repack_size(orc.Q4_0, 0, 256) == 0
