"""Seeded synthetic inputs in GGUF block layouts.

This module draws random scales, quants and activations and packs them into
the byte layouts the library consumes. It holds none of the contraction's
arithmetic: no activation quantisation, no dot products, no dequantisation.
Both the CUDA path (through the tests and the benchmark) and the CPU oracle
read the bytes it produces; neither imports the other.

Draw recipe (one numpy PCG64 stream per tensor, seeded with
``[seed, config_id, tensor_id]``): block scales first in row-major order, then
the element quants in row-major order, then packing. fp16 fields are the
float64 draw rounded to binary16 by numpy (round to nearest even).

Byte layouts (little endian, fp16 = IEEE binary16), element i of a 32-block:

* Q4_0, 18 B: d f16, qs[16]; q_i = qs[i] & 15 for i < 16, qs[i-16] >> 4 else.
* Q4_1, 20 B: d f16, m f16, qs[16]; same nibble order.
* Q8_0, 34 B: d f16, qs[32] int8.
* Q4_K, 144 B per 256: d f16, dmin f16, scales[12], qs[128]; the 64-element
  group g uses qs[32g:32g+32], low nibbles for elements 64g..64g+31 (sub-block
  2g), high nibbles for 64g+32..64g+63 (sub-block 2g+1); six-bit scale and min
  of sub-block j packed in scales[12] as described in ``pack_q4_k``.
* Q5_K, 176 B per 256: d f16, dmin f16, scales[12], qh[32], qs[128]; the
  low four bits and the scale/min packing as Q4_K, the fifth bit of element
  i in qh[i % 32], bit i // 32.
* Q6_K, 210 B per 256: ql[128], qh[64], scales[16] int8, d f16; element i
  (half h = i // 128, quadrant q = i % 128 // 32, l = i % 32) has its low four
  bits in ql[64h + l + 32 (q & 1)] (low nibble for q < 2, high for q >= 2)
  and its high two bits in qh[32h + l] bits 2q, 2q+1; sub-block i // 16 has
  scale scales[i // 16].

Field order of Q4_K, Q5_K, Q6_K and Q8_0 follows alice-llm's "Quantization Block Specs"
table; the nibble order and the Q4_0/Q4_1 layouts are the standard GGUF ones
(the pages name the formats without printing them).
"""
from __future__ import annotations

import numpy as np

QK = 32          # elements per Q4_0 / Q4_1 / Q8_0 / Q8_1 block
QK_K = 256       # elements per Q4_K / Q8_K superblock

BLOCK_BYTES = {"q4_0": 18, "q4_1": 20, "q8_0": 34, "q8_1": 36, "q4_k": 144, "q8_k": 292}
BLOCK_ELEMS = {"q4_0": QK, "q4_1": QK, "q8_0": QK, "q8_1": QK, "q4_k": QK_K, "q8_k": QK_K}


def row_bytes(fmt: str, K: int) -> int:
    """Bytes of one row of K elements in format ``fmt``."""
    return K // BLOCK_ELEMS[fmt] * BLOCK_BYTES[fmt]


def stream(seed: int, config_id: int, tensor_id: int) -> np.random.Generator:
    return np.random.default_rng([seed, config_id, tensor_id])


def _f16_bits(v) -> np.ndarray:
    return np.asarray(v, dtype=np.float64).astype(np.float16).view(np.uint16)


def _nibble_bytes(q: np.ndarray) -> np.ndarray:
    """q: [..., 32] ints 0..15 -> [..., 16] bytes (element i<16 low, i>=16 high)."""
    q = q.astype(np.uint8)
    return (q[..., :16] | (q[..., 16:] << 4)).astype(np.uint8)


def pack_q4_0(d_bits: np.ndarray, q: np.ndarray) -> np.ndarray:
    """d_bits: [N, nb] uint16 fp16 bits; q: [N, nb*32] ints 0..15 -> [N, nb*18] bytes."""
    N, nb = d_bits.shape
    out = np.zeros((N, nb, 18), np.uint8)
    out[:, :, 0:2] = d_bits.astype("<u2").reshape(N, nb, 1).view(np.uint8)
    out[:, :, 2:18] = _nibble_bytes(q.reshape(N, nb, 32))
    return out.reshape(N, nb * 18)


def pack_q4_1(d_bits: np.ndarray, m_bits: np.ndarray, q: np.ndarray) -> np.ndarray:
    N, nb = d_bits.shape
    out = np.zeros((N, nb, 20), np.uint8)
    out[:, :, 0:2] = d_bits.astype("<u2").reshape(N, nb, 1).view(np.uint8)
    out[:, :, 2:4] = m_bits.astype("<u2").reshape(N, nb, 1).view(np.uint8)
    out[:, :, 4:20] = _nibble_bytes(q.reshape(N, nb, 32))
    return out.reshape(N, nb * 20)


def pack_q8_0(d_bits: np.ndarray, q: np.ndarray) -> np.ndarray:
    """q: [N, nb*32] ints in [-128, 127]."""
    N, nb = d_bits.shape
    out = np.zeros((N, nb, 34), np.uint8)
    out[:, :, 0:2] = d_bits.astype("<u2").reshape(N, nb, 1).view(np.uint8)
    out[:, :, 2:34] = q.reshape(N, nb, 32).astype(np.int8).view(np.uint8)
    return out.reshape(N, nb * 34)


def pack_q4_k(d_bits, dmin_bits, sc, mn, q) -> np.ndarray:
    """Pack Q4_K superblocks.

    d_bits, dmin_bits: [N, ns] uint16; sc, mn: [N, ns, 8] ints 0..63;
    q: [N, ns*256] ints 0..15. The twelve scale bytes hold, for sub-block j:
    bytes 0-3: low six bits = sc[0..3], top two bits = sc[4..7] >> 4;
    bytes 4-7: low six bits = mn[0..3], top two bits = mn[4..7] >> 4;
    bytes 8-11: low nibble = sc[4..7] & 15, high nibble = mn[4..7] & 15.
    """
    N, ns = d_bits.shape
    sc = sc.astype(np.uint8)
    mn = mn.astype(np.uint8)
    out = np.zeros((N, ns, 144), np.uint8)
    out[:, :, 0:2] = d_bits.astype("<u2").reshape(N, ns, 1).view(np.uint8)
    out[:, :, 2:4] = dmin_bits.astype("<u2").reshape(N, ns, 1).view(np.uint8)
    s = np.zeros((N, ns, 12), np.uint8)
    s[..., 0:4] = (sc[..., 0:4] & 63) | ((sc[..., 4:8] >> 4) << 6)
    s[..., 4:8] = (mn[..., 0:4] & 63) | ((mn[..., 4:8] >> 4) << 6)
    s[..., 8:12] = (sc[..., 4:8] & 15) | ((mn[..., 4:8] & 15) << 4)
    out[:, :, 4:16] = s
    qq = q.reshape(N, ns, 4, 2, 32).astype(np.uint8)  # [group][lo/hi half][32]
    out[:, :, 16:144] = (qq[:, :, :, 0, :] | (qq[:, :, :, 1, :] << 4)).reshape(N, ns, 128)
    return out.reshape(N, ns * 144)


# ---------------------------------------------------------------- draws
def gen_q4_0(rng, N: int, K: int, scale: float = 0.01) -> np.ndarray:
    nb = K // QK
    d = _f16_bits(np.abs(rng.standard_normal((N, nb))) * scale)
    q = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    return pack_q4_0(d, q)


def pack_q5_k(d_bits, dmin_bits, sc, mn, q) -> np.ndarray:
    """Pack Q5_K superblocks: as pack_q4_k for the low four bits of q (ints
    0..31, [N, ns*256]), plus qh[32] holding bit 4 of element i in qh[i % 32]
    bit i // 32."""
    N, ns = d_bits.shape
    q = q.reshape(N, ns, 256).astype(np.uint8)
    q4 = pack_q4_k(d_bits, dmin_bits, sc, mn, (q & 15).reshape(N, ns * 256)).reshape(N, ns, 144)
    hi = (q >> 4).reshape(N, ns, 8, 32)                   # [sub-block][l]
    qh = np.zeros((N, ns, 32), np.uint8)
    for j in range(8):
        qh |= (hi[:, :, j, :] << j).astype(np.uint8)
    out = np.zeros((N, ns, 176), np.uint8)
    out[:, :, 0:16] = q4[:, :, 0:16]
    out[:, :, 16:48] = qh
    out[:, :, 48:176] = q4[:, :, 16:144]
    return out.reshape(N, ns * 176)


def pack_q6_k(d_bits, sc, q) -> np.ndarray:
    """Pack Q6_K superblocks. d_bits: [N, ns] uint16; sc: [N, ns, 16] ints
    -128..127; q: [N, ns*256] ints 0..63 (the six-bit quants)."""
    N, ns = d_bits.shape
    qq = q.reshape(N, ns, 2, 4, 32).astype(np.uint8)      # [half][quadrant][l]
    out = np.zeros((N, ns, 210), np.uint8)
    lo = qq & 15
    ql = np.zeros((N, ns, 2, 64), np.uint8)
    ql[..., 0:32] = lo[:, :, :, 0, :] | (lo[:, :, :, 2, :] << 4)
    ql[..., 32:64] = lo[:, :, :, 1, :] | (lo[:, :, :, 3, :] << 4)
    hi = qq >> 4
    qh = hi[:, :, :, 0, :] | (hi[:, :, :, 1, :] << 2) | (hi[:, :, :, 2, :] << 4) | (hi[:, :, :, 3, :] << 6)
    out[:, :, 0:128] = ql.reshape(N, ns, 128)
    out[:, :, 128:192] = qh.reshape(N, ns, 64)
    out[:, :, 192:208] = sc.astype(np.int8).view(np.uint8)
    out[:, :, 208:210] = d_bits.astype("<u2").reshape(N, ns, 1).view(np.uint8)
    return out.reshape(N, ns * 210)


def gen_q4_1(rng, N: int, K: int, scale: float = 0.01) -> np.ndarray:
    nb = K // QK
    d = _f16_bits(np.abs(rng.standard_normal((N, nb))) * scale)
    m = _f16_bits(rng.standard_normal((N, nb)) * scale)
    q = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    return pack_q4_1(d, m, q)


def gen_q8_0(rng, N: int, K: int, scale: float = 0.005) -> np.ndarray:
    nb = K // QK
    d = _f16_bits(np.abs(rng.standard_normal((N, nb))) * scale)
    q = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    return pack_q8_0(d, q)


def gen_q4_k(rng, N: int, K: int, scale: float = 0.01) -> np.ndarray:
    ns = K // QK_K
    d = _f16_bits(np.abs(rng.standard_normal((N, ns))) * scale)
    dmin = _f16_bits(np.abs(rng.standard_normal((N, ns))) * scale)
    sc = rng.integers(0, 64, size=(N, ns, 8), dtype=np.uint8)
    mn = rng.integers(0, 64, size=(N, ns, 8), dtype=np.uint8)
    q = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    return pack_q4_k(d, dmin, sc, mn, q)


def gen_q5_k(rng, N: int, K: int, scale: float = 0.01) -> np.ndarray:
    ns = K // QK_K
    d = _f16_bits(np.abs(rng.standard_normal((N, ns))) * scale)
    dmin = _f16_bits(np.abs(rng.standard_normal((N, ns))) * scale)
    sc = rng.integers(0, 64, size=(N, ns, 8), dtype=np.uint8)
    mn = rng.integers(0, 64, size=(N, ns, 8), dtype=np.uint8)
    q = rng.integers(0, 32, size=(N, K), dtype=np.uint8)
    return pack_q5_k(d, dmin, sc, mn, q)


def gen_q6_k(rng, N: int, K: int, scale: float = 0.001) -> np.ndarray:
    ns = K // QK_K
    d = _f16_bits(np.abs(rng.standard_normal((N, ns))) * scale)
    sc = rng.integers(-64, 64, size=(N, ns, 16), dtype=np.int8)
    q = rng.integers(0, 64, size=(N, K), dtype=np.uint8)
    return pack_q6_k(d, sc, q)


GEN = {"q4_0": gen_q4_0, "q4_1": gen_q4_1, "q8_0": gen_q8_0, "q4_k": gen_q4_k, "q5_k": gen_q5_k, "q6_k": gen_q6_k}
ACT_FOR = {"q4_0": "q8_0", "q8_0": "q8_0", "q4_1": "q8_1", "q4_k": "q8_k", "q5_k": "q8_k", "q6_k": "q8_k"}


def gen_weights(fmt: str, rng, N: int, K: int) -> np.ndarray:
    return GEN[fmt](rng, N, K)


def gen_x(rng, M: int, K: int) -> np.ndarray:
    """Activations: float64 N(0,1) cast to fp32, shape [M, K]."""
    return rng.standard_normal((M, K)).astype(np.float32)


def gen_routing(rng, T: int, E: int, topk: int):
    """Per token: topk distinct experts drawn uniformly, router weights softmax(N(0,1))."""
    ids = np.stack([rng.permutation(E)[:topk] for _ in range(T)]).astype(np.int32)
    logits = rng.standard_normal((T, topk))
    w = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


# ---------------------------------------------------------------- named workloads
# Shapes of the five synthetic workloads (Llama-3-8B layer shapes and an
# LFM2.5-8B-A1B-like routed FFN stand in for model files that are not here).
DECODE_SUITE_Q8_0 = [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336), (128256, 4096)]


def decode_q4_0_small(seed: int = 0):
    """Q4_0 GEMV 2048x2048, M=1."""
    W = gen_q4_0(stream(seed, 1, 0), 2048, 2048)
    x = gen_x(stream(seed, 1, 1), 1, 2048)
    return W, x


def decode_q8_0_layer(seed: int, i: int, N: int, K: int):
    """Layer i of the Q8_0 decode suite: W [N, K] and x [1, K]."""
    W = gen_q8_0(stream(seed, 2, 2 * i), N, K)
    x = gen_x(stream(seed, 2, 2 * i + 1), 1, K)
    return W, x


def decode_q8_0_suite(seed: int = 0, shapes=None):
    """Q8_0 decode GEMVs at Llama-3-8B shapes (N, K), M=1: list of (W, x)."""
    return [decode_q8_0_layer(seed, i, N, K) for i, (N, K) in enumerate(shapes or DECODE_SUITE_Q8_0)]


def prefill_q4_k(seed: int = 0, M: int = 512, N: int = 14336, K: int = 4096):
    W = gen_q4_k(stream(seed, 3, 0), N, K)
    x = gen_x(stream(seed, 3, 1), M, K)
    return W, x


def prefill_32(fmt: str, seed: int = 0, M: int = 512, N: int = 14336, K: int = 4096):
    """Prefill GEMM of a 32-element format (q4_0, q4_1, q8_0): Llama-3-8B FFN
    gate shape, 512 prompt tokens."""
    tid = {"q4_0": 0, "q4_1": 2, "q8_0": 4}[fmt]
    W = GEN[fmt](stream(seed, 9, tid), N, K)
    x = gen_x(stream(seed, 9, tid + 1), M, K)
    return W, x


def moe_ffn(seed: int = 0, T: int = 256, E: int = 32, topk: int = 4, K: int = 2048, F: int = 1792):
    """Routed FFN: per expert Q4_0 gate/up [F, K] and down [K, F]."""
    Wg = np.stack([gen_q4_0(stream(seed, 4, 10 + e), F, K) for e in range(E)])
    Wu = np.stack([gen_q4_0(stream(seed, 4, 10 + E + e), F, K) for e in range(E)])
    Wd = np.stack([gen_q4_0(stream(seed, 4, 10 + 2 * E + e), K, F) for e in range(E)])
    ids, rw = gen_routing(stream(seed, 4, 0), T, E, topk)
    x = gen_x(stream(seed, 4, 1), T, K)
    return Wg, Wu, Wd, ids, rw, x


def lm_head_q4_1(seed: int = 0, N: int = 128256, K: int = 4096, M: int = 16):
    W = gen_q4_1(stream(seed, 5, 0), N, K)
    x = gen_x(stream(seed, 5, 1), M, K)
    return W, x


def lm_head_q6_k(seed: int = 0, N: int = 128256, K: int = 2048, M: int = 4):
    """Tied-embedding LM head in Q6_K (Llama-3.2-1B: vocabulary x hidden 2048)."""
    W = gen_q6_k(stream(seed, 7, 0), N, K)
    x = gen_x(stream(seed, 7, 1), M, K)
    return W, x


def ffn_q5_k(seed: int = 0, N: int = 14336, K: int = 4096, M: int = 4):
    """Dense FFN gate projection in Q5_K [N, K] (Llama-3-8B shapes)."""
    W = gen_q5_k(stream(seed, 8, 0), N, K)
    x = gen_x(stream(seed, 8, 1), M, K)
    return W, x


def ffn_swiglu_q4_k(seed: int = 0, F: int = 14336, K: int = 4096, M: int = 4):
    """Dense SwiGLU FFN gate and up projections, Q4_K [F, K] each (Llama-3-8B shapes)."""
    Wg = gen_q4_k(stream(seed, 6, 0), F, K)
    Wu = gen_q4_k(stream(seed, 6, 1), F, K)
    x = gen_x(stream(seed, 6, 2), M, K)
    return Wg, Wu, x
