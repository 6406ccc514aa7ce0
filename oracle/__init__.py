"""CPU oracle (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package. The library under test never does.

Thin ctypes wrapper over ``oracle.c`` (plain single-threaded C, fp64 after the
exact integer block dots, activation quantisation decided in fp32). The shared
object is compiled on first use with gcc, or by ``build()``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

Q4_0, Q4_1, Q8_0, Q8_1, Q4_K, Q5_K, Q6_K, Q8_K = 2, 3, 8, 9, 12, 13, 14, 15
FMT = {"q4_0": Q4_0, "q4_1": Q4_1, "q8_0": Q8_0, "q8_1": Q8_1, "q4_k": Q4_K, "q5_k": Q5_K, "q6_k": Q6_K,
       "q8_k": Q8_K}
ACT_FOR = {Q4_0: Q8_0, Q8_0: Q8_0, Q4_1: Q8_1, Q4_K: Q8_K, Q5_K: Q8_K, Q6_K: Q8_K}
BLOCK = {Q4_0: (32, 18), Q4_1: (32, 20), Q8_0: (32, 34), Q8_1: (32, 36), Q4_K: (256, 144), Q5_K: (256, 176),
         Q6_K: (256, 210), Q8_K: (256, 292)}


def row_bytes(fmt: int, K: int) -> int:
    e, b = BLOCK[fmt]
    return K // e * b


def build(force: bool = False) -> str:
    """Compile liboracle.so (gcc, -O2, no FMA contraction, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            P, I64, I = C.c_void_p, C.c_int64, C.c_int
            L.oracle_half_to_double.argtypes = [C.c_uint16]
            L.oracle_half_to_double.restype = C.c_double
            L.oracle_float_to_half.argtypes = [C.c_float]
            L.oracle_float_to_half.restype = C.c_uint16
            for q in ("q8_0", "q8_1", "q8_k"):
                f = getattr(L, f"oracle_quantize_{q}")
                f.argtypes = [I64, I64, P, P]
                f.restype = None
            L.oracle_q4k_scale_min.argtypes = [P, I, P, P]
            L.oracle_weight_value.argtypes = [I, P, I64]
            L.oracle_weight_value.restype = C.c_double
            L.oracle_act_value.argtypes = [I, P, I64]
            L.oracle_act_value.restype = C.c_double
            L.oracle_matmul.argtypes = [I, I64, I64, I64, P, P, P, P]
            L.oracle_matmul.restype = I
            L.oracle_matmul_rows.argtypes = [I, I64, I64, I64, P, P, I64, I64, P, P]
            L.oracle_matmul_rows.restype = I
            L.oracle_moe.argtypes = [I64] * 5 + [P] * 12
            L.oracle_moe.restype = I
            L.oracle_moe_down.argtypes = [I64] * 5 + [P] * 7
            L.oracle_moe_down.restype = I
            L.oracle_swiglu.argtypes = [I, I64, I64, I64, P, P, P, P, P]
            L.oracle_swiglu.restype = I
            L.oracle_repack_size.argtypes = [I, I64, I64]
            L.oracle_repack_size.restype = I64
            L.oracle_repack.argtypes = [I, I64, I64, P, P]
            L.oracle_repack.restype = I
            _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(C.c_void_p) if a is not None else None


def half_to_double(bits: int) -> float:
    return lib().oracle_half_to_double(bits)


def float_to_half(x: float) -> int:
    return lib().oracle_float_to_half(x)


def quantize(act_fmt: int, x: np.ndarray) -> np.ndarray:
    """fp32 [M, K] -> bytes [M, row_bytes] in Q8_0 / Q8_1 / Q8_K."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    out = np.zeros((M, row_bytes(act_fmt, K)), np.uint8)
    name = {Q8_0: "q8_0", Q8_1: "q8_1", Q8_K: "q8_k"}[act_fmt]
    getattr(lib(), f"oracle_quantize_{name}")(M, K, _p(x), _p(out))
    return out


def q4k_scale_min(scale_bytes: bytes, j: int):
    S = np.frombuffer(bytes(scale_bytes), np.uint8).copy()
    sc, mn = C.c_int(), C.c_int()
    lib().oracle_q4k_scale_min(_p(S), j, C.byref(sc), C.byref(mn))
    return sc.value, mn.value


def weight_value(fmt: int, row: np.ndarray, k: int) -> float:
    row = np.ascontiguousarray(row, dtype=np.uint8)
    return lib().oracle_weight_value(fmt, _p(row), k)


def act_value(fmt: int, row: np.ndarray, k: int) -> float:
    row = np.ascontiguousarray(row, dtype=np.uint8)
    return lib().oracle_act_value(fmt, _p(row), k)


def matmul(wfmt: int, W: np.ndarray, xq: np.ndarray, K: int, rows=None):
    """y[m][n] (fp64) and sum|terms| for the rows ``rows`` (a range or None = all).

    W: [N, row_bytes] uint8; xq: [M, act_row_bytes] uint8.
    Returns (y, absterms), each [M, N]; columns outside ``rows`` are NaN."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    N, M = W.shape[0], xq.shape[0]
    y = np.full((M, N), np.nan)
    at = np.full((M, N), np.nan)
    n0, n1 = (0, N) if rows is None else (rows.start, rows.stop)
    rc = lib().oracle_matmul_rows(wfmt, M, N, K, _p(W), _p(xq), n0, n1, _p(y), _p(at))
    if rc != 0:
        raise ValueError("oracle_matmul rejected its arguments")
    return y, at


def swiglu(wfmt: int, Wg: np.ndarray, Wu: np.ndarray, xq: np.ndarray, K: int):
    """Dense SwiGLU gate / up in fp64: h [M, F] = silu(Wg . x) * (Wu . x), and
    aux [M, F, 4] = (g, u, sum|terms| of g, sum|terms| of u)."""
    Wg, Wu = (np.ascontiguousarray(a, dtype=np.uint8) for a in (Wg, Wu))
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    F, M = Wg.shape[0], xq.shape[0]
    h = np.zeros((M, F))
    aux = np.zeros((M, F, 4))
    rc = lib().oracle_swiglu(wfmt, M, F, K, _p(Wg), _p(Wu), _p(xq), _p(h), _p(aux))
    if rc != 0:
        raise ValueError("oracle_swiglu rejected its arguments")
    return h, aux


def moe(Wg, Wu, Wd, ids, rw, xq, K: int, F: int):
    """Routed expert FFN in fp64. Returns dict(y, y_abs, h, hq, gu_aux)."""
    E = Wg.shape[0]
    T, topk = ids.shape
    Wg, Wu, Wd = (np.ascontiguousarray(a, dtype=np.uint8) for a in (Wg, Wu, Wd))
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    rw = np.ascontiguousarray(rw, dtype=np.float32)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    y = np.zeros((T, K))
    y_abs = np.zeros((T, K))
    h = np.zeros((T, topk, F))
    hq = np.zeros((T, topk, row_bytes(Q8_0, F)), np.uint8)
    aux = np.zeros((T, topk, F, 4))
    scratch = np.zeros(2 * F)
    rc = lib().oracle_moe(T, K, F, E, topk, _p(Wg), _p(Wu), _p(Wd), _p(ids), _p(rw), _p(xq),
                          _p(y), _p(y_abs), _p(h), _p(hq), _p(aux), _p(scratch))
    if rc != 0:
        raise ValueError("oracle_moe rejected its arguments")
    return dict(y=y, y_abs=y_abs, h=h, hq=hq, gu_aux=aux)


def moe_down(Wd, ids, rw, hq, K: int, F: int, valid=None):
    """The routed FFN from given hidden quantisations on: per (token, slot) the
    down projection of hq[t][s] (Q8_0 rows over F), combined with the router
    weights, in fp64. Pairs with valid == 0 are skipped. Returns (y, y_abs), [T, K]."""
    E = Wd.shape[0]
    T, topk = ids.shape
    Wd = np.ascontiguousarray(Wd, dtype=np.uint8)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    rw = np.ascontiguousarray(rw, dtype=np.float32)
    hq = np.ascontiguousarray(hq, dtype=np.uint8).reshape(T, topk, row_bytes(Q8_0, F))
    v = None if valid is None else np.ascontiguousarray(valid, dtype=np.int32).reshape(T, topk)
    y = np.zeros((T, K))
    y_abs = np.zeros((T, K))
    rc = lib().oracle_moe_down(T, K, F, E, topk, _p(Wd), _p(ids), _p(rw), _p(v) if v is not None else None,
                               _p(hq), _p(y), _p(y_abs))
    if rc != 0:
        raise ValueError("oracle_moe_down rejected its arguments")
    return y, y_abs


def repack_size(fmt: int, N: int, K: int) -> int:
    """Bytes of the packed layout of an N x K weight matrix (-1 if not packable)."""
    return lib().oracle_repack_size(fmt, N, K)


def repack(fmt: int, W: np.ndarray, K: int) -> np.ndarray:
    """The packed layout (cq_repack's, include/cq.h) of W [N, row_bytes], as uint8 bytes."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    size = repack_size(fmt, W.shape[0], K)
    if size < 0:
        raise ValueError("oracle_repack_size rejected its arguments")
    out = np.zeros(size, np.uint8)
    if lib().oracle_repack(fmt, W.shape[0], K, _p(W), _p(out)) != 0:
        raise ValueError("oracle_repack rejected its arguments")
    return out
