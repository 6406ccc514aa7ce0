"""Python binding of libcq (include/cq.h): argument marshalling only.

The raw functions carry the C names and arguments (integers for pointers and
the stream) and return the integer cq_status. The ``*_t`` helpers take torch
CUDA tensors, allocate outputs with torch, call the C function on the current
stream and raise ``CqError`` on a non-zero status. Every step of the
computation runs in libcq's CUDA kernels; there is no other path. Importing
this module does not need a GPU; calling it does, and a missing libcq.so is
an error, never a fallback.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libcq.so")

Q4_0, Q4_1, Q8_0, Q8_1, Q4_K, Q5_K, Q6_K, Q8_K = 2, 3, 8, 9, 12, 13, 14, 15
ACT_FOR = {Q4_0: Q8_0, Q8_0: Q8_0, Q4_1: Q8_1, Q4_K: Q8_K, Q5_K: Q8_K, Q6_K: Q8_K}
BLOCK = {Q4_0: (32, 18), Q4_1: (32, 20), Q8_0: (32, 34), Q8_1: (32, 36), Q4_K: (256, 144), Q5_K: (256, 176),
         Q6_K: (256, 210), Q8_K: (256, 292)}
FMT = {"q4_0": Q4_0, "q4_1": Q4_1, "q8_0": Q8_0, "q8_1": Q8_1, "q4_k": Q4_K, "q5_k": Q5_K, "q6_k": Q6_K,
       "q8_k": Q8_K}

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_FORMAT, ERR_SHAPE, ERR_ALIGNMENT, ERR_WORKSPACE, ERR_CUDA, \
    ERR_DEVICE_STATUS, ERR_TIMEOUT = range(9)
DEV_BAD_EXPERT_ID, DEV_DUP_EXPERT_ID, DEV_WAIT_TIMEOUT = 0x1, 0x2, 0x4

# Every symbol include/cq.h declares, with (restype, argtypes).
_P, _I64, _I, _SZ = C.c_void_p, C.c_int64, C.c_int, C.c_size_t
SIGNATURES = {
    "cq_quantize_act": (_I, [_I, _I64, _I64, _P, _P, _P]),
    "cq_gemv": (_I, [_I, _I64, _I64, _I64, _P, _P, _P, _P]),
    "cq_gemv_x": (_I, [_I, _I64, _I64, _I64, _P, _P, _P, _P, _P]),
    "cq_gemv_swiglu": (_I, [_I, _I64, _I64, _I64, _P, _P, _P, _P, _P]),
    "cq_gemm": (_I, [_I, _I64, _I64, _I64, _P, _P, _P, _P]),
    "cq_gemm_noalloc": (_I, [_I, _I64, _I64, _I64, _P, _P, _P, _P]),
    "cq_gemm_workspace_size": (_SZ, [_I, _I64, _I64, _I64]),
    "cq_gemm_ws": (_I, [_I, _I64, _I64, _I64, _P, _P, _P, _P, _SZ, _P]),
    "cq_moe_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _I64]),
    "cq_moe_gemv": (_I, [_I, _I64, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "cq_moe_gemv_noalloc": (_I, [_I, _I64, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P]),
    "cq_moe_workspace_offsets": (_I, [_I64, _I64, _I64, _I64, _I64, _P, _P, _P]),
    "cq_moe_read_status": (_I, [_P, _P, _P]),
    "cq_moe_noalloc_read_status": (_I, [_P, _P]),
    "cq_read_device_status": (_I, [_P, _P, _P]),
    "cq_read_global_status": (_I, [_P, _I]),
    "cq_status_string": (C.c_char_p, [_I]),
    "cq_set_option": (_I, [_I, _I64]),
    "cq_selftest_wait_timeout": (_I, [_I64, _P, _P]),
    "cq_repack_size": (_SZ, [_I, _I64, _I64]),
    "cq_repack": (_I, [_I, _I64, _I64, _P, _P, _P]),
    "cq_gemv_packed": (_I, [_I, _I64, _I64, _I64, _P, _P, _P, _P]),
}

OPT_WEIGHTS_CONST = 1

_lock = threading.Lock()
_lib = None


class CqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_string(status)} (status {status})")
        self.status = status


def lib(path: str | None = None):
    """Load libcq.so (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"{p} is missing: build it with `python -m gemm_gguf_block_gb300.build`")
            L = C.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype, f.argtypes = res, args
            if path is not None:
                return L
            _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().cq_status_string(s).decode()


# ------------------------------------------------------------------ raw C calls
def cq_quantize_act(act_fmt, M, K, x, xq, stream=0):
    return lib().cq_quantize_act(act_fmt, M, K, x, xq, stream)


def cq_gemv(w_fmt, M, N, K, W, xq, y, stream=0):
    return lib().cq_gemv(w_fmt, M, N, K, W, xq, y, stream)


def cq_gemv_x(w_fmt, M, N, K, W, x, xq, y, stream=0):
    return lib().cq_gemv_x(w_fmt, M, N, K, W, x, xq, y, stream)


def cq_gemv_swiglu(w_fmt, M, F, K, W_gate, W_up, xq, h, stream=0):
    return lib().cq_gemv_swiglu(w_fmt, M, F, K, W_gate, W_up, xq, h, stream)


def cq_gemm(w_fmt, M, N, K, W, xq, y, stream=0):
    return lib().cq_gemm(w_fmt, M, N, K, W, xq, y, stream)


def cq_gemm_noalloc(w_fmt, M, N, K, W, xq, y, stream=0):
    return lib().cq_gemm_noalloc(w_fmt, M, N, K, W, xq, y, stream)


def cq_selftest_wait_timeout(limit_ns, stream=0):
    """(status, device code) of the bounded-wait self-test."""
    code = C.c_int32(0)
    st = lib().cq_selftest_wait_timeout(limit_ns, C.byref(code), stream)
    return st, code.value


def cq_set_option(opt, value):
    return lib().cq_set_option(opt, value)


def cq_repack_size(w_fmt, N, K):
    return lib().cq_repack_size(w_fmt, N, K)


def cq_repack(w_fmt, N, K, W, Wp, stream=0):
    return lib().cq_repack(w_fmt, N, K, W, Wp, stream)


def cq_gemv_packed(w_fmt, M, N, K, Wp, xq, y, stream=0):
    return lib().cq_gemv_packed(w_fmt, M, N, K, Wp, xq, y, stream)


def cq_gemm_workspace_size(w_fmt, M, N, K):
    return lib().cq_gemm_workspace_size(w_fmt, M, N, K)


def cq_gemm_ws(w_fmt, M, N, K, W, xq, y, ws, ws_bytes, stream=0):
    return lib().cq_gemm_ws(w_fmt, M, N, K, W, xq, y, ws, ws_bytes, stream)


def cq_moe_workspace_size(T, K, F, E, topk):
    return lib().cq_moe_workspace_size(T, K, F, E, topk)


def cq_moe_gemv(w_fmt, T, K, F, E, topk, W_gate, W_up, W_down, ids, route_w, xq, y, ws, ws_bytes, stream=0):
    return lib().cq_moe_gemv(w_fmt, T, K, F, E, topk, W_gate, W_up, W_down, ids, route_w, xq, y, ws,
                             ws_bytes, stream)


def cq_moe_gemv_noalloc(w_fmt, T, K, F, E, topk, W_gate, W_up, W_down, ids, route_w, xq, y, stream=0):
    """Routed FFN without a caller workspace (scratch in a fixed device array of the library)."""
    return lib().cq_moe_gemv_noalloc(w_fmt, T, K, F, E, topk, W_gate, W_up, W_down, ids, route_w, xq, y, stream)


def cq_moe_workspace_offsets(T, K, F, E, topk):
    a, b, c = C.c_size_t(), C.c_size_t(), C.c_size_t()
    st = lib().cq_moe_workspace_offsets(T, K, F, E, topk, C.addressof(a), C.addressof(b), C.addressof(c))
    return st, a.value, b.value, c.value


def cq_moe_read_status(ws, stream=0):
    code = C.c_int32()
    st = lib().cq_moe_read_status(ws, C.addressof(code), stream)
    return st, code.value


def cq_moe_noalloc_read_status(stream=0):
    code = C.c_int32()
    st = lib().cq_moe_noalloc_read_status(C.addressof(code), stream)
    return st, code.value


def cq_read_device_status(ws=None, stream=0):
    """(status, code) of a MoE workspace's status word, or (ws None) of the library's own word."""
    code = C.c_int32()
    st = lib().cq_read_device_status(ws, C.addressof(code), stream)
    return st, code.value


def cq_read_global_status(clear=1):
    code = C.c_int32()
    st = lib().cq_read_global_status(C.addressof(code), clear)
    return st, code.value


# --------------------------------------------------------- torch conveniences
def _torch():
    import torch
    return torch


def _stream_handle():
    return _torch().cuda.current_stream().cuda_stream


def row_bytes(fmt: int, K: int) -> int:
    e, b = BLOCK[fmt]
    return K // e * b


def _check(fn, st):
    if st != OK:
        raise CqError(fn, st)


def quantize_act_t(x, act_fmt: int):
    """x: CUDA fp32 [M, K] -> uint8 [M, row_bytes(act_fmt, K)]."""
    torch = _torch()
    M, K = x.shape
    xq = torch.empty((M, row_bytes(act_fmt, K)), dtype=torch.uint8, device=x.device)
    _check("cq_quantize_act", cq_quantize_act(act_fmt, M, K, x.data_ptr(), xq.data_ptr(), _stream_handle()))
    return xq


def gemv_t(W, xq, w_fmt: int, K: int, out=None):
    """W: uint8 [N, row_bytes]; xq: uint8 [M, act_row_bytes] (M <= 16) -> fp32 [M, N]."""
    torch = _torch()
    N, M = W.shape[0], xq.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=W.device)
    _check("cq_gemv", cq_gemv(w_fmt, M, N, K, W.data_ptr(), xq.data_ptr(), y.data_ptr(), _stream_handle()))
    return y


def repack_t(W, w_fmt: int, K: int):
    """cq_repack: W uint8 [N, row_bytes] -> the packed layout, uint8 [cq_repack_size]."""
    torch = _torch()
    N = W.shape[0]
    size = cq_repack_size(w_fmt, N, K)
    if size == 0 and N > 0:
        raise CqError("cq_repack_size", ERR_SHAPE)
    Wp = torch.empty(size, dtype=torch.uint8, device=W.device)
    _check("cq_repack", cq_repack(w_fmt, N, K, W.data_ptr(), Wp.data_ptr(), _stream_handle()))
    return Wp


def gemv_packed_t(Wp, xq, w_fmt: int, N: int, K: int, out=None):
    """cq_gemv_packed: Wp from repack_t; xq uint8 [M, act_row_bytes] (M <= 16) -> fp32 [M, N]."""
    torch = _torch()
    M = xq.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=Wp.device)
    _check("cq_gemv_packed", cq_gemv_packed(w_fmt, M, N, K, Wp.data_ptr(), xq.data_ptr(), y.data_ptr(),
                                            _stream_handle()))
    return y


def gemv_x_t(W, x, w_fmt: int, out=None):
    """cq_gemv_x: x fp32 [M, K] (M <= 16) -> (y fp32 [M, N], xq uint8 [M, act_row_bytes])."""
    torch = _torch()
    M, K = x.shape
    N = W.shape[0]
    xq = torch.empty((M, row_bytes(ACT_FOR[w_fmt], K)), dtype=torch.uint8, device=x.device)
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=x.device)
    _check("cq_gemv_x", cq_gemv_x(w_fmt, M, N, K, W.data_ptr(), x.data_ptr(), xq.data_ptr(), y.data_ptr(),
                                  _stream_handle()))
    return y, xq


def gemv_swiglu_t(Wg, Wu, xq, w_fmt: int, K: int, out=None):
    """cq_gemv_swiglu: Wg, Wu uint8 [F, row_bytes]; xq uint8 [M, act_row_bytes] (M <= 16)
    -> h fp32 [M, F] = silu(Wg . x) * (Wu . x)."""
    torch = _torch()
    F, M = Wg.shape[0], xq.shape[0]
    h = out if out is not None else torch.empty((M, F), dtype=torch.float32, device=Wg.device)
    _check("cq_gemv_swiglu", cq_gemv_swiglu(w_fmt, M, F, K, Wg.data_ptr(), Wu.data_ptr(), xq.data_ptr(),
                                            h.data_ptr(), _stream_handle()))
    return h


def gemm_t(W, xq, w_fmt: int, K: int, out=None):
    torch = _torch()
    N, M = W.shape[0], xq.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=W.device)
    _check("cq_gemm", cq_gemm(w_fmt, M, N, K, W.data_ptr(), xq.data_ptr(), y.data_ptr(), _stream_handle()))
    return y


def gemm_noalloc_t(W, xq, w_fmt: int, K: int, out=None):
    torch = _torch()
    N, M = W.shape[0], xq.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=W.device)
    _check("cq_gemm_noalloc", cq_gemm_noalloc(w_fmt, M, N, K, W.data_ptr(), xq.data_ptr(), y.data_ptr(),
                                              _stream_handle()))
    return y


def gemm_ws_t(W, xq, w_fmt: int, K: int, ws=None, out=None):
    """cq_gemm_ws with a workspace tensor (allocated here when not given)."""
    torch = _torch()
    N, M = W.shape[0], xq.shape[0]
    need = cq_gemm_workspace_size(w_fmt, M, N, K)
    if ws is None:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=W.device)
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=W.device)
    _check("cq_gemm_ws", cq_gemm_ws(w_fmt, M, N, K, W.data_ptr(), xq.data_ptr(), y.data_ptr(), ws.data_ptr(),
                                    ws.numel(), _stream_handle()))
    return y


def moe_t(W_gate, W_up, W_down, ids, route_w, xq, K: int, F: int, ws=None, out=None):
    """Routed FFN. Returns (y [T, K] fp32, workspace uint8 tensor)."""
    torch = _torch()
    E = W_gate.shape[0]
    T, topk = ids.shape
    need = cq_moe_workspace_size(T, K, F, E, topk)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=xq.device)
    y = out if out is not None else torch.empty((T, K), dtype=torch.float32, device=xq.device)
    _check("cq_moe_gemv", cq_moe_gemv(Q4_0, T, K, F, E, topk, W_gate.data_ptr(), W_up.data_ptr(),
                                      W_down.data_ptr(), ids.data_ptr(), route_w.data_ptr(), xq.data_ptr(),
                                      y.data_ptr(), ws.data_ptr(), ws.numel(), _stream_handle()))
    return y, ws
