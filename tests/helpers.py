"""Shared helpers for the parity tests (CUDA path vs the CPU oracle)."""
import numpy as np

TOL = 2e-5   # |y - y_ref| <= TOL * sum|terms| per output (the contract's fp32 bound)

W_NAMES = {2: "q4_0", 3: "q4_1", 8: "q8_0", 12: "q4_k"}


def torch_cuda():
    import pytest
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def cq_built():
    """Build libcq.so (if stale) and return the binding module."""
    from gemm_gguf_block_gb300 import build, cq
    build.build()
    cq.lib()
    return cq


def dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_within(y, y_ref, absterms, tol=TOL, what=""):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = tol * absterms
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs outside the bound; first at {tuple(i)}: "
                             f"got {y[tuple(i)]!r} want {y_ref[tuple(i)]!r} err {err[tuple(i)]:.3e} "
                             f"bound {bound[tuple(i)]:.3e}")
