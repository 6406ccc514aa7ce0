"""The C ABI without a GPU: the library builds, loads, exports every symbol
include/cq.h declares, and rejects bad arguments before touching the device."""
import ctypes as C
import os
import re

import pytest

from gemm_gguf_block_gb300 import build, cq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return cq.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "cq.h")).read()
    return sorted(set(re.findall(r"\b(cq_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
        assert n in cq.SIGNATURES, f"binding lacks {n}"


def test_status_strings(L):
    for s in range(9):
        assert cq.status_string(s)
    assert cq.status_string(0) == "ok"


A = 1 << 20   # an aligned fake address: validation fails before it is ever used


@pytest.mark.parametrize("fn", ["cq_gemv", "cq_gemm"])
def test_validation_before_launch(L, fn):
    f = getattr(cq, fn)
    fmt = cq.Q4_K
    assert f(99, 1, 8, 256, A, A, A) == cq.ERR_UNSUPPORTED_FORMAT
    assert f(cq.Q8_1, 1, 8, 256, A, A, A) == cq.ERR_UNSUPPORTED_FORMAT
    assert f(fmt, 1, 8, 100, A, A, A) == cq.ERR_SHAPE          # K % 256
    assert f(fmt, 1, 8, 0, A, A, A) == cq.ERR_SHAPE
    assert f(fmt, -1, 8, 256, A, A, A) == cq.ERR_INVALID_ARG
    assert f(fmt, 1, 8, 256, A + 4, A, A) == cq.ERR_ALIGNMENT
    assert f(fmt, 1, 8, 256, A, A + 2, A) == cq.ERR_ALIGNMENT
    assert f(fmt, 1, 8, 256, A, A, A + 2) == cq.ERR_ALIGNMENT
    assert f(fmt, 1, 8, 256, None, A, A) == cq.ERR_INVALID_ARG
    assert f(fmt, 0, 8, 256, None, None, None) == cq.OK       # empty: a no-op
    assert f(fmt, 3, 0, 256, None, None, None) == cq.OK


def test_gemv_token_limit(L):
    assert cq.cq_gemv(cq.Q8_0, 17, 8, 256, A, A, A) == cq.ERR_SHAPE


def test_gemm_32_block_formats(L):
    """cq_gemm takes Q4_0 / Q4_1 / Q8_0 at any M; their activation rows go
    through TMA, so xq must be 16-byte aligned. cq_gemm_ws takes one operand
    image per 64 tokens and 128 columns: 17408 bytes (Q8_0 activations) or
    18432 (Q8_1, with the s table)."""
    for fmt, img in ((cq.Q4_0, 17408), (cq.Q4_1, 18432), (cq.Q8_0, 17408)):
        assert cq.cq_gemm_workspace_size(fmt, 512, 4096, 4096) == 8 * 32 * img
        assert cq.cq_gemm_workspace_size(fmt, 65, 8, 256) == 2 * 2 * img
        assert cq.cq_gemm(fmt, 4, 8, 100, A, A, A) == cq.ERR_SHAPE
        assert cq.cq_gemm(fmt, 4, 8, 256, A, A + 4, A) == cq.ERR_ALIGNMENT
        assert cq.cq_gemm(fmt, 4, 8, 256, A + 2, A, A) == cq.ERR_ALIGNMENT
        assert cq.cq_gemm(fmt, 4, 8, 256, A, None, A) == cq.ERR_INVALID_ARG
        assert cq.cq_gemm(fmt, 0, 8, 256, None, None, None) == cq.OK
        need = cq.cq_gemm_workspace_size(fmt, 4, 8, 256)
        assert need == 2 * img
        assert cq.cq_gemm_ws(fmt, 4, 8, 256, A, A, A, None, need) == cq.ERR_WORKSPACE
        assert cq.cq_gemm_ws(fmt, 4, 8, 256, A, A, A, A, need - 1) == cq.ERR_WORKSPACE
        assert cq.cq_gemm_ws(fmt, 4, 8, 256, A, A, A, A + 128, need) == cq.ERR_ALIGNMENT
        assert cq.cq_gemm_ws(fmt, 4, 8, 256, A, A + 8, A, A, need) == cq.ERR_ALIGNMENT
        assert cq.cq_gemm_ws(fmt, 0, 8, 256, None, None, None, None, 0) == cq.OK


def test_gemm_ws_validation(L):
    need = cq.cq_gemm_workspace_size(cq.Q4_K, 512, 14336, 4096)
    assert need == 4 * 16 * (69632 + 512)
    assert cq.cq_gemm_workspace_size(cq.Q6_K, 512, 14336, 4096) == 0
    assert cq.cq_gemm_workspace_size(cq.Q4_K, 512, 14336, 100) == 0
    f = cq.cq_gemm_ws
    assert f(cq.Q6_K, 4, 8, 2048, A, A, A, A, need) == cq.ERR_UNSUPPORTED_FORMAT
    assert f(cq.Q4_K, 4, 8, 100, A, A, A, A, need) == cq.ERR_SHAPE
    small = cq.cq_gemm_workspace_size(cq.Q4_K, 4, 8, 256)
    assert small > 0
    assert f(cq.Q4_K, 4, 8, 256, A, A, A, None, small) == cq.ERR_WORKSPACE
    assert f(cq.Q4_K, 4, 8, 256, A, A, A, A, small - 1) == cq.ERR_WORKSPACE
    assert f(cq.Q4_K, 4, 8, 256, A, A, A, A + 16, small) == cq.ERR_ALIGNMENT
    assert f(cq.Q4_K, 4, 8, 256, A, A + 2, A, A, small) == cq.ERR_ALIGNMENT
    assert f(cq.Q4_K, 0, 8, 256, None, None, None, None, 0) == cq.OK


def test_gemv_x_validation(L):
    f = cq.cq_gemv_x
    assert f(99, 1, 8, 256, A, A, A, A) == cq.ERR_UNSUPPORTED_FORMAT
    assert f(cq.Q8_0, 17, 8, 256, A, A, A, A) == cq.ERR_SHAPE
    assert f(cq.Q8_0, 1, 8, 100, A, A, A, A) == cq.ERR_SHAPE
    assert f(cq.Q8_0, 1, 8, 256, A, None, A, A) == cq.ERR_INVALID_ARG
    assert f(cq.Q8_0, 1, 8, 256, A, A, None, A) == cq.ERR_INVALID_ARG
    assert f(cq.Q8_0, 1, 8, 256, A, A + 4, A, A) == cq.ERR_ALIGNMENT
    assert f(cq.Q8_0, 1, 8, 256, A, A, A + 4, A) == cq.ERR_ALIGNMENT
    assert f(cq.Q8_0, 1, 8, 256, A, A, A, A + 4) == cq.ERR_ALIGNMENT
    assert f(cq.Q8_0, 0, 8, 256, None, None, None, None) == cq.OK


def test_q6k_shape_rule(L):
    """Q6_K rows reach a 16-byte boundary only every eight superblocks: K % 2048."""
    assert cq.cq_gemv(cq.Q6_K, 1, 8, 256, A, A, A) == cq.ERR_SHAPE
    assert cq.cq_gemv(cq.Q6_K, 1, 8, 3072, A, A, A) == cq.ERR_SHAPE
    assert cq.cq_gemv_x(cq.Q6_K, 1, 8, 1024, A, A, A, A) == cq.ERR_SHAPE
    assert cq.cq_gemv_swiglu(cq.Q6_K, 1, 8, 512, A, A, A, A) == cq.ERR_SHAPE
    assert cq.cq_gemm(cq.Q6_K, 4, 8, 2048, A, A, A) == cq.ERR_UNSUPPORTED_FORMAT
    assert cq.cq_gemv(cq.Q6_K, 0, 8, 2048, None, None, None) == cq.OK


def test_q5k_shape_rule(L):
    """Q5_K rows are 176 bytes a superblock, so any K % 256 == 0 keeps them aligned."""
    assert cq.cq_gemv(cq.Q5_K, 1, 8, 128, A, A, A) == cq.ERR_SHAPE
    assert cq.cq_gemv(cq.Q5_K, 1, 8, 300, A, A, A) == cq.ERR_SHAPE
    assert cq.cq_gemv_x(cq.Q5_K, 1, 8, 1000, A, A, A, A) == cq.ERR_SHAPE
    assert cq.cq_gemv_swiglu(cq.Q5_K, 1, 8, 640, A, A, A, A) == cq.ERR_SHAPE
    assert cq.cq_gemm(cq.Q5_K, 4, 8, 2048, A, A, A) == cq.ERR_UNSUPPORTED_FORMAT
    assert cq.cq_gemv(cq.Q5_K, 0, 8, 256, None, None, None) == cq.OK
    assert cq.cq_gemv_x(cq.Q5_K, 0, 8, 768, None, None, None, None) == cq.OK


def test_gemv_swiglu_validation(L):
    f = cq.cq_gemv_swiglu
    assert f(99, 1, 8, 256, A, A, A, A) == cq.ERR_UNSUPPORTED_FORMAT
    assert f(cq.Q8_1, 1, 8, 256, A, A, A, A) == cq.ERR_UNSUPPORTED_FORMAT
    assert f(cq.Q4_K, 17, 8, 256, A, A, A, A) == cq.ERR_SHAPE
    assert f(cq.Q4_K, 0, 8, 256, A, A, A, A) == cq.ERR_SHAPE
    assert f(cq.Q4_K, 1, 0, 256, A, A, A, A) == cq.ERR_SHAPE
    assert f(cq.Q4_K, 1, 8, 100, A, A, A, A) == cq.ERR_SHAPE
    assert f(cq.Q8_0, 1, 8, 65536, A, A, A, A) == cq.ERR_SHAPE        # 1024 chunks > 512
    assert f(cq.Q4_K, 1, 8, 256, None, A, A, A) == cq.ERR_INVALID_ARG
    assert f(cq.Q4_K, 1, 8, 256, A, None, A, A) == cq.ERR_INVALID_ARG
    assert f(cq.Q4_K, 1, 8, 256, A, A, A, None) == cq.ERR_INVALID_ARG
    assert f(cq.Q4_K, 1, 8, 256, A + 4, A, A, A) == cq.ERR_ALIGNMENT
    assert f(cq.Q4_K, 1, 8, 256, A, A + 8, A, A) == cq.ERR_ALIGNMENT
    assert f(cq.Q4_K, 1, 8, 256, A, A, A + 2, A) == cq.ERR_ALIGNMENT
    assert f(cq.Q4_K, 1, 8, 256, A, A, A, A + 4) == cq.ERR_ALIGNMENT


def test_selftest_validation(L):
    assert cq.cq_selftest_wait_timeout(10)[0] == cq.ERR_INVALID_ARG
    assert cq.cq_selftest_wait_timeout(2_000_000_000)[0] == cq.ERR_INVALID_ARG


def test_set_option(L):
    assert cq.cq_set_option(cq.OPT_WEIGHTS_CONST, 1) == cq.OK
    assert cq.cq_set_option(cq.OPT_WEIGHTS_CONST, 0) == cq.OK
    assert cq.cq_set_option(cq.OPT_WEIGHTS_CONST, 2) == cq.ERR_INVALID_ARG
    assert cq.cq_set_option(99, 1) == cq.ERR_INVALID_ARG


def test_quantize_validation(L):
    assert cq.cq_quantize_act(cq.Q4_0, 1, 256, A, A) == cq.ERR_UNSUPPORTED_FORMAT
    assert cq.cq_quantize_act(cq.Q8_0, 1, 96, A, A) == cq.ERR_SHAPE
    assert cq.cq_quantize_act(cq.Q8_K, 1, 256, A + 4, A) == cq.ERR_ALIGNMENT
    assert cq.cq_quantize_act(cq.Q8_1, 0, 256, None, None) == cq.OK


def test_moe_validation(L):
    ws = cq.cq_moe_workspace_size(256, 2048, 1792, 32, 4)
    assert ws > 0
    st, so, ho, qo = cq.cq_moe_workspace_offsets(256, 2048, 1792, 32, 4)
    assert st == cq.OK and so % 256 == 0 and ho % 256 == 0 and qo % 256 == 0
    assert max(so, ho, qo) < ws
    args = dict(T=4, K=256, F=256, E=8, topk=2)
    need = cq.cq_moe_workspace_size(*args.values())

    def call(fmt=cq.Q4_0, ws_bytes=need, ws=A, **kw):
        a = {**args, **kw}
        return cq.cq_moe_gemv(fmt, a["T"], a["K"], a["F"], a["E"], a["topk"], A, A, A, A, A, A, A, ws, ws_bytes)

    assert call(fmt=cq.Q8_0) == cq.ERR_UNSUPPORTED_FORMAT
    assert call(ws_bytes=need - 1) == cq.ERR_WORKSPACE
    assert call(ws=None) == cq.ERR_WORKSPACE
    assert call(ws=A + 16) == cq.ERR_ALIGNMENT      # workspace must be 256-byte aligned
    assert call(K=300) == cq.ERR_SHAPE
    assert call(F=200) == cq.ERR_SHAPE
    assert call(topk=9) == cq.ERR_SHAPE             # topk > E
    assert call(topk=0) == cq.ERR_SHAPE
    assert call(E=300) == cq.ERR_SHAPE
    assert call(T=0) == cq.OK


def test_status_readers_validate(L):
    """The status read-outs reject a null out_code before touching the device."""
    assert L.cq_read_device_status(None, None, None) == cq.ERR_INVALID_ARG
    assert L.cq_read_device_status(A, None, None) == cq.ERR_INVALID_ARG
    assert L.cq_moe_noalloc_read_status(None, None) == cq.ERR_INVALID_ARG
    assert L.cq_moe_read_status(None, None, None) == cq.ERR_INVALID_ARG


def test_library_reads_no_environment():
    """Kernel choices are fixed in the code: no source of the library reads an
    environment variable, so nothing outside a call's arguments and
    cq_set_option can change which kernel runs."""
    csrc = os.path.join(ROOT, "gemm_gguf_block_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, name)).read()
        assert "getenv" not in text and "secure_getenv" not in text, name


def test_repack_validation(L):
    assert cq.cq_repack_size(cq.Q4_0, 16, 256) == 16 * 8 * 18
    assert cq.cq_repack_size(cq.Q4_1, 17, 256) == 32 * 8 * 20       # rows padded to 16
    assert cq.cq_repack_size(cq.Q8_0, 1, 512) == 16 * 16 * 34
    assert cq.cq_repack_size(cq.Q4_K, 16, 256) == 0
    assert cq.cq_repack_size(cq.Q4_0, 16, 100) == 0
    f = cq.cq_repack
    assert f(cq.Q4_K, 16, 256, A, A) == cq.ERR_UNSUPPORTED_FORMAT
    assert f(cq.Q4_0, 16, 100, A, A) == cq.ERR_SHAPE
    assert f(cq.Q4_0, -1, 256, A, A) == cq.ERR_INVALID_ARG
    assert f(cq.Q4_0, 16, 256, None, A) == cq.ERR_INVALID_ARG
    assert f(cq.Q4_0, 16, 256, A, None) == cq.ERR_INVALID_ARG
    assert f(cq.Q4_0, 16, 256, A + 2, A) == cq.ERR_ALIGNMENT
    assert f(cq.Q4_0, 16, 256, A, A + 8) == cq.ERR_ALIGNMENT
    assert f(cq.Q4_0, 0, 256, None, None) == cq.OK
    g = cq.cq_gemv_packed
    assert g(cq.Q4_K, 1, 8, 256, A, A, A) == cq.ERR_UNSUPPORTED_FORMAT
    assert g(cq.Q4_1, 17, 8, 256, A, A, A) == cq.ERR_SHAPE
    assert g(cq.Q4_1, 1, 8, 100, A, A, A) == cq.ERR_SHAPE
    assert g(cq.Q4_1, 1, 8, 256, None, A, A) == cq.ERR_INVALID_ARG
    assert g(cq.Q4_1, 1, 8, 256, A + 4, A, A) == cq.ERR_ALIGNMENT
    assert g(cq.Q4_1, 1, 8, 256, A, A + 2, A) == cq.ERR_ALIGNMENT
    assert g(cq.Q4_1, 1, 8, 256, A, A, A + 4) == cq.ERR_ALIGNMENT
    assert g(cq.Q4_1, 0, 8, 256, None, None, None) == cq.OK


def test_gemm_noalloc_validation(L):
    f = cq.cq_gemm_noalloc
    assert f(99, 1, 8, 256, A, A, A) == cq.ERR_UNSUPPORTED_FORMAT
    assert f(cq.Q4_K, 1, 8, 100, A, A, A) == cq.ERR_SHAPE
    assert f(cq.Q4_K, -1, 8, 256, A, A, A) == cq.ERR_INVALID_ARG
    assert f(cq.Q4_K, 1, 8, 256, None, A, A) == cq.ERR_INVALID_ARG
    assert f(cq.Q4_K, 1, 8, 256, A + 4, A, A) == cq.ERR_ALIGNMENT
    assert f(cq.Q4_0, 1, 8, 256, A, A + 4, A) == cq.ERR_ALIGNMENT        # TMA-read activations: 16 bytes
    assert f(cq.Q4_K, 0, 8, 256, None, None, None) == cq.OK
