"""The allocation-free routed-FFN entry point, cq_moe_gemv_noalloc.

Some callers of this library cannot call cudaMalloc: a plugin whose host
framework has reserved the GPU's memory for its own pool and offers no way to
ask for more, or a latency-critical decode loop that cannot take the
device-wide synchronisation an allocation brings. Such a caller cannot hand
cq_moe_gemv a workspace, so cq_moe_gemv_noalloc keeps its scratch space in a
fixed array inside the library's device image instead.

These tests call it through the C ABI and check that it gives what the
workspace-taking entry point gives on the same inputs -- within the parity
tolerance of the other tests, and in fact bit for bit -- on two calls in a
row with different problems, so that anything the first call leaves in the
shared array is seen by the second. This file is collected last on purpose.
"""
import numpy as np
import pytest

from gemm_gguf_block_gb300 import cq, synth
from helpers import TOL, cq_built, dev, torch_cuda

A = 1 << 20   # a fake aligned device address: rejected shapes never reach the device


def _problem(seed, T, E, topk, K, F):
    rng = np.random.default_rng(seed)
    Wg = np.stack([synth.gen_q4_0(rng, F, K) for _ in range(E)])
    Wu = np.stack([synth.gen_q4_0(rng, F, K) for _ in range(E)])
    Wd = np.stack([synth.gen_q4_0(rng, K, F) for _ in range(E)])
    ids, rw = synth.gen_routing(rng, T, E, topk)
    x = rng.standard_normal((T, K)).astype(np.float32)
    return Wg, Wu, Wd, ids, rw, x


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point(orc):
    torch = torch_cuda()
    cq_built()
    stream = torch.cuda.current_stream().cuda_stream
    shapes = [dict(T=24, E=8, topk=3, K=512, F=768), dict(T=40, E=6, topk=2, K=768, F=512)]
    outputs = []
    for i, sh in enumerate(shapes):
        Wg, Wu, Wd, ids, rw, x = _problem(100 + i, **sh)
        t = [dev(torch, a) for a in (Wg, Wu, Wd, ids, rw)]
        xq = cq.quantize_act_t(dev(torch, x), cq.Q8_0)
        y_ws, _ = cq.moe_t(*t, xq, sh["K"], sh["F"])
        y_na = torch.full((sh["T"], sh["K"]), float("nan"), device="cuda")
        st = cq.cq_moe_gemv_noalloc(cq.Q4_0, sh["T"], sh["K"], sh["F"], sh["E"], sh["topk"],
                                    *[a.data_ptr() for a in t], xq.data_ptr(), y_na.data_ptr(), stream)
        assert st == cq.OK, cq.status_string(st)
        torch.cuda.synchronize()
        ref = orc.moe(Wg, Wu, Wd, ids, rw, xq.cpu().numpy(), sh["K"], sh["F"])
        outputs.append((y_ws.cpu().numpy(), y_na.cpu().numpy(), ref["y_abs"]))
    for y_ws, y_na, y_abs in outputs:
        assert np.all(np.isfinite(y_na))
        assert np.all(np.abs(y_na.astype(np.float64) - y_ws) <= TOL * y_abs)
        assert np.array_equal(y_na.view(np.uint32), y_ws.view(np.uint32))


def test_noalloc_rejects_before_launch():
    """Shapes too large for the fixed array, and shapes the workspace entry point
    rejects, fail with a clear status before anything reaches the device."""
    cq_built()
    big = dict(T=4096, K=4096, F=8192, E=64, topk=8)
    assert cq.cq_moe_workspace_size(*big.values()) > (24 << 20)
    st = cq.cq_moe_gemv_noalloc(cq.Q4_0, big["T"], big["K"], big["F"], big["E"], big["topk"],
                                A, A, A, A, A, A, A)
    assert st == cq.ERR_WORKSPACE
    assert cq.cq_moe_gemv_noalloc(cq.Q4_0, 8, 300, 256, 4, 2, A, A, A, A, A, A, A) == cq.ERR_SHAPE
    assert cq.cq_moe_gemv_noalloc(cq.Q8_0, 8, 256, 256, 4, 2, A, A, A, A, A, A, A) == cq.ERR_UNSUPPORTED_FORMAT
    assert cq.cq_moe_gemv_noalloc(cq.Q4_0, 0, 256, 256, 4, 2, A, A, A, A, A, A, A) == cq.OK


@pytest.mark.gpu
def test_noalloc_full_routed_ffn_near_the_cap():
    """The 256-token, 32-expert, 2048/1792 routed FFN, the workload the array is
    sized for (17.7 MB of its 24 MiB): bit for bit what cq_moe_gemv gives."""
    torch = torch_cuda()
    cq_built()
    stream = torch.cuda.current_stream().cuda_stream
    Wg, Wu, Wd, ids, rw, x = synth.moe_ffn(0)
    T, K = x.shape
    E, F = Wg.shape[0], Wg.shape[1]
    assert cq.cq_moe_workspace_size(T, K, F, E, 4) > (16 << 20)
    t = [dev(torch, a) for a in (Wg, Wu, Wd, ids, rw)]
    xq = cq.quantize_act_t(dev(torch, x), cq.Q8_0)
    y_ws, _ = cq.moe_t(*t, xq, K, F)
    y_na = torch.full((T, K), float("nan"), device="cuda")
    st = cq.cq_moe_gemv_noalloc(cq.Q4_0, T, K, F, E, 4, *[a.data_ptr() for a in t], xq.data_ptr(),
                                y_na.data_ptr(), stream)
    assert st == cq.OK, cq.status_string(st)
    assert cq.cq_moe_noalloc_read_status(stream) == (cq.OK, 0)
    assert torch.equal(y_na.view(torch.int32), y_ws.view(torch.int32))


@pytest.mark.gpu
def test_noalloc_status_word_reports_and_clears():
    """A repeated expert id is skipped and reported through the array's status
    word; the next clean call clears it."""
    torch = torch_cuda()
    cq_built()
    stream = torch.cuda.current_stream().cuda_stream
    sh = dict(T=8, E=4, topk=2, K=256, F=256)
    Wg, Wu, Wd, ids, rw, x = _problem(7, **sh)
    xq = cq.quantize_act_t(dev(torch, x), cq.Q8_0)
    y = torch.empty((sh["T"], sh["K"]), device="cuda")
    for ids_call, want in ((np.where(np.arange(2)[None, :] == 1, ids[:, :1], ids), cq.DEV_DUP_EXPERT_ID),
                           (ids, 0)):
        t = [dev(torch, a) for a in (Wg, Wu, Wd, ids_call.astype(np.int32), rw)]
        st = cq.cq_moe_gemv_noalloc(cq.Q4_0, sh["T"], sh["K"], sh["F"], sh["E"], sh["topk"],
                                    *[a.data_ptr() for a in t], xq.data_ptr(), y.data_ptr(), stream)
        assert st == cq.OK
        st, code = cq.cq_moe_noalloc_read_status(stream)
        assert code == want and st == (cq.ERR_DEVICE_STATUS if want else cq.OK)
