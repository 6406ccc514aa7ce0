#!/usr/bin/env python
"""Benchmark of the GGUF block-quantized hot path on GB300.

Headline workload: the Q8_0 decode GEMV suite at Llama-3-8B layer shapes,
M = 1 token -- 4096x4096, 1024x4096, 14336x4096, 4096x14336 and the LM head
128256x4096 (705 MB of weights). One step = for each layer, quantise the fp32
activation to Q8_0 (cq_quantize_act) and run the GEMV (cq_gemv). Value: weight
bytes streamed per second over the whole step (GB/s), inputs resident in HBM.
The weights of one step (705 MB) exceed the 129 MB L2, so every step streams
them from HBM.

Also printed in the same JSON line: the prefill GEMMs (Q4_K, and Q8_0 / Q4_0 /
Q4_1; M=512, K=4096, N=14336) in int8-equivalent TOPS, the routed-expert FFN
and the Q4_1 LM head at M = 1/4/8/16, the single-call latency of the small
Q4_0 GEMV, the fused dense SwiGLU gate + up projection (Q4_K 14336x4096 each,
M = 1/4), the Q6_K tied-embedding LM head (128256x2048, M = 1/4), the Q5_K
FFN gate projection (14336x4096, M = 1/4), the roofline of the dominant
kernel, the CPU oracle's rate on the host cores, and the end-to-end rate with
host buffers.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl cq|reference]

Multi-GPU (torchrun): every rank runs its own replica of the workload (the
path has no exchange step); the time is the maximum over ranks and the value
is the aggregate over all ranks (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode GEMV weight GB/s (% of HBM peak); prefill GEMM int8 TOPS (% of peak)"
WORKLOAD = ("Q8_0 decode GEMV suite, Llama-3-8B layer shapes (NxK) 4096x4096, 1024x4096, 14336x4096, "
            "4096x14336, 128256x4096; M=1 token; activations fp32 N(0,1) quantized to Q8_0 in-step")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def _traffic(kernel_file: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on the
    current source of the kernels it covers (the summary records a hash of the
    decode step's sources: the quantiser, the GEMV and their headers)."""
    path = os.path.join(ROOT, "profiles", kernel_file)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s*\(source sha256 ([0-9a-f]+)\)", text)
    if not m:
        return None
    from gemm_gguf_block_gb300.build import GEMV_STEP_SOURCES, source_hash
    return float(m.group(1)) if source_hash(GEMV_STEP_SOURCES) == m.group(2) else None


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in the background."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def window(self, t0, t1):
        return [r for (t, r) in self.rows if t0 <= t <= t1]

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    @staticmethod
    def summary(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if len(r) > 5 + i and r[5 + i] == "Active"})
        pw = [float(r[3]) for r in rows if re.match(r"^[0-9.]+$", r[3])]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


def _gpu_query_id(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev] if vis else str(dev)


# --------------------------------------------------------------- CPU oracle
def _oracle_suite(suite, row_frac=1.0):
    """The oracle over the suite (or the first row_frac of each matrix's rows).
    Returns (seconds, weight bytes processed)."""
    import oracle
    t = time.perf_counter()
    nbytes = 0
    for W, x in suite:
        K = x.shape[1]
        rows = max(1, int(W.shape[0] * row_frac))
        xq = oracle.quantize(oracle.Q8_0, x)
        oracle.matmul(oracle.Q8_0, W[:rows], xq, K)
        nbytes += W[:rows].nbytes
    return time.perf_counter() - t, nbytes


def host_cpu():
    """The host's CPU model and core counts (lscpu, else /proc/cpuinfo and os.cpu_count)."""
    info = {"logical_cpus": os.cpu_count(), "machine": os.uname().machine}
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        kv = dict(line.split(":", 1) for line in out.splitlines() if ":" in line)
        kv = {k.strip(): v.strip() for k, v in kv.items()}
        for key, name in (("Model name", "model"), ("Socket(s)", "sockets"),
                          ("Core(s) per socket", "cores_per_socket"), ("Thread(s) per core", "threads_per_core"),
                          ("CPU(s)", "logical_cpus")):
            if key in kv:
                v = kv[key]
                info[name] = int(v) if v.isdigit() else v
    except (OSError, subprocess.SubprocessError, ValueError):
        pass
    if "model" not in info:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part")):
                    info["model"] = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    if isinstance(info.get("sockets"), int) and isinstance(info.get("cores_per_socket"), int):
        info["physical_cores"] = info["sockets"] * info["cores_per_socket"]
    elif isinstance(info.get("logical_cpus"), int) and isinstance(info.get("threads_per_core"), int):
        info["physical_cores"] = info["logical_cpus"] // max(1, info["threads_per_core"])
    return info


def cpu_baseline(suite, min_s=8.0, max_reps=20):
    dt_total, b_total, reps = 0.0, 0, 0
    while reps < max_reps and (reps == 0 or dt_total < min_s):
        dt, b = _oracle_suite(suite)
        dt_total += dt
        b_total += b
        reps += 1
    return {"value": b_total / dt_total / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "host": host_cpu(),
            "sample": f"the whole Q8_0 suite step (quantise + all 5 matrices), {reps} repetition(s), "
                      f"{dt_total:.1f} s single-threaded (1 of the host's cores)"}


# ----------------------------------------------------------------- reference
def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    from gemm_gguf_block_gb300 import synth
    oracle.build()
    suite = synth.decode_q8_0_suite(args.seed)
    frac = 1.0 / 64
    for _ in range(args.warmup):
        _oracle_suite(suite, frac)
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        _, b = _oracle_suite(suite, frac)
        nbytes += b
    dt = time.perf_counter() - t0
    v = nbytes / dt / 1e9
    sample = "first 1/64 of the rows of each of the 5 matrices, plus the full activation quantisation, per step"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "i8xi8->i64, f64 scales", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
                         "host": host_cpu()},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ------------------------------------------------------------- multi-rank
def dist_init(world):
    """gloo process group for the replicas' barrier and timing reduction (None at N=1)."""
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group("gloo")
    return dist


def max_over_ranks(dist, v):
    """The largest of every rank's value (a no-op without a process group)."""
    if dist is None:
        return v
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0])


def aggregate_gbs(world, bytes_per_rank_step, ms_per_step):
    """Whole-job rate: every rank streams its own replica's bytes per step."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


# --------------------------------------------------------------- GPU timing
def _flush(torch, buf, rbuf):
    """Evict the 129 MB L2 between timed calls: write a 256 MB buffer, then read
    another 256 MB one, so the L2 is left holding clean lines and the timed
    call does not pay for writing the flush's dirty lines back."""
    buf.add_(1)
    rbuf.sum()


def time_calls(torch, fn, iters, warmup, flush=None):
    """Median per-call time (ms) with CUDA events on the current stream."""
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    times = []
    for _ in range(iters):
        if flush is not None:
            flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        b.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times)


class _Ctx:
    """Device helpers shared by the secondary workloads."""

    def __init__(self, torch, iters=10, warmup=3):
        self.torch = torch
        self.iters, self.warmup = iters, warmup
        self.flushbuf = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device="cuda")
        self.flushread = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device="cuda")

    def dev(self, a):
        return self.torch.from_numpy(np.ascontiguousarray(a)).cuda()

    def flush(self):
        _flush(self.torch, self.flushbuf, self.flushread)

    def stream(self):
        return self.torch.cuda.current_stream().cuda_stream

    def time(self, fn, flush=True):
        return time_calls(self.torch, fn, self.iters, self.warmup, self.flush if flush else None)


L2_BYTES = 129e6


def per_shape_rotated(torch, cq, layers, launches_min=60, reps=5):
    """Per decode shape, the GEMV as it runs inside the step: a CUDA graph of
    back-to-back cq_gemv launches (programmatic dependent launch, the
    weights-constant option, as in the step) over rotated copies of that
    shape's weights -- together at least 2.5x the L2, so every launch streams
    its weights from HBM. Per-launch time = graph time / launches (median of
    `reps` replays)."""
    out = []
    sh = torch.cuda.current_stream().cuda_stream
    for L in layers:
        W = L["W"]
        copies = max(1, int(np.ceil(2.5 * L2_BYTES / W.numel())))
        Wc = [W] + [W.clone() for _ in range(copies - 1)]
        n = max(launches_min, copies) // copies * copies
        y = torch.empty_like(L["y"])

        def run(s):
            for i in range(n):
                cq.cq_gemv(cq.Q8_0, 1, L["N"], L["K"], Wc[i % copies].data_ptr(), L["xq"].data_ptr(),
                           y.data_ptr(), s)
        run(sh)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run(torch.cuda.current_stream().cuda_stream)
        g.replay()
        torch.cuda.synchronize()
        ms = time_calls(torch, g.replay, reps, 1)
        us = 1e3 * ms / n
        out.append({"shape": f"{L['N']}x{L['K']}", "us": us, "gbs": L["bytes"] / (us * 1e-6) / 1e9,
                    "copies": copies, "launches": n})
        del Wc, g
        torch.cuda.empty_cache()
    return out


def rotated_graph_us(torch, make_call, nbytes, launches_min=60, reps=5):
    """Per-call time of back-to-back calls in one CUDA graph, as a decode loop
    issues them (programmatic dependent launch, weights-constant option), each
    call on its own copy of the weights -- the copies together at least 2.5x
    the L2, so every call streams from HBM. make_call(i, stream) issues call i
    on copy i; returns (us per call, copies)."""
    copies = max(1, int(np.ceil(2.5 * L2_BYTES / nbytes)))
    n = max(launches_min, copies) // copies * copies
    sh = torch.cuda.current_stream().cuda_stream
    for i in range(copies):
        make_call(i, sh)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream().cuda_stream
        for i in range(n):
            make_call(i % copies, cs)
    g.replay()
    torch.cuda.synchronize()
    us = 1e3 * time_calls(torch, g.replay, reps, 1) / n
    del g
    return us, copies


def case_gemm(c, cq, synth, peaks, seed):
    """Prefill GEMM: Q4_K, M=512, K=4096, N=14336, through cq_gemm_ws (activations
    converted once into the caller's workspace), cq_gemm (the same with a
    workspace from the library's pool) and cq_gemm_noalloc (converted per tile)."""
    W, x = synth.prefill_q4_k(seed)
    M, K = x.shape
    N = W.shape[0]
    Wd, xd = c.dev(W), c.dev(x)
    xq = cq.quantize_act_t(xd, cq.Q8_K)
    y = c.torch.empty((M, N), dtype=c.torch.float32, device="cuda")
    need = cq.cq_gemm_workspace_size(cq.Q4_K, M, N, K)
    ws = c.torch.empty(need, dtype=c.torch.uint8, device="cuda")
    ms = c.time(lambda: cq.cq_gemm_ws(cq.Q4_K, M, N, K, Wd.data_ptr(), xq.data_ptr(), y.data_ptr(), ws.data_ptr(),
                                      need, c.stream()))
    ms_plain = c.time(lambda: cq.cq_gemm(cq.Q4_K, M, N, K, Wd.data_ptr(), xq.data_ptr(), y.data_ptr(), c.stream()))
    ms_na = c.time(lambda: cq.cq_gemm_noalloc(cq.Q4_K, M, N, K, Wd.data_ptr(), xq.data_ptr(), y.data_ptr(),
                                              c.stream()))
    tops = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    return {"shape": f"M={M} N={N} K={K}", "call": "cq_gemm_ws", "ms": ms, "int8_equiv_tops": tops,
            "peak_tflops": peaks["bf16"], "peak_note": "fp16 tensor peak = measured bf16 x 1",
            "frac": tops / peaks["bf16"], "cq_gemm_ms": ms_plain,
            "cq_gemm_tops": 2.0 * M * N * K / (ms_plain * 1e-3) / 1e12, "cq_gemm_noalloc_ms": ms_na}


def case_gemm_32(c, cq, synth, peaks, seed, fmts=("q8_0", "q4_0", "q4_1")):
    """Prefill GEMM of the 32-element formats (tcgen05 kernel): M=512, K=4096,
    N=14336 per format, through cq_gemm_ws (activation operand images built
    once into a workspace), through cq_gemm (the same, workspace from the
    library's pool) and through cq_gemm_noalloc (built in every CTA)."""
    res = {}
    for fmt in fmts:
        wfmt = cq.FMT[fmt]
        W, x = synth.prefill_32(fmt, seed)
        M, K = x.shape
        N = W.shape[0]
        Wd = c.dev(W)
        xq = cq.quantize_act_t(c.dev(x), cq.ACT_FOR[wfmt])
        y = c.torch.empty((M, N), dtype=c.torch.float32, device="cuda")
        need = cq.cq_gemm_workspace_size(wfmt, M, N, K)
        ws = c.torch.empty(need, dtype=c.torch.uint8, device="cuda")
        ms = c.time(lambda: cq.cq_gemm_ws(wfmt, M, N, K, Wd.data_ptr(), xq.data_ptr(), y.data_ptr(), ws.data_ptr(),
                                          need, c.stream()))
        ms_plain = c.time(lambda: cq.cq_gemm(wfmt, M, N, K, Wd.data_ptr(), xq.data_ptr(), y.data_ptr(),
                                             c.stream()))
        ms_na = c.time(lambda: cq.cq_gemm_noalloc(wfmt, M, N, K, Wd.data_ptr(), xq.data_ptr(), y.data_ptr(),
                                                  c.stream()))
        tops = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        res[fmt] = {"shape": f"M={M} N={N} K={K}", "call": "cq_gemm_ws", "ms": ms, "int8_equiv_tops": tops,
                    "frac_of_fp16_peak": tops / peaks["bf16"], "cq_gemm_ms": ms_plain, "cq_gemm_noalloc_ms": ms_na}
        del Wd, xq, y, ws
    return res


def case_moe(c, cq, synth, peaks, seed):
    """Routed-expert FFN: 256 tokens, 32 experts, top-4, Q4_0 2048/1792."""
    Wg, Wu, Wdn, ids, rw, x = synth.moe_ffn(seed)
    T, K = x.shape
    F, E = Wg.shape[1], Wg.shape[0]
    tg, tu, td, ti, tr, tx = (c.dev(a) for a in (Wg, Wu, Wdn, ids, rw, x))
    xq = cq.quantize_act_t(tx, cq.Q8_0)
    need = cq.cq_moe_workspace_size(T, K, F, E, 4)
    ws = c.torch.empty(need, dtype=c.torch.uint8, device="cuda")
    y = c.torch.empty((T, K), dtype=c.torch.float32, device="cuda")
    ms = c.time(lambda: cq.cq_moe_gemv(cq.Q4_0, T, K, F, E, 4, tg.data_ptr(), tu.data_ptr(), td.data_ptr(),
                                       ti.data_ptr(), tr.data_ptr(), xq.data_ptr(), y.data_ptr(), ws.data_ptr(),
                                       need, c.stream()))
    wbytes = Wg.nbytes + Wu.nbytes + Wdn.nbytes
    ops = 2.0 * T * 4 * 3 * F * K
    return {"shape": f"T={T} E={E} top4 K={K} F={F}", "ms": ms, "weight_gbs": wbytes / ms / 1e6,
            "int8_equiv_tops": ops / (ms * 1e-3) / 1e12, "hbm_frac": wbytes / ms / 1e6 / peaks["hbm"]}


def case_lm_head(c, cq, synth, peaks, seed, ms_list=(1, 4, 8, 16)):
    """Batched LM head: Q4_1 128256x4096 at M tokens."""
    W, x = synth.lm_head_q4_1(seed)
    N, K = W.shape[0], x.shape[1]
    Wd, xd = c.dev(W), c.dev(x)
    xq = cq.quantize_act_t(xd, cq.Q8_1)
    # the same head repacked once (cq_repack) and read by cq_gemv_packed
    Wp = cq.repack_t(Wd, cq.Q4_1, K)
    res = {}
    for M in ms_list:
        y = c.torch.empty((M, N), dtype=c.torch.float32, device="cuda")
        ms = c.time(lambda: cq.cq_gemv(cq.Q4_1, M, N, K, Wd.data_ptr(), xq.data_ptr(), y.data_ptr(), c.stream()))
        res[str(M)] = {"ms": ms, "weight_gbs": W.nbytes / ms / 1e6, "hbm_frac": W.nbytes / ms / 1e6 / peaks["hbm"]}
        pms = c.time(lambda: cq.cq_gemv_packed(cq.Q4_1, M, N, K, Wp.data_ptr(), xq.data_ptr(), y.data_ptr(),
                                               c.stream()))
        res[str(M)]["packed"] = {"ms": pms, "weight_gbs": W.nbytes / pms / 1e6}
    if "1" in res:
        for M in res:
            res[M]["t_over_t1"] = res[M]["ms"] / res["1"]["ms"]
            res[M]["packed"]["t_over_t1"] = res[M]["packed"]["ms"] / res["1"]["ms"]
    return res


def case_swiglu(c, cq, synth, peaks, seed, ms_list=(1, 4)):
    """Dense SwiGLU FFN gate + up in one call (cq_gemv_swiglu): Q4_K 14336x4096
    each, M tokens; beside it the same result from two cq_gemv calls and a
    torch silu * mul."""
    torch = c.torch
    Wg, Wu, x = synth.ffn_swiglu_q4_k(seed)
    F, K = Wg.shape[0], x.shape[1]
    tg, tu = c.dev(Wg), c.dev(Wu)
    xq = cq.quantize_act_t(c.dev(x), cq.Q8_K)
    wbytes = Wg.nbytes + Wu.nbytes
    res = {"shape": f"F={F} K={K} (gate + up)", "weight_bytes": wbytes}
    for M in ms_list:
        h = torch.empty((M, F), dtype=torch.float32, device="cuda")
        g = torch.empty((M, F), dtype=torch.float32, device="cuda")
        u = torch.empty((M, F), dtype=torch.float32, device="cuda")
        ms = c.time(lambda: cq.cq_gemv_swiglu(cq.Q4_K, M, F, K, tg.data_ptr(), tu.data_ptr(), xq.data_ptr(),
                                              h.data_ptr(), c.stream()))

        def separate():
            cq.cq_gemv(cq.Q4_K, M, F, K, tg.data_ptr(), xq.data_ptr(), g.data_ptr(), c.stream())
            cq.cq_gemv(cq.Q4_K, M, F, K, tu.data_ptr(), xq.data_ptr(), u.data_ptr(), c.stream())
            torch.mul(torch.nn.functional.silu(g), u, out=h)
        ms_sep = c.time(separate)
        copies = max(1, int(np.ceil(2.5 * L2_BYTES / wbytes)))
        Wg_c = [tg] + [tg.clone() for _ in range(copies - 1)]
        Wu_c = [tu] + [tu.clone() for _ in range(copies - 1)]
        us_b2b, _ = rotated_graph_us(torch, lambda i, s: cq.cq_gemv_swiglu(
            cq.Q4_K, M, F, K, Wg_c[i].data_ptr(), Wu_c[i].data_ptr(), xq.data_ptr(), h.data_ptr(), s), wbytes)
        del Wg_c, Wu_c
        res[str(M)] = {"ms": ms, "weight_gbs": wbytes / ms / 1e6, "hbm_frac": wbytes / ms / 1e6 / peaks["hbm"],
                       "separate_calls_ms": ms_sep,
                       "back_to_back": {"us": us_b2b, "weight_gbs": wbytes / us_b2b / 1e3,
                                        "hbm_frac": wbytes / us_b2b / 1e3 / peaks["hbm"]}}
    return res


def _kquant_gemv(c, cq, peaks, wfmt, W, x, ms_list):
    N, K = W.shape[0], x.shape[1]
    Wd = c.dev(W)
    xq = cq.quantize_act_t(c.dev(x), cq.Q8_K)
    res = {"shape": f"N={N} K={K}"}
    copies = max(1, int(np.ceil(2.5 * L2_BYTES / W.nbytes)))
    Wc = [Wd] + [Wd.clone() for _ in range(copies - 1)]
    for M in ms_list:
        y = c.torch.empty((M, N), dtype=c.torch.float32, device="cuda")
        ms = c.time(lambda: cq.cq_gemv(wfmt, M, N, K, Wd.data_ptr(), xq.data_ptr(), y.data_ptr(), c.stream()))
        us_b2b, _ = rotated_graph_us(c.torch, lambda i, s: cq.cq_gemv(wfmt, M, N, K, Wc[i].data_ptr(), xq.data_ptr(),
                                                                     y.data_ptr(), s), W.nbytes)
        res[str(M)] = {"ms": ms, "weight_gbs": W.nbytes / ms / 1e6, "hbm_frac": W.nbytes / ms / 1e6 / peaks["hbm"],
                       "back_to_back": {"us": us_b2b, "weight_gbs": W.nbytes / us_b2b / 1e3,
                                        "hbm_frac": W.nbytes / us_b2b / 1e3 / peaks["hbm"]}}
    del Wc
    return res


def case_lm_head_q6k(c, cq, synth, peaks, seed, ms_list=(1, 4)):
    """Tied-embedding LM head in Q6_K: 128256x2048 (Llama-3.2-1B) at M tokens."""
    W, x = synth.lm_head_q6_k(seed)
    return _kquant_gemv(c, cq, peaks, cq.Q6_K, W, x, ms_list)


def case_ffn_q5k(c, cq, synth, peaks, seed, ms_list=(1, 4)):
    """Dense FFN gate projection in Q5_K: 14336x4096 at M tokens."""
    W, x = synth.ffn_q5_k(seed)
    return _kquant_gemv(c, cq, peaks, cq.Q5_K, W, x, ms_list)


def case_q4_0_small(c, cq, synth, peaks, seed):
    """Small Q4_0 GEMV 2048x2048 (2.4 MB, fits in L2): the device time of one
    call, and the rate over 256 distinct copies (576 MiB > L2) replayed
    back to back as one CUDA graph."""
    torch = c.torch
    W, x = synth.decode_q4_0_small(seed)
    K = x.shape[1]
    copies = 256
    Wd = c.dev(np.broadcast_to(W, (copies,) + W.shape).copy())
    xq = cq.quantize_act_t(c.dev(x), cq.Q8_0)
    y = torch.empty((1, 2048), dtype=torch.float32, device="cuda")
    one = lambda i=0, sh=None: cq.cq_gemv(cq.Q4_0, 1, 2048, K, Wd[i].data_ptr(), xq.data_ptr(), y.data_ptr(),
                                          sh if sh is not None else c.stream())
    for _ in range(c.warmup):
        one()
    # device time of one call: the stream is held busy while the events and
    # the call are queued, so host launch overhead stays outside the interval
    s = torch.cuda.current_stream()
    lat = []
    for _ in range(5 * c.iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(200000)
        a.record(s)
        one()
        b.record(s)
        b.synchronize()
        lat.append(a.elapsed_time(b))
    def graph_us(call):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream().cuda_stream
            for i in range(copies):
                call(i, cs)
        g.replay()
        torch.cuda.synchronize()
        us = 1e3 * time_calls(torch, g.replay, max(3, c.iters), 2) / copies
        del g
        return us

    us_rot = graph_us(one)
    # The launch floor: the same kernel and launch path with almost no work
    # (8 weight rows), back to back in a graph and as one cold call; and the
    # full call with its weights resident in L2 (no rotation).
    tiny = lambda i=0, sh=None: cq.cq_gemv(cq.Q4_0, 1, 8, K, Wd[i].data_ptr(), xq.data_ptr(), y.data_ptr(),
                                           sh if sh is not None else c.stream())
    us_floor = graph_us(tiny)
    us_l2 = graph_us(lambda i, sh: one(0, sh))
    lat_tiny = []
    for _ in range(5 * c.iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(200000)
        a.record(s)
        tiny()
        b.record(s)
        b.synchronize()
        lat_tiny.append(a.elapsed_time(b))
    return {"device_us_one_call": 1e3 * statistics.median(lat), "rotated_gbs": W.nbytes / us_rot / 1e3,
            "rotated_us_per_call": us_rot,
            "rotation": f"{copies} copies ({copies * W.nbytes / 2**20:.0f} MiB > L2) in one CUDA graph",
            "launch_floor": {"graph_us_per_launch_8_rows": us_floor, "device_us_one_call_8_rows":
                             1e3 * statistics.median(lat_tiny), "graph_us_per_call_l2_resident": us_l2,
                             "note": "same kernel with 8 of 2048 rows: launch, prologue and one pass of the "
                                     "pipeline with no streaming"}}


CASES = {"prefill_gemm_q4_k": case_gemm, "prefill_gemm_32": case_gemm_32, "moe_q4_0": case_moe, "lm_head_q4_1": case_lm_head,
         "decode_q4_0_2048": case_q4_0_small, "ffn_swiglu_q4_k": case_swiglu, "lm_head_q6_k": case_lm_head_q6k,
         "ffn_q5_k": case_ffn_q5k}


def secondary(torch, cq, synth, peaks, seed):
    c = _Ctx(torch)
    out = {}
    for name, fn in CASES.items():
        out[name] = fn(c, cq, synth, peaks, seed)
        torch.cuda.empty_cache()
    return out


def run_case(args):
    """One secondary workload alone, `steps` timed calls after `warmup` (for profiling)."""
    import torch
    from gemm_gguf_block_gb300 import build as gb, cq, synth
    gb.build()
    c = _Ctx(torch, iters=args.steps, warmup=args.warmup)
    assert cq.cq_set_option(cq.OPT_WEIGHTS_CONST, 1) == cq.OK     # as in the decode step
    fn = CASES[args.case]
    kw = {}
    if args.case in ("lm_head_q4_1", "ffn_swiglu_q4_k", "lm_head_q6_k", "ffn_q5_k") and args.m:
        kw["ms_list"] = tuple(int(v) for v in args.m.split(","))
    r = fn(c, cq, synth, _peaks(), args.seed, **kw)
    print(json.dumps({"case": args.case, "steps": args.steps, "warmup": args.warmup, "result": r}))


def run_cq(args, rank, world, local_rank):
    import torch
    from gemm_gguf_block_gb300 import build as gb, cq, synth

    gb.build()
    torch.cuda.set_device(local_rank)
    dist = dist_init(world)
    peaks = _peaks()
    # Decode serving: the weights are constant while the step runs, so the
    # GEMVs may start streaming them before the preceding kernel completes.
    assert cq.cq_set_option(cq.OPT_WEIGHTS_CONST, 1) == cq.OK
    suite = synth.decode_q8_0_suite(args.seed)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    # The five activations (and the five outputs) are views of one buffer each,
    # on the device and in pinned host memory, so a step's inputs go in with
    # one copy and its outputs come back with one.
    k_tot = sum(x.shape[1] for _, x in suite)
    n_tot = sum(W.shape[0] for W, _ in suite)
    x_all = torch.empty(k_tot, dtype=torch.float32, device="cuda")
    y_all = torch.empty(n_tot, dtype=torch.float32, device="cuda")
    xh_all = torch.empty(k_tot, dtype=torch.float32).pin_memory()
    yh_all = torch.empty(n_tot, dtype=torch.float32).pin_memory()
    layers = []
    ko = no = 0
    for W, x in suite:
        N, K = W.shape[0], x.shape[1]
        xh_all[ko:ko + K].copy_(torch.from_numpy(x[0]))
        layers.append(dict(
            N=N, K=K, ko=ko, no=no, W=torch.from_numpy(W).cuda(), x=x_all[ko:ko + K],
            xq=torch.empty(cq.row_bytes(cq.Q8_0, K), dtype=torch.uint8, device="cuda"),
            y=y_all[no:no + N], bytes=W.nbytes + cq.row_bytes(cq.Q8_0, K) + 4 * N))
        ko += K
        no += N
    x_all.copy_(xh_all)
    wbytes = sum(W.nbytes for W, _ in suite)

    def step(sh, stream, ev=None):
        for i, L in enumerate(layers):
            st = cq.cq_quantize_act(cq.Q8_0, 1, L["K"], L["x"].data_ptr(), L["xq"].data_ptr(), sh)
            if ev is not None:
                ev[i][0].record(stream)
            st |= cq.cq_gemv(cq.Q8_0, 1, L["N"], L["K"], L["W"].data_ptr(), L["xq"].data_ptr(),
                             L["y"].data_ptr(), sh)
            if ev is not None:
                ev[i][1].record(stream)
            if st:
                raise RuntimeError(f"cq call failed with status {st}")

    for _ in range(args.warmup):
        step(sh, stream)
    torch.cuda.synchronize()

    # The timed steps replay a CUDA graph of U steps (the same cq_quantize_act /
    # cq_gemv launches, captured once), which removes the per-launch host and
    # launch-queue overhead.
    U = min(args.steps, 10)

    def capture(nsteps, with_events):
        evs = None
        if with_events:
            try:
                evs = [[(torch.cuda.Event(enable_timing=True, external=True),
                         torch.cuda.Event(enable_timing=True, external=True)) for _ in layers]
                       for _ in range(nsteps)]
            except TypeError:
                return None, None
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream()
            for k in range(nsteps):
                step(cs.cuda_stream, cs, evs[k] if evs else None)
        return g, evs

    g_main, _ = capture(U, False)
    g_rest = capture(args.steps % U, False)[0] if args.steps % U else None
    g_main.replay()
    if g_rest:
        g_rest.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(_gpu_query_id(torch, local_rank))
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps // U):
        g_main.replay()
    if g_rest:
        g_rest.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    time.sleep(0.25)
    sampler.stop()
    ms = max_over_ranks(dist, e0.elapsed_time(e1))
    ms_step = ms / args.steps
    value = aggregate_gbs(world, wbytes, ms_step)

    # Per-launch GEMV durations: the same graph, instrumented with timing events
    # around every GEMV launch (recorded inside the graph), replayed right after
    # the timed region for as many steps. The events themselves lengthen the
    # step, which is why the headline value comes from the plain graph.
    g_ev, ev = capture(U, True)
    gemv_ms = [[] for _ in layers]
    if g_ev is not None:
        for _ in range(max(1, args.steps // U)):
            g_ev.replay()
            torch.cuda.synchronize()
            for e in ev:
                for i in range(len(layers)):
                    gemv_ms[i].append(e[i][0].elapsed_time(e[i][1]))
        timing_src = (f"CUDA events recorded inside an instrumented copy of the step graph, "
                      f"{len(gemv_ms[0])} steps replayed after the timed region")
    else:
        gemv_ms = [[float("nan")] for _ in layers]
        timing_src = "unavailable (no graph-recordable events)"
    tot_bytes = sum(L["bytes"] for L in layers) * len(gemv_ms[0])
    tot_ms = sum(sum(v) for v in gemv_ms)
    achieved_instr = tot_bytes / (tot_ms * 1e-3) / 1e9
    alg_bytes_per_launch = sum(L["bytes"] for L in layers) / len(layers)
    instrumented = {f"{L['N']}x{L['K']}": {"us": 1e3 * statistics.mean(gemv_ms[i]),
                                            "gbs": L["bytes"] / (statistics.mean(gemv_ms[i]) * 1e-3) / 1e9}
                    for i, L in enumerate(layers)}
    # The dominant kernel's launch duration as it runs in the step: per shape,
    # back-to-back launches with the step's launch overlap (rotated weights).
    rot = per_shape_rotated(torch, cq, layers)
    rot_us_step = sum(r["us"] for r in rot)
    achieved = sum(L["bytes"] for L in layers) / (rot_us_step * 1e-6) / 1e9
    per_shape = {r["shape"]: {k: r[k] for k in ("us", "gbs", "copies", "launches")} for r in rot}
    lm_us, lm_bytes = rot[-1]["us"], layers[-1]["bytes"]
    clocks = ClockSampler.summary(sampler.window(t_wall0, t_wall1))
    if clocks["samples"] == 0:
        clocks = ClockSampler.summary([r for _, r in sampler.rows])
        clocks["window"] = "whole run (timed region shorter than the sampling interval)"

    # End to end through the public API: every step copies the activations in
    # from pinned host memory, quantises and multiplies each layer, and copies
    # every output back to pinned host memory. Timed twice: replaying a CUDA
    # graph that holds U such steps (copies included), as a serving loop
    # would, and with each call issued from Python (host launch cost included).
    def e2e_step(stream_handle):
        x_all.copy_(xh_all, non_blocking=True)
        for L in layers:
            cq.cq_quantize_act(cq.Q8_0, 1, L["K"], L["x"].data_ptr(), L["xq"].data_ptr(), stream_handle)
            cq.cq_gemv(cq.Q8_0, 1, L["N"], L["K"], L["W"].data_ptr(), L["xq"].data_ptr(), L["y"].data_ptr(),
                       stream_handle)
        yh_all.copy_(y_all, non_blocking=True)

    for _ in range(max(3, args.warmup)):
        e2e_step(sh)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        e2e_step(sh)
    b.record(stream)
    b.synchronize()
    e2e_stream_ms = max_over_ranks(dist, a.elapsed_time(b) / args.steps)

    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e):
        cs = torch.cuda.current_stream()
        for _ in range(U):
            e2e_step(cs.cuda_stream)
    for _ in range(3):
        g_e2e.replay()
    torch.cuda.synchronize()
    reps = max(1, args.steps // U)
    a.record(stream)
    for _ in range(reps):
        g_e2e.replay()
    b.record(stream)
    b.synchronize()
    e2e_seq_ms = max_over_ranks(dist, a.elapsed_time(b) / (reps * U))

    # Pipelined, as a serving loop would run it: two sets of activation and
    # output buffers, the copies on a side stream, so that step i+1's inputs
    # come in and step i's outputs go out while the neighbouring step's kernels
    # run. Every step still copies its own inputs in and its outputs back.
    xb = [x_all, torch.empty_like(x_all)]
    yb = [y_all, torch.empty_like(y_all)]
    xhb = [xh_all, xh_all.clone().pin_memory()]
    yhb = [yh_all, torch.empty_like(yh_all).pin_memory()]

    def kernels(bi, stream_handle):
        for L in layers:
            xv = xb[bi][L["ko"]:L["ko"] + L["K"]]
            yv = yb[bi][L["no"]:L["no"] + L["N"]]
            cq.cq_quantize_act(cq.Q8_0, 1, L["K"], xv.data_ptr(), L["xq"].data_ptr(), stream_handle)
            cq.cq_gemv(cq.Q8_0, 1, L["N"], L["K"], L["W"].data_ptr(), L["xq"].data_ptr(), yv.data_ptr(),
                       stream_handle)

    UP_ = 2 * U
    side = torch.cuda.Stream()
    g_pipe = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_pipe):
        cs = torch.cuda.current_stream()
        side.wait_stream(cs)
        xr = [torch.cuda.Event() for _ in range(UP_)]
        done = [torch.cuda.Event() for _ in range(UP_)]
        yfree = [torch.cuda.Event() for _ in range(UP_)]
        with torch.cuda.stream(side):
            xb[0].copy_(xhb[0], non_blocking=True)
            xr[0].record(side)
        for i in range(UP_):
            bi = i % 2
            cs.wait_event(xr[i])
            if i >= 2:
                cs.wait_event(yfree[i - 2])          # step i-2's outputs have left y[bi]
            kernels(bi, cs.cuda_stream)
            done[i].record(cs)
            with torch.cuda.stream(side):
                if i + 1 < UP_:
                    if i >= 1:
                        side.wait_event(done[i - 1])  # step i-1 has read x[(i+1) % 2]
                    xb[(i + 1) % 2].copy_(xhb[(i + 1) % 2], non_blocking=True)
                    xr[i + 1].record(side)
                side.wait_event(done[i])
                yhb[bi].copy_(yb[bi], non_blocking=True)
                yfree[i].record(side)
        cs.wait_stream(side)
    for _ in range(3):
        g_pipe.replay()
    torch.cuda.synchronize()
    reps_p = max(1, args.steps // UP_)
    a.record(stream)
    for _ in range(reps_p):
        g_pipe.replay()
    b.record(stream)
    b.synchronize()
    e2e_ms = max_over_ranks(dist, a.elapsed_time(b) / (reps_p * UP_))
    same_out = bool(torch.equal(yhb[0], yhb[1]))

    sec = {}
    cpu = None
    if rank == 0:
        if not args.no_secondary:
            del layers
            torch.cuda.empty_cache()
            sec = secondary(torch, cq, synth, peaks, args.seed)
        cpu = cpu_baseline(suite)
    if dist:
        dist.barrier()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "i8xi8->i32, f32 scales", "data": "synthetic",
        "hbm_frac": value / world / peaks["hbm"],
        "config": {"workload": WORKLOAD, "weight_bytes_per_step": wbytes, "weights_const_option": 1,
                   "l2": "inputs larger than L2: 705 MB of weights streamed per step (L2 129 MB)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": "gemv_kernel<Q8_0,1> (the 5 launches of a step, one per shape)",
                     "timing": ("per shape, a CUDA graph of back-to-back cq_gemv launches over rotated weight "
                                "copies (>= 2.5x L2), programmatic dependent launch and the weights-constant "
                                "option as in the step; achieved = the step's GEMV bytes / the sum of the five "
                                "per-launch times"),
                     "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s", "frac": achieved / peaks["hbm"],
                     "algorithmic_bytes_per_launch": alg_bytes_per_launch,
                     "gemv_us_per_step": rot_us_step, "step_us": ms_step * 1e3,
                     "lm_head_launch": {"us": lm_us, "gbs": lm_bytes / (lm_us * 1e-6) / 1e9,
                                        "frac": lm_bytes / (lm_us * 1e-6) / 1e9 / peaks["hbm"]},
                     "instrumented": {"timing": timing_src, "achieved": achieved_instr,
                                      "frac": achieved_instr / peaks["hbm"], "per_shape": instrumented,
                                      "note": "events between launches break the launch overlap: a lower bound"},
                     "peak_src": f"{peaks['src']} hbm_gbs (copy, read+write bytes)",
                     "traffic": _traffic("gemv_q8_0_decode_suite.md")},
        "per_shape": per_shape,
        "cpu_baseline": cpu,
        "e2e": {"value": aggregate_gbs(world, wbytes, e2e_ms), "unit": "GB/s",
                "timing": (f"CUDA graph of {UP_} pipelined steps replayed {reps_p}x: per step one H2D copy of the "
                           f"activations, the quantise + GEMV calls, one D2H copy of the outputs; the copies run on "
                           f"a side stream into double buffers, overlapping the neighbouring steps' kernels"),
                "outputs_equal_across_buffers": same_out,
                "sequential": {"value": aggregate_gbs(world, wbytes, e2e_seq_ms), "unit": "GB/s",
                               "ms_per_step": e2e_seq_ms,
                               "timing": f"CUDA graph of {U} steps, copies and kernels in one stream"},
                "stream_launched": {"value": aggregate_gbs(world, wbytes, e2e_stream_ms), "unit": "GB/s",
                                    "ms_per_step": e2e_stream_ms},
                "h2d_bytes_per_step": 4 * k_tot, "d2h_bytes_per_step": 4 * n_tot,
                "copies_per_step": "one host-to-device (all activations), one device-to-host (all outputs)"},
        "gpu_launches": 2 * len(suite) * args.steps,
        "timed_region": f"{args.steps} steps as replays of a CUDA graph of {U} steps",
        "clocks": clocks,
        "secondary": sec,
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="cq", choices=["cq", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--case", choices=sorted(CASES), help="run one secondary workload alone (for profiling)")
    ap.add_argument("--m", default="", help="with --case lm_head_q4_1, ffn_swiglu_q4_k, lm_head_q6_k or ffn_q5_k: comma-separated token counts")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.case:
        run_case(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_cq(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
