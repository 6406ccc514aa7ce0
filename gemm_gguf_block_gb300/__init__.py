"""GGUF block-quantized GEMV / GEMM / routed-expert FFN for GB300 (sm_103a).

The compute lives in ``libcq.so`` (hand-written CUDA behind a C ABI declared in
``include/cq.h``). ``gemm_gguf_block_gb300.cq`` is the thin Python binding with
the same call names; it loads the library on first use and raises if it is
missing. There is no CPU fallback.
"""
