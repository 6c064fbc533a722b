"""CPU oracle for the VQ KV-cache decode path — TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 restatement of what the method computes, written from the
VecInfer pages (VecInfer: Efficient LLM Inference with Low-Bit KV Cache via
Outlier-Suppressed Vector Quantization).  It is used by ``tests/``, by
``__graft_entry__.smoke()`` and by the ``cpu_baseline`` leg of ``bench.py``
and nowhere else: the library's product path never imports it and has no CPU
fallback.  It shares no code, header, table or constant with the CUDA path.

Pinned functions are listed in ``tests/test_oracle.py``; every function in
``vqkv_oracle`` has at least one pin there (no function is "parity unpinned").
"""
from .vqkv_oracle import *  # noqa: F401,F403
