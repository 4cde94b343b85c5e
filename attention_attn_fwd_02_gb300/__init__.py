"""Fused softmax attention forward for one GB300 (sm_103a).

The compute lives in ``libattn.so`` (hand-written CUDA, built from ``csrc/``);
``attn`` is a thin ctypes binding to its C ABI (``include/attn.h``).  The
binding loads the library on first use and raises if it is missing: there is
no CPU fallback.  ``workloads`` draws seeded synthetic inputs.
"""
