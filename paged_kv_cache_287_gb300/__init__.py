"""Attention over a paged KV cache on GB300 (sm_103a).

The compute lives in ``libpagedattn.so`` (CUDA kernels behind a C ABI,
declared in ``include/pa.h``); ``binding`` marshals PyTorch tensors into
those calls.  ``workloads`` draws seeded synthetic inputs.
"""

__all__ = ["binding", "workloads"]
