"""Paged GQA decode attention with per-tile LSE and an FP32 LSE merge, for GB300.

The compute path is the C-ABI library ``libpagedattn.so`` (hand-written sm_103a
CUDA kernels plus the staging runtime); ``binding`` is a thin ctypes layer over
it.  ``workloads`` holds the seeded synthetic inputs.
"""

__all__ = ["binding", "workloads"]
