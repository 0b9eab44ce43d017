"""Paged GQA decode attention with per-tile LSE and an FP32 LSE merge, for GB300.

The compute path is the C-ABI library ``libpagedattn.so`` (hand-written sm_103a
CUDA kernels plus the native staging runtime, admission planner and page
converter); ``binding`` is a thin ctypes layer over it, ``decode`` sequences
its calls into decode steps (resident, staged, per-tile staged and planned
routes), ``busmodel`` is the staged route's latency model and ``workloads``
holds the seeded synthetic inputs.  ``build`` compiles the library in place.
"""

__all__ = ["binding", "busmodel", "decode", "workloads"]
