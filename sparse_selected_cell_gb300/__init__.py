"""Selected-cell (QSA union) prompt attention for GB300 (sm_103a).

The compute path lives in ``libqsa.so`` (CUDA kernels behind a C ABI); the
``qsa`` module is a thin ctypes binding over it and ``gen`` draws the seeded
synthetic workloads.  Nothing here falls back to a CPU implementation.
"""
__all__ = ["gen", "qsa"]
