"""FP64 CPU oracle for selected-cell attention -- TEST INFRASTRUCTURE ONLY.

Used by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py``; never by the CUDA path.
"""
