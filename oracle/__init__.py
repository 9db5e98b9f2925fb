"""CPU oracle for the fine-grained FP8 GEMM path (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never does.
"""
