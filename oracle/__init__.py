"""CPU oracle for fine-grained FP8 quantization and the block-scaled GEMM (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import
this package. It shares no code with ``fp8_fine_grained_23_b300``.
"""
