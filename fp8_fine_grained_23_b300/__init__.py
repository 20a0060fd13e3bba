"""fp8bs: fine-grained FP8 (E4M3) quantization and block-scaled FP8 GEMM for B300 (sm_103a).

The compute path is the C-ABI library ``libfp8bs.so`` (declared in ``include/fp8bs.h``); the
Python binding is :mod:`fp8_fine_grained_23_b300.fp8bs`. Seeded synthetic inputs are in
:mod:`fp8_fine_grained_23_b300.workloads`.
"""
