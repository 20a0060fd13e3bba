"""C-ABI checks that need no GPU: the library loads, exports every function that
include/fp8bs.h declares, and rejects bad arguments on the host before touching a device."""
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8bs.h")


@pytest.fixture(scope="module")
def F():
    from fp8_fine_grained_23_b300 import build
    build.build()
    from fp8_fine_grained_23_b300 import fp8bs
    return fp8bs


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8\w+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("fp8_quant_act_1x128", "fp8_quant_weight_128x128", "fp8_blockscaled_gemm",
              "fp8_blockscaled_grouped_gemm", "fp8bs_status_string", "fp8bs_last_error",
              "fp8_quant_act_128x1", "fp8_quant_weight_128x128_t", "fp8_blockscaled_gemm_1d1d",
              "fp8_blockscaled_grouped_gemm_swiglu_quant", "fp8_moe_permute", "fp8_moe_combine",
              "fp8_blockscaled_gemm_quant"):
        assert n in names


def test_library_exports_every_declared_symbol(F):
    for n in declared_functions():
        assert hasattr(F.lib, n), f"libfp8bs.so does not export {n}"


def test_status_strings(F):
    assert F.fp8bs_status_string(0) == "FP8BS_OK"
    assert F.fp8bs_status_string(-5) == "FP8BS_ERR_TIMEOUT"
    assert F.fp8bs_status_string(123) == "FP8BS_ERR_UNKNOWN"


# Fake, never-dereferenced pointers: argument errors must be caught on the host first.
P16, P4 = 0x1000, 0x2004


@pytest.mark.parametrize("args,expect", [
    ((P16, 4, 100, 128, P16, 128, P4), -1),       # K % 128 != 0
    ((P16, 4, 128, 64, P16, 128, P4), -1),        # ldx < K
    ((P16, -1, 128, 128, P16, 128, P4), -1),      # M < 0
    ((None, 4, 128, 128, P16, 128, P4), -1),      # null input
    ((P16 + 2, 4, 128, 128, P16, 128, P4), -2),   # misaligned input
    ((P16, 4, 128, 132, P16, 128, P4), -2),       # ldx % 8 != 0
    ((P16, 4, 128, 128, P16, 136, P4), -2),       # ldq % 16 != 0
    ((P16, 4, 128, 128, P16, 128, P4 + 1), -2),   # misaligned scales
    ((P16, 0, 128, 128, P16, 128, P4), 0),        # M == 0: no-op, no device touched
])
def test_quant_act_argument_checks(F, args, expect):
    assert F.lib.fp8_quant_act_1x128(*args, None) == expect


@pytest.mark.parametrize("args,expect", [
    ((P16, 256, 100, 128, P16, 128, P4), -1),
    ((P16, 0, 128, 128, P16, 128, P4), 0),
    ((P16, 256, 128, 128, P16 + 8, 128, P4), -2),
])
def test_quant_weight_argument_checks(F, args, expect):
    assert F.lib.fp8_quant_weight_128x128(*args, None) == expect


@pytest.mark.parametrize("mnk,ldc,dt,expect", [
    ((4, 24, 128), 24, 0, -1),       # N % 16 != 0
    ((4, 32, 100), 32, 0, -1),       # K % 128 != 0
    ((4, 32, 128), 16, 0, -1),       # ldc < N
    ((4, 32, 128), 36, 0, -2),       # ldc * 2 % 16 != 0
    ((4, 32, 128), 32, 7, -1),       # unknown output dtype
    ((0, 32, 128), 32, 0, 0),        # M == 0 is a no-op
])
def test_gemm_argument_checks(F, mnk, ldc, dt, expect):
    M, N, K = mnk
    assert F.lib.fp8_blockscaled_gemm(P16, P4, P16, P4, M, N, K, P16, ldc, dt, None) == expect


def test_grouped_gemm_argument_checks(F):
    g = F.lib.fp8_blockscaled_grouped_gemm
    assert g(P16, P4, P16, P4, P4, 0, 8, 32, 128, P16, 32, 0, None) == -1      # G < 1
    assert g(P16, P4, P16, P4, P4, 1025, 8, 32, 128, P16, 32, 0, None) == -1   # G too large
    assert g(P16, P4, P16, P4, None, 2, 8, 32, 128, P16, 32, 0, None) == -1    # no offsets
    assert g(P16, P4, P16, P4, P4 + 1, 2, 8, 32, 128, P16, 32, 0, None) == -2
    assert g(P16, P4, P16, P4, P4, 2, 0, 32, 128, P16, 32, 0, None) == 0       # R == 0


@pytest.mark.parametrize("fn", ["fp8_quant_act_128x1", "fp8_quant_weight_128x128_t"])
@pytest.mark.parametrize("args,expect", [
    ((P16, 200, 128, 128, P16, 208, P4), -1),     # rows % 128 != 0 (the contracted index)
    ((P16, 256, 100, 128, P16, 256, P4), -1),     # K % 128 != 0
    ((P16, 256, 128, 128, P16, 128, P4), -1),     # ldqt < rows
    ((P16, 256, 128, 64, P16, 256, P4), -1),      # ld_in < K
    ((P16, 128 * 65536, 128, 128, P16, 128 * 65536, P4), -1),   # grid limit on row blocks
    ((None, 256, 128, 128, P16, 256, P4), -1),    # null input
    ((P16 + 2, 256, 128, 128, P16, 256, P4), -2), # misaligned input
    ((P16, 256, 128, 128, P16, 264, P4), -2),     # ldqt % 16 != 0
    ((P16, 256, 128, 128, P16, 256, P4 + 1), -2), # misaligned scales
    ((P16, 0, 128, 128, P16, 0, P4), 0),          # no rows: no-op
])
def test_transpose_quant_argument_checks(F, fn, args, expect):
    assert getattr(F.lib, fn)(*args, None) == expect


@pytest.mark.parametrize("mnk,ldc,dt,expect", [
    ((4, 24, 128), 24, 0, -1),
    ((4, 32, 100), 32, 0, -1),
    ((4, 32, 128), 36, 0, -2),
    ((0, 32, 128), 32, 0, 0),
])
def test_gemm_1d1d_argument_checks(F, mnk, ldc, dt, expect):
    M, N, K = mnk
    assert F.lib.fp8_blockscaled_gemm_1d1d(P16, P4, P16, P4, M, N, K, P16, ldc, dt, None) == expect


def test_swiglu_quant_argument_checks(F):
    f = F.lib.fp8_blockscaled_grouped_gemm_swiglu_quant
    ok = (P16, P4, P16, P4, P4, 2, 8, 512, 128, P16, 256, P4)
    assert f(*ok[:6], 0, *ok[7:], None) == 0                                      # R == 0
    assert f(*ok[:5], 0, *ok[6:], None) == -1                                     # G < 1
    assert f(*ok[:7], 384, *ok[8:], None) == -1                                   # N2 % 256
    assert f(*ok[:10], 128, ok[11], None) == -1                                   # ldh < N2/2
    assert f(*ok[:10], 264, ok[11], None) == -2                                   # ldh % 16
    assert f(*ok[:9], P16 + 4, *ok[10:], None) == -2                              # h_q alignment
    assert f(*ok[:11], P4 + 1, None) == -2                                        # h_s alignment
    assert f(*ok[:11], None, None) == -1                                          # no h_s


def test_moe_dispatch_argument_checks(F):
    pm = F.lib.fp8_moe_permute
    assert pm(P16, 256, P4, 8, P4, 0, 256, P16, 256, P4, None) == 0               # R == 0
    assert pm(P16, 256, P4, 8, P4, 4, 200, P16, 256, P4, None) == -1              # K % 128
    assert pm(P16, 128, P4, 8, P4, 4, 256, P16, 256, P4, None) == -1              # ldq < K
    assert pm(P16, 264, P4, 8, P4, 4, 256, P16, 256, P4, None) == -2              # ldq % 16
    assert pm(P16 + 8, 256, P4, 8, P4, 4, 256, P16, 256, P4, None) == -2          # q alignment
    cm = F.lib.fp8_moe_combine
    assert cm(P16, 64, 8, P4, P4, 0, 8, 64, P16, 64, None) == 0                   # T == 0
    assert cm(P16, 64, 8, P4, P4, 4, 0, 64, P16, 64, None) == -1                  # topk < 1
    assert cm(P16, 64, 8, P4, P4, 4, 33, 64, P16, 64, None) == -1                 # topk > 32
    assert cm(P16, 64, 8, P4, P4, 4, 8, 60, P16, 64, None) == -1                  # N % 8
    assert cm(P16, 68, 8, P4, P4, 4, 8, 64, P16, 64, None) == -2                  # ldy % 8
    assert cm(P16 + 4, 64, 8, P4, P4, 4, 8, 64, P16, 64, None) == -2              # y alignment


def test_gemm_quant_argument_checks(F):
    g = F.lib.fp8_blockscaled_gemm_quant
    assert g(P16, P4, P16, P4, 0, 256, 128, P16, 256, P4, None) == 0      # M == 0
    assert g(P16, P4, P16, P4, 4, 192, 128, P16, 256, P4, None) == -1     # N % 128
    assert g(P16, P4, P16, P4, 4, 256, 128, P16, 128, P4, None) == -1     # ldcq < N
    assert g(P16, P4, P16, P4, 4, 256, 128, P16, 264, P4, None) == -2     # ldcq % 16
    assert g(P16, P4, P16, P4, 4, 256, 128, P16 + 1, 256, P4, None) == -2 # c_q alignment
    assert g(P16, P4, P16, P4, 4, 256, 128, P16, 256, None, None) == -1   # no c_s


def test_debug_hook_rejects_negative_index(F):
    assert F.lib.fp8bs_debug_skip_release(-1) == F.FP8BS_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_valid_call_without_gpu_fails_loudly(F):
    st = F.lib.fp8_quant_act_1x128(P16, 4, 128, 128, P16, 128, P4, None)
    assert st in (F.FP8BS_ERR_CUDA, F.FP8BS_ERR_UNSUPPORTED_DEVICE)
    with pytest.raises(F.Fp8bsError):
        F._check("fp8_quant_act_1x128", st)
