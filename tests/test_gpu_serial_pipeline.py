"""Parity of the serialised-pipeline debug build (libfp8bs_serial.so, `build.py --serial`).

That build runs every pipelined kernel with the shallowest pipeline its structure allows: one
operand stage, one scale slot and one TMEM accumulator in the tiled GEMMs, one operand stage and
one TMEM accumulator in the few-row GEMM. Every role then waits for the previous one at every
step, so a barrier that is missing, waited on with the wrong phase or arrived on too early shows
up as a different result or a timeout. The same small and ragged parity checks as the regular build run here against
the oracle (quantizer codes and scales bit-exact, GEMMs within 1e-5 * sum|a_k w_k| + 1 ulp).
"""
import ctypes

import numpy as np
import pytest
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests import test_gpu_backward as BW
from tests import test_gpu_gemm as GM
from tests import test_gpu_grouped as GR
from tests.gpu_common import F, assert_within_tolerance  # noqa: F401
from tests.helpers import bits_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def FS(F):
    """The binding with its library swapped for the serial build for this module's tests."""
    from fp8_fine_grained_23_b300 import build
    from fp8_fine_grained_23_b300 import fp8bs as mod
    regular = mod.lib
    serial = ctypes.CDLL(build.build(serial=True))
    for name in dir(regular):
        if name.startswith("fp8"):
            fn = getattr(regular, name)
            sf = getattr(serial, name)
            sf.argtypes, sf.restype = fn.argtypes, fn.restype
    for name in ("fp8_quant_act_1x128", "fp8_quant_weight_128x128", "fp8_blockscaled_gemm",
                 "fp8_blockscaled_grouped_gemm", "fp8_blockscaled_gemm_1d1d",
                 "fp8_quant_act_128x1", "fp8bs_last_error"):
        assert getattr(serial, name).restype is not None, name
    mod.lib = serial
    try:
        yield F
    finally:
        mod.lib = regular


def test_serial_build_is_loaded(FS):
    from fp8_fine_grained_23_b300 import fp8bs as mod
    assert mod.lib._name.endswith("libfp8bs_serial.so")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_serial_tiny_workload(FS, out_dtype):
    a, w = W.gemm_inputs(W.TINY, "cpu")
    GM.check_full(FS, a, w, out_dtype)


# few-row kernel: one tile; split K over 2 CTAs; 300 tiles on the persistent grid (two or three
# per CTA); token tile 64; then the tiled kernel
@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (16, 1536, 1024), (16, 38400, 256),
                                   (64, 272, 384), (65, 400, 512), (257, 400, 1024),
                                   (383, 1040, 256)])
def test_serial_ragged_gemm(FS, M, N, K):
    g = W.generator(900 + M + N, "cpu")
    a = W.activations(M, K, g, "cpu")
    w = W.weights(N, K, g, "cpu")
    GM.check_full(FS, a, w, torch.bfloat16)


def test_serial_store_warp_variant(FS):
    """The store-warp variant (BF16 output of a long-K, many-tile launch) in the serial build:
    equal to the FP32 output rounded to BF16, element by element."""
    _, _, c16, c32 = GM.store_warp_case(FS)
    assert torch.equal(c16, c32.to(torch.bfloat16))


@pytest.mark.parametrize("counts,N,K", [([0, 1, 130, 37, 128], 144, 256),
                                        ([128, 256, 0, 1, 127, 129], 512, 384)])
def test_serial_grouped(FS, counts, N, K):
    R = int(sum(counts))
    g = W.generator(700 + R + N, "cpu")
    a = W.activations(R, K, g, "cpu")
    ws = [W.weights(N, K, g, "cpu") for _ in counts]
    off, aq, a_s, wq, w_s, c = GR.run_grouped(FS, a, ws, counts, torch.float32)
    qa, sa = O.quant_act_1x128(bits_of(a))
    qws = [O.quant_weight_128x128(bits_of(w_)) for w_ in ws]
    pr = np.repeat(np.arange(R), N)
    pn = np.tile(np.arange(N), R)
    c64, cabs = O.grouped_gemm_points(qa, sa, np.stack([q for q, _ in qws]),
                                      np.stack([s for _, s in qws]), off, pr, pn)
    assert_within_tolerance(c.cpu().numpy().ravel(), c64, cabs, "f32", "serial grouped")


def test_serial_gemm_1d1d(FS):
    aq, a_s, bq, b_s = BW._operands_1d1d(129, 272, 384, seed=5)
    c = FS.fp8_blockscaled_gemm_1d1d(*(torch.from_numpy(t).cuda() for t in (aq, a_s, bq, b_s)),
                                     out_dtype=torch.float32)
    assert FS.fp8bs_last_error() == FS.FP8BS_OK
    c64, cabs = O.gemm_1d1d_f64(aq, a_s, bq, b_s)
    assert_within_tolerance(c.cpu().numpy(), c64, cabs, "f32", "serial 1d1d")


def test_serial_and_regular_builds_agree(FS, F):
    """Same inputs through both builds: identical GEMM outputs (the accumulation order does not
    depend on the pipeline depth)."""
    from fp8_fine_grained_23_b300 import build
    g = W.generator(42, "cpu")
    a = W.activations(300, 1024, g, "cpu").cuda()
    w = W.weights(528, 1024, g, "cpu").cuda()
    aq, a_s = FS.fp8_quant_act_1x128(a)
    wq, w_s = FS.fp8_quant_weight_128x128(w)
    c_serial = FS.fp8_blockscaled_gemm(aq, a_s, wq, w_s)
    regular = ctypes.CDLL(build.LIB_PATH)
    fn = regular.fp8_blockscaled_gemm
    fn.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 3 + [ctypes.c_void_p, ctypes.c_int64,
                                                                 ctypes.c_int, ctypes.c_void_p]
    c_regular = torch.empty_like(c_serial)
    assert fn(aq.data_ptr(), a_s.data_ptr(), wq.data_ptr(), w_s.data_ptr(), 300, 528, 1024,
              c_regular.data_ptr(), 528, 0, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(c_serial, c_regular)
