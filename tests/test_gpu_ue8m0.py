"""GPU parity of the power-of-two (UE8M0) scale variant (not on the pages; see
include/fp8bs.h): codes and scales bit-exact against the oracle for both quantizers, and the
unchanged GEMM fed with such scales within |gpu - oracle| <= 1e-5 * sum|a_hat w_hat| + 1 ulp."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.gpu_common import (F, assert_codes_equal, assert_scales_equal,  # noqa: F401
                              assert_within_tolerance)
from tests.helpers import bits_of

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K", [(256, 512), (3, 384), (1000, 7168)])
def test_act_ue8m0_bit_exact(F, M, K):
    x = W.activations(M, K, W.generator(50 + M, "cpu"), "cpu", zero_tile_p=0.02)
    x[0, 0:128] *= 1e-36          # a tile whose exponent clamps at -127
    q, s = F.fp8_quant_act_1x128_ue8m0(x.cuda())
    oq, os_ = O.quant_act_1x128_ue8m0(bits_of(x))
    assert_codes_equal(q, oq)
    assert_scales_equal(s, os_)


@pytest.mark.parametrize("N,K", [(300, 256), (2048, 7168)])
def test_weight_ue8m0_bit_exact(F, N, K):
    w = W.weights(N, K, W.generator(60 + N, "cpu"), "cpu", outlier_p=1e-3, zero_block_p=0.05)
    q, s = F.fp8_quant_weight_128x128_ue8m0(w.cuda())
    oq, os_ = O.quant_weight_128x128_ue8m0(bits_of(w))
    assert_codes_equal(q, oq)
    assert_scales_equal(s, os_)


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_gemm_with_ue8m0_scales(F, out):
    a, w = W.gemm_inputs(W.TINY, "cpu")
    aq, a_s = F.fp8_quant_act_1x128_ue8m0(a.cuda())
    wq, w_s = F.fp8_quant_weight_128x128_ue8m0(w.cuda())
    c = F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out_dtype=out)
    qa, sa = O.quant_act_1x128_ue8m0(bits_of(a))
    qw, sw = O.quant_weight_128x128_ue8m0(bits_of(w))
    c64, cabs = O.gemm_f64(qa, sa, qw, sw)
    name = "f32" if out == torch.float32 else "bf16"
    assert_within_tolerance(c.float().cpu().numpy(), c64, cabs, name, f"ue8m0 tiny {name}")
