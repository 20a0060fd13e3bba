"""GPU parity of fp8_blockscaled_gemm_quant: the block-scaled GEMM with its output re-quantized to
E4M3 in 1x128 tiles (the pages accumulate in higher precision, then convert back to FP8 for the
next computation; the tile rule is the activation quantizer's). C is an FP32 accumulation, so
codes are checked against the oracle's FP64 C with R14's bound |C_gpu - C| <= 1e-5 sum|a w| +
1 FP32 ulp propagated through the quantization: the scale, the tile maximum and every value."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.gpu_common import (F, check_requant_tiles, oracle_points,  # noqa: F401
                              oracle_quant_act, oracle_quant_weight)
from tests.helpers import bits_of, gemm_tolerance

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (129, 640, 128), (300, 1152, 1024), (1, 256, 384)])
def test_requantized_output_small(F, M, N, K):
    g = W.generator(M + N + K, "cpu")
    a = W.activations(M, K, g, "cpu")
    w = W.weights(N, K, g, "cpu")
    aq, a_s = F.fp8_quant_act_1x128(a.cuda())
    wq, w_s = F.fp8_quant_weight_128x128(w.cuda())
    cq, cs = F.fp8_blockscaled_gemm_quant(aq, a_s, wq, w_s)
    assert F.fp8bs_last_error() == F.FP8BS_OK
    c64, cabs = O.gemm_f64(*O.quant_act_1x128(bits_of(a)), *O.quant_weight_128x128(bits_of(w)))
    check_requant_tiles(cq.cpu().numpy(), cs.cpu().numpy().T, c64,
                        gemm_tolerance(c64, cabs, "f32"), f"{M}x{N}x{K}")
    # the leading dimension of the codes is honoured and nothing past N is written
    buf = torch.full((M, N + 32), 0xA5, dtype=torch.uint8, device="cuda")
    cq2, _ = F.fp8_blockscaled_gemm_quant(aq, a_s, wq, w_s, c_q=buf[:, :N])
    assert torch.equal(cq2, cq) and torch.all(buf[:, N:] == 0xA5)


def test_requantized_output_full_size_sampled(F):
    """The dense workload 4096x18432x7168 (the launch the host gives the store-warp variant): 48
    whole rows (all 144 output tiles each); the same launch into a wider code buffer writes the
    same codes and nothing past N."""
    shape = W.DENSE
    a, w = W.gemm_inputs(shape, "cuda")
    aq, a_s = F.fp8_quant_act_1x128(a)
    wq, w_s = F.fp8_quant_weight_128x128(w)
    cq, cs = F.fp8_blockscaled_gemm_quant(aq, a_s, wq, w_s)
    assert F.fp8bs_last_error() == F.FP8BS_OK
    qa, sa = oracle_quant_act(bits_of(a))
    qw, sw = oracle_quant_weight(bits_of(w))
    rows = np.unique(np.concatenate([[0, shape.M - 1],
                                     np.random.default_rng(3).choice(shape.M, 46, replace=False)]))
    pm, pn = np.repeat(rows, shape.N), np.tile(np.arange(shape.N), rows.size)
    c64, cabs = oracle_points(qa, sa, qw, sw, pm, pn)
    c64, cabs = c64.reshape(rows.size, shape.N), cabs.reshape(rows.size, shape.N)
    sel = torch.from_numpy(rows).cuda()
    check_requant_tiles(cq[sel].cpu().numpy(), cs[:, sel].cpu().numpy().T, c64,
                        gemm_tolerance(c64, cabs, "f32"), "dense 4096x18432x7168 sampled rows")
    buf = torch.full((shape.M, shape.N + 64), 0xA5, dtype=torch.uint8, device="cuda")
    cq2, cs2 = F.fp8_blockscaled_gemm_quant(aq, a_s, wq, w_s, c_q=buf[:, :shape.N])
    assert F.fp8bs_last_error() == F.FP8BS_OK
    assert torch.equal(cq2, cq) and torch.equal(cs2, cs)
    assert bool(torch.all(buf[:, shape.N:] == 0xA5))
