"""GPU parity of the E4M3 quantizers: codes and FP32 scales bit-exact to the oracle.

Covers the tiny workload, ragged and strided shapes, adversarial values (zero, negative-zero,
subnormal-only, BF16-max tiles, exact rounding ties, outliers), and the full-size activation and
weight shapes of the dense, MLA and bandwidth-sweep workloads.
"""
import pytest
import torch

from fp8_fine_grained_23_b300 import workloads as W
from tests.gpu_common import (F, assert_codes_equal, assert_scales_equal, oracle_quant_act,  # noqa: F401
                              oracle_quant_weight)
from tests.helpers import bits_of

pytestmark = pytest.mark.gpu


def check_act(F, x: torch.Tensor, ldx_pad: int = 0, ldq_pad: int = 0):
    """x: BF16 [M][K] on any device; optional padding of the leading dimensions."""
    M, K = x.shape
    xg = torch.zeros(M, K + ldx_pad, dtype=torch.bfloat16, device="cuda")
    xg[:, :K] = x.to("cuda")
    qbuf = torch.full((M, K + ldq_pad), 0xAB, dtype=torch.uint8, device="cuda")
    q = qbuf[:, :K]
    s = torch.full((K // 128, M), -7.0, dtype=torch.float32, device="cuda")
    F.fp8_quant_act_1x128(xg[:, :K], q, s)
    torch.cuda.synchronize()
    qo, so = oracle_quant_act(bits_of(x))
    assert_codes_equal(q, qo)
    assert_scales_equal(s, so)
    if ldq_pad:
        assert torch.all(qbuf[:, K:] == 0xAB), "wrote outside the K columns"


def check_weight(F, w: torch.Tensor):
    N, K = w.shape
    wg = w.to("cuda")
    q, s = F.fp8_quant_weight_128x128(wg)
    torch.cuda.synchronize()
    qo, so = oracle_quant_weight(bits_of(w))
    assert_codes_equal(q, qo)
    assert_scales_equal(s, so)


def test_tiny_workload(F):
    a, w = W.gemm_inputs(W.TINY, "cpu")
    check_act(F, a)
    check_weight(F, w)


@pytest.mark.parametrize("M,K", [(1, 128), (3, 256), (5, 384), (129, 640), (257, 1536), (33, 1152),
                                 (2, 1024)])
def test_act_ragged_shapes(F, M, K):
    g = W.generator(100 + M, "cpu")
    check_act(F, W.activations(M, K, g, "cpu", zero_tile_p=0.05))


def test_act_strided(F):
    g = W.generator(7, "cpu")
    check_act(F, W.activations(67, 512, g, "cpu"), ldx_pad=64, ldq_pad=128)


def test_act_special_values(F):
    rows = []
    z = torch.zeros(128)
    rows.append(z.clone())                                     # all zero
    rows.append(torch.full((128,), -0.0))                      # all negative zero
    t = torch.full((128,), 2.0 ** -133)
    t[::3] = -(2.0 ** -130)
    rows.append(t)                                             # BF16 subnormals only
    t = torch.full((128,), 3.3895313892515355e38)              # BF16 max
    t[1::2] *= -0.5
    rows.append(t)
    mids = torch.tensor([448.0, 432.0, -432.0, 1.0625, 1.1875, -1.1875, 3 * 2.0 ** -10,
                         2.0 ** -10, -(2.0 ** -10), 0.0146484375, -0.0, 0.0, 300.0, 464.0 / 2])
    t = torch.zeros(128)
    t[:mids.numel()] = mids                                    # exact ties at scale 1
    rows.append(t)
    t = torch.randn(128)
    t[5] = 1e4                                                 # one outlier
    rows.append(t)
    t = torch.full((128,), 1e-30)
    t[7] = -2.0 ** -64                                         # amax exactly 2^-64
    rows.append(t)
    t = torch.full((128,), 1e-25)
    t[9] = 2.0 ** -64 * 0.99                                   # just below 2^-64 (tiny path)
    rows.append(t)
    x = torch.stack(rows).to(torch.bfloat16)
    x = torch.cat([x, x.flip(0)], dim=1)                       # K = 256, rows reused
    check_act(F, x)


def test_weight_ragged_and_special(F):
    g = W.generator(31, "cpu")
    check_weight(F, W.weights(200, 384, g, "cpu", outlier_p=0.01, zero_block_p=0.2))
    check_weight(F, W.weights(1, 128, g, "cpu"))
    w = W.weights(256, 256, g, "cpu").float()
    w[:128, :128] = 0.0
    w[128:, 128:] = 2.0 ** -131
    w[130, 200] = -(2.0 ** -129)
    check_weight(F, w.to(torch.bfloat16))


def test_full_size_dense_and_mla(F):
    for shape in (W.DENSE,) + W.MLA:
        a, w = W.gemm_inputs(shape, "cuda")
        check_act(F, a.cpu())
        check_weight(F, w.cpu())
        del a, w


@pytest.mark.parametrize("M", W.SWEEP_ACT_M)
def test_full_size_sweep_activations(F, M):
    check_act(F, W.sweep_activations(M, "cuda").cpu())


def test_full_size_sweep_weight(F):
    check_weight(F, W.sweep_weight("cuda").cpu())


def test_stacked_expert_weights(F):
    """[E][N][K] passed as one [E*N][K] matrix gives per-expert [E][N/128][K/128] scales."""
    shape = W.MOE
    w = W.moe_expert_weights(shape, 512, 1024, "gate_up", "cuda", experts=[3, 77, 200])
    q, s = F.fp8_quant_weight_128x128(w.view(-1, 1024))
    torch.cuda.synchronize()
    for i in range(3):
        qo, so = oracle_quant_weight(bits_of(w[i].cpu()))
        assert_codes_equal(q.view(3, 512, 1024)[i], qo)
        assert_scales_equal(s.view(3, 4, 8)[i], so)
