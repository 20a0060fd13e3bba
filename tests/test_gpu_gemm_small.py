"""GPU parity of the few-row path of fp8_blockscaled_gemm (M <= 64: C^T = W A^T on the tensor
cores, with the K loop split over a cluster of up to 8 CTAs when the weight tiles are few)
against the oracle, within |gpu - oracle| <= 1e-5 * sum|a_hat w_hat| + 1 ulp of the output type.
The shapes pick every split factor (1, 2, 4, 8), token tiles of 32 and 64, ragged N and K, the
decode-size versions of the dense and MLA projections, unsplit problems with more weight tiles
than SMs (the persistent grid takes two or three tiles per CTA), and sizes on both sides of the
switch to the tiled CTA-pair kernel (M = 64 / 65, 100, 128)."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.gpu_common import (F, assert_within_tolerance, oracle_points,  # noqa: F401
                              oracle_quant_act, oracle_quant_weight)
from tests.helpers import bits_of

pytestmark = pytest.mark.gpu


def run(F, M, N, K, out_dtype, seed):
    g = W.generator(seed, "cuda")
    a = W.activations(M, K, g, "cuda")
    w = W.weights(N, K, g, "cuda")
    aq, a_s = F.fp8_quant_act_1x128(a)
    wq, w_s = F.fp8_quant_weight_128x128(w)
    c = F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out_dtype=out_dtype)
    assert F.fp8bs_last_error() == F.FP8BS_OK
    c2 = F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out_dtype=out_dtype)
    assert torch.equal(c, c2), "repeated calls must give identical results"
    qa, sa = oracle_quant_act(bits_of(a))
    qw, sw = oracle_quant_weight(bits_of(w))
    mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    c64, cabs = oracle_points(qa, sa, qw, sw, mm.ravel(), nn.ravel())
    name = "f32" if out_dtype == torch.float32 else "bf16"
    assert_within_tolerance(c.float().cpu().numpy().ravel(), c64, cabs, name, f"{M}x{N}x{K} {name}")


@pytest.mark.parametrize("M,N,K", [
    (1, 1536, 7168),      # 12 weight tiles: split 8
    (16, 7168, 2048),     # 56 tiles: split 2
    (33, 640, 1536),      # 5 tiles, 12 K blocks: split 4, token tile 64
    (64, 18432, 7168),    # 144 tiles: no split
    (65, 384, 256),       # first size on the tiled kernel
    (100, 1040, 384),     # ragged N, 3 K blocks, token tile 128
    (128, 256, 128),      # one K block
    (7, 24576, 1536),     # MLA q-up at decode size: 192 tiles, up to two per CTA
    (17, 38400, 384),     # 300 tiles: up to three per CTA, token tile 32
    (40, 40960, 256),     # 320 tiles: up to three per CTA, token tile 64, ragged M
])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_few_rows(F, M, N, K, out):
    run(F, M, N, K, out, seed=M + N + K)


def test_boundary_129_rows_uses_the_tiled_kernel(F):
    run(F, 129, 512, 256, torch.float32, seed=5)
