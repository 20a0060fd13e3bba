"""GPU parity of the backward-pass path against the oracle.

The pages use E4M3 for the backward pass as well (codingmall.com "Định dạng E4M3 hợp nhất";
dtcms.com §三.2). Reading: the data-gradient GEMM dX = dY W takes dY in 1x128 tiles and W^T
codes in 128x128 blocks; the weight-gradient GEMM dW = dY^T X takes dY and X in 128x1 tiles
with a per-row scale on both operands. Codes and scales must match the oracle bit for bit;
GEMM elements must lie within |gpu - oracle| <= 1e-5 * sum_k |a_hat_k b_hat_k| + 1 ulp of the
output type. Small cases compare everything; the full-size backward of the dense projection
(M=4096 tokens, N=18432, K=7168) compares every code and scale and sampled GEMM elements.
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.gpu_common import (F, assert_codes_equal, assert_scales_equal,  # noqa: F401
                              assert_within_tolerance, oracle_points, oracle_points_1d1d,
                              oracle_quant_act, oracle_quant_act_128x1, oracle_quant_weight_t)
from tests.helpers import bits_of

pytestmark = pytest.mark.gpu


def _special_columns(x: torch.Tensor) -> torch.Tensor:
    """An all-zero 128x1 tile, a tiny-amax one and a lone outlier, on a CPU BF16 tensor."""
    x = x.clone()
    x[0:128, 1] = 0
    x[0:128, 2] *= 1e-30
    x[5, 3] = 3.0e4
    return x


@pytest.mark.parametrize("M,K", [(128, 128), (256, 384), (384, 1024), (1024, 7168)])
def test_quant_act_128x1(F, M, K):
    x = _special_columns(W.activations(M, K, W.generator(40 + M, "cpu"), "cpu"))
    qt, s = F.fp8_quant_act_128x1(x.cuda())
    assert F.fp8bs_last_error() == F.FP8BS_OK
    oq, os_ = O.quant_act_128x1(bits_of(x))
    assert_codes_equal(qt, oq)
    assert_scales_equal(s, os_)


def test_quant_act_128x1_leading_dimensions(F):
    """ldx > K reads only K columns; ldqt > M leaves the padding bytes of qt untouched."""
    M, K = 256, 256
    big = W.activations(M, K + 64, W.generator(50, "cpu"), "cpu")
    x = big[:, :K]
    qt_buf = torch.full((K, M + 32), 0xA5, dtype=torch.uint8, device="cuda")
    s = torch.empty(M // 128, K, dtype=torch.float32, device="cuda")
    F.fp8_quant_act_128x1(big.cuda()[:, :K], qt=qt_buf[:, :M], scales=s)
    oq, os_ = O.quant_act_128x1(bits_of(x))
    assert_codes_equal(qt_buf[:, :M], oq)
    assert_scales_equal(s, os_)
    assert torch.all(qt_buf[:, M:] == 0xA5)
    # M == 0 is a no-op
    F.fp8_quant_act_128x1(torch.empty(0, K, dtype=torch.bfloat16, device="cuda"))


@pytest.mark.parametrize("N,K", [(128, 128), (384, 256), (1024, 7168)])
def test_quant_weight_t(F, N, K):
    w = W.weights(N, K, W.generator(60 + N, "cpu"), "cpu", outlier_p=1e-3, zero_block_p=0.05)
    w[0:128, 0:128] = 0
    qt, st = F.fp8_quant_weight_128x128_t(w.cuda())
    assert F.fp8bs_last_error() == F.FP8BS_OK
    oq, os_ = O.quant_weight_128x128_t(bits_of(w))
    assert_codes_equal(qt, oq)
    assert_scales_equal(st, os_)
    # the same blocks as the forward quantizer, transposed
    q, s = F.fp8_quant_weight_128x128(w.cuda())
    assert torch.equal(qt, q.t()) and torch.equal(st, s.t())


def _operands_1d1d(M, N, K, seed):
    """Oracle-quantized 1d1d operands of ragged size: rows of 128x1-quantized tensors, cut."""
    mpad, npad = -(-M // 128) * 128, -(-N // 128) * 128
    g = W.generator(seed, "cpu")
    a = W.activations(K, mpad, g, "cpu")          # [tokens][channels]
    b = W.activations(K, npad, g, "cpu", sigma=2.0 ** -8)
    aq, a_s = O.quant_act_128x1(bits_of(a))       # [mpad][K], [K/128][mpad]
    bq, b_s = O.quant_act_128x1(bits_of(b))
    return (np.ascontiguousarray(aq[:M]), np.ascontiguousarray(a_s[:, :M]),
            np.ascontiguousarray(bq[:N]), np.ascontiguousarray(b_s[:, :N]))


@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (129, 272, 384), (200, 400, 512),
                                   (256, 256, 1024), (383, 1040, 256)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_gemm_1d1d_ragged(F, M, N, K, out):
    aq, a_s, bq, b_s = _operands_1d1d(M, N, K, seed=M * 7 + N)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    c = F.fp8_blockscaled_gemm_1d1d(torch.from_numpy(aq).cuda(), torch.from_numpy(a_s).cuda(),
                                    torch.from_numpy(bq).cuda(), torch.from_numpy(b_s).cuda(),
                                    out_dtype=dt)
    assert F.fp8bs_last_error() == F.FP8BS_OK
    c64, cabs = O.gemm_1d1d_f64(aq, a_s, bq, b_s)
    assert_within_tolerance(c.float().cpu().numpy(), c64, cabs, out, f"1d1d {M}x{N}x{K} {out}")


def test_gemm_1d1d_row_scales_matter(F):
    """Scaling one B row's scales by 2 doubles exactly that output column (power of two)."""
    aq, a_s, bq, b_s = _operands_1d1d(128, 256, 512, seed=77)
    b2 = b_s.copy()
    b2[:, 37] *= 2
    args = [torch.from_numpy(t).cuda() for t in (aq, a_s, bq)]
    c1 = F.fp8_blockscaled_gemm_1d1d(*args, torch.from_numpy(b_s).cuda(), out_dtype=torch.float32)
    c2 = F.fp8_blockscaled_gemm_1d1d(*args, torch.from_numpy(b2).cuda(), out_dtype=torch.float32)
    others = [i for i in range(256) if i != 37]
    assert torch.equal(c2[:, 37], 2 * c1[:, 37])
    assert torch.equal(c2[:, others], c1[:, others])


def _sample(n, count, rng):
    idx = np.unique(np.concatenate([[0, n - 1], rng.choice(n, count, replace=False)]))
    return idx.astype(np.int64)


def test_full_size_backward(F):
    """Backward of the dense projection (M=4096, N=18432, K=7168) as a training step runs it:
    dY and X in 128x1 tiles, dY in 1x128 tiles, W^T codes; bit-exact codes and scales, and
    sampled elements of dW (FP32) and dX (BF16) against the oracle on its own quantization."""
    shape = W.DENSE
    x, w, dy = W.backward_inputs(shape, "cuda")
    # GPU path
    dyt_q, dyt_s = F.fp8_quant_act_128x1(dy)           # [N][M], [M/128][N]
    xt_q, xt_s = F.fp8_quant_act_128x1(x)              # [K][M], [M/128][K]
    dy_q, dy_s = F.fp8_quant_act_1x128(dy)             # [M][N], [N/128][M]
    wt_q, wt_s = F.fp8_quant_weight_128x128_t(w)       # [K][N], [K/128][N/128]
    dw = F.fp8_blockscaled_gemm_1d1d(dyt_q, dyt_s, xt_q, xt_s, out_dtype=torch.float32)
    dx = F.fp8_blockscaled_gemm(dy_q, dy_s, wt_q, wt_s, out_dtype=torch.bfloat16)
    assert F.fp8bs_last_error() == F.FP8BS_OK
    dw_g, dx_g = dw.cpu().numpy(), dx.float().cpu().numpy()
    del dw, dx
    # oracle on the same BF16 inputs
    xb, wb, dyb = bits_of(x), bits_of(w), bits_of(dy)
    o_dyt = oracle_quant_act_128x1(dyb)
    assert_codes_equal(dyt_q, o_dyt[0])
    assert_scales_equal(dyt_s, o_dyt[1])
    o_xt = oracle_quant_act_128x1(xb)
    assert_codes_equal(xt_q, o_xt[0])
    assert_scales_equal(xt_s, o_xt[1])
    o_dy = oracle_quant_act(dyb)
    assert_codes_equal(dy_q, o_dy[0])
    assert_scales_equal(dy_s, o_dy[1])
    o_wt = oracle_quant_weight_t(wb)
    assert_codes_equal(wt_q, o_wt[0])
    assert_scales_equal(wt_s, o_wt[1])
    rng = np.random.default_rng(5)
    # dW [N][K]: sampled rows x columns
    rows, cols = _sample(shape.N, 120, rng), _sample(shape.K, 120, rng)
    pm, pn = np.repeat(rows, cols.size), np.tile(cols, rows.size)
    c64, cabs = oracle_points_1d1d(o_dyt[0], o_dyt[1], o_xt[0], o_xt[1], pm, pn)
    assert_within_tolerance(dw_g[pm, pn], c64, cabs, "f32", "dW sampled")
    # dX [M][K]: sampled rows x columns (contraction over N = 18432)
    rows, cols = _sample(shape.M, 120, rng), _sample(shape.K, 120, rng)
    pm, pn = np.repeat(rows, cols.size), np.tile(cols, rows.size)
    c64, cabs = oracle_points(o_dy[0], o_dy[1], o_wt[0], o_wt[1], pm, pn)
    assert_within_tolerance(dx_g[pm, pn], c64, cabs, "bf16", "dX sampled")
