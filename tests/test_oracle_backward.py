"""Pins of the oracle's backward-pass functions.

The pages use the same E4M3 format in the backward pass as in the forward pass
(codingmall.com "Định dạng E4M3 hợp nhất"; dtcms.com §三.2). A block-scaled contraction needs
one scale per 128-long block of the contracted index, so the data-gradient GEMM dX = dY W
(contracting over N) takes dY in 1x128 tiles and W as W^T in its 128x128 blocks, and the
weight-gradient GEMM dW = dY^T X (contracting over the tokens) takes dY and X in 128x1 tiles
with a per-row scale on both operands. These tests pin the new oracle functions to:
  * the already pinned forward quantizers: a 128x1 tile of x is a 1x128 tile of x^T, and the
    transposed weight codes are the forward codes transposed;
  * the quantizer invariants, checked directly (tile max 448, zero tiles, round-trip bound);
  * an exact closed form for the per-row-scaled GEMM (E4M3-valued operands with tile max 448
    give s == 1 and the plain FP64 matrix product), and its K=128 single-block form;
  * the unquantized FP64 products dY^T X and dY W within the bound the quantization errors
    imply (a wrong scale index, a transposed operand or a dropped block fails it).
"""
import numpy as np
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.helpers import bf16_to_f64, bits_of, dequant_act, e4m3_half_ulp, e4m3_values


def _tensor(rows, cols, seed, std=1.0):
    g = W.generator(seed, "cpu")
    if std == 1.0:
        return W.activations(rows, cols, g, "cpu")
    return W.weights(rows, cols, g, "cpu")


def _dequant_128x1(qt, s):
    """x_hat[m, k] from transposed codes qt [K][M] and scales s [M/128][K]."""
    v = e4m3_values(qt).T                                   # [M][K]
    return v * np.repeat(s.astype(np.float64), 128, axis=0)


def test_128x1_is_1x128_of_the_transpose():
    x = _tensor(384, 256, seed=21)
    x[128:256, 7] = 0                                       # one all-zero 128x1 tile
    qt, s = O.quant_act_128x1(bits_of(x))
    q2, s2 = O.quant_act_1x128(bits_of(x.T.contiguous()))
    assert qt.shape == (256, 384) and s.shape == (3, 256)
    assert np.array_equal(qt, q2) and np.array_equal(s, s2)


def test_128x1_invariants():
    x = _tensor(256, 200, seed=22)
    x[0:128, 3] = 0
    x[128:256, 150] *= 1e-30                                # a tiny-amax tile (BF16 keeps it)
    xb = bits_of(x)
    qt, s = O.quant_act_128x1(xb)
    x64 = bf16_to_f64(xb)
    for mb in range(2):
        tile = x64[mb * 128:(mb + 1) * 128]                 # [128][K]
        amax = np.abs(tile).max(axis=0)
        vals = np.abs(e4m3_values(qt[:, mb * 128:(mb + 1) * 128]))   # [K][128]
        nz = amax > 0
        assert np.array_equal(s[mb][nz], (amax[nz].astype(np.float32) / np.float32(448)))
        assert np.all(vals[nz].max(axis=1) == 448)
        assert np.all(s[mb][~nz] == 1) and np.all(qt[~nz, mb * 128:(mb + 1) * 128] == 0)
    assert not np.all(s[0] == 1) and (~(np.abs(x64[:128]).max(axis=0) > 0)).sum() == 1
    # round trip within half an E4M3 step of x * (448 / amax), scaled back
    xh = _dequant_128x1(qt, s)
    r = (np.float32(448) / np.repeat(s * np.float32(448), 128, axis=0)).astype(np.float64)
    bound = e4m3_half_ulp(x64 * r) * np.repeat(s.astype(np.float64), 128, axis=0)
    assert np.all(np.abs(x64 - xh) <= bound * (1 + 2.0 ** -20) + 1e-300)


def test_weight_t_is_forward_transposed():
    w = _tensor(384, 256, seed=23, std=0.02)
    w[128:256, 0:128] = 0                                   # one zero block
    qt, st = O.quant_weight_128x128_t(bits_of(w))
    q, s = O.quant_weight_128x128(bits_of(w))
    assert qt.shape == (256, 384) and st.shape == (2, 3)
    assert np.array_equal(qt, q.T) and np.array_equal(st, s.T)
    assert st[0, 1] == 1 and np.all(qt[0:128, 128:256] == 0)


def _e4m3_rows(rng, rows, K):
    """Codes whose every (row, 128-block) holds a +-448, so the tile scale is exactly 1."""
    c = rng.choice(np.arange(0x28, 0x7F), size=(rows, K)).astype(np.uint8)
    c |= (rng.integers(0, 2, (rows, K)) << 7).astype(np.uint8)
    for kb in range(K // 128):
        c[np.arange(rows), kb * 128 + rng.integers(0, 128, rows)] = 0x7E
    return c


def test_1d1d_exact_when_scales_are_one():
    rng = np.random.default_rng(24)
    M, N, K = 40, 72, 512
    ca, cb = _e4m3_rows(rng, M, K), _e4m3_rows(rng, N, K)
    # quantize through the 128x1 path: rows of the operand are channels, K the tokens
    a = torch.from_numpy(e4m3_values(ca).T.copy()).to(torch.bfloat16)   # [K][M]
    b = torch.from_numpy(e4m3_values(cb).T.copy()).to(torch.bfloat16)   # [K][N]
    aq, a_s = O.quant_act_128x1(bits_of(a))
    bq, b_s = O.quant_act_128x1(bits_of(b))
    assert np.all(a_s == 1) and np.all(b_s == 1)
    assert np.array_equal(aq, ca) and np.array_equal(bq, cb)
    c64, cabs = O.gemm_1d1d_f64(aq, a_s, bq, b_s)
    va, vb = e4m3_values(ca), e4m3_values(cb)
    assert np.array_equal(c64, va @ vb.T)                   # exact: < 53-bit span at K=512
    assert np.array_equal(cabs, np.abs(va) @ np.abs(vb).T)


def test_1d1d_single_block_closed_form():
    """K = 128: C[m][n] = s_a[m] * s_b[n] * (A_hat B_hat^T)[m][n], one rounding."""
    a = _tensor(128, 48, seed=25)        # tokens x channels
    b = _tensor(128, 80, seed=26)
    aq, a_s = O.quant_act_128x1(bits_of(a))
    bq, b_s = O.quant_act_128x1(bits_of(b))
    c64, _ = O.gemm_1d1d_f64(aq, a_s, bq, b_s)
    block = e4m3_values(aq) @ e4m3_values(bq).T
    sc = a_s[0].astype(np.float64)[:, None] * b_s[0].astype(np.float64)[None, :]
    assert np.array_equal(c64, sc * block)


def test_wgrad_within_quantization_bound():
    """dW = dY^T X from 128x1-quantized dY and X, against the unquantized FP64 product."""
    dy = _tensor(384, 96, seed=27)       # [tokens][N]
    x = _tensor(384, 160, seed=28)       # [tokens][K]
    dyb, xb = bits_of(dy), bits_of(x)
    aq, a_s = O.quant_act_128x1(dyb)     # [N][tokens]
    bq, b_s = O.quant_act_128x1(xb)      # [K][tokens]
    c64, cabs = O.gemm_1d1d_f64(aq, a_s, bq, b_s)
    dy64, x64 = bf16_to_f64(dyb), bf16_to_f64(xb)
    exact = dy64.T @ x64
    d_dy = np.abs(dy64 - _dequant_128x1(aq, a_s))
    d_x = np.abs(x64 - _dequant_128x1(bq, b_s))
    bound = d_dy.T @ np.abs(x64) + np.abs(dy64).T @ d_x + d_dy.T @ d_x
    slack = 1e-12 * (np.abs(dy64).T @ np.abs(x64)) + 1e-12
    assert np.all(np.abs(c64 - exact) <= bound + slack)
    assert np.median(np.abs(c64 - exact) / (np.abs(dy64).T @ np.abs(x64))) < 0.05
    # with the operands' scales swapped between rows the bound fails (the pin has teeth)
    c_bad, _ = O.gemm_1d1d_f64(aq, a_s[:, ::-1].copy(), bq, b_s)
    assert not np.all(np.abs(c_bad - exact) <= bound + slack)
    # FP32-partial variant within its rounding bound
    mm, nn = np.meshgrid(np.arange(96), np.arange(160), indexing="ij")
    p64, pabs, p32 = O.gemm_1d1d_points(aq, a_s, bq, b_s, mm.ravel(), nn.ravel(), want_f32=True)
    assert np.array_equal(p64, c64.ravel())
    assert np.all(np.abs(p32 - p64) <= (128 + 3 + 2) * 2.0 ** -24 * pabs + 1e-30)


def test_dgrad_within_quantization_bound():
    """dX = dY W with dY in 1x128 tiles and W^T codes in 128x128 blocks, through the dense
    block-scaled GEMM oracle, against the unquantized FP64 product."""
    dy = _tensor(64, 384, seed=29)       # [tokens][N]
    w = _tensor(384, 256, seed=30, std=0.02)   # [N][K]
    dyb, wb = bits_of(dy), bits_of(w)
    aq, a_s = O.quant_act_1x128(dyb)
    wqt, wst = O.quant_weight_128x128_t(wb)    # [K][N], [K/128][N/128]
    c64, _ = O.gemm_f64(aq, a_s, wqt, wst)
    dy64, w64 = bf16_to_f64(dyb), bf16_to_f64(wb)
    exact = dy64 @ w64
    d_dy = np.abs(dy64 - dequant_act(aq, a_s))
    wt_hat = e4m3_values(wqt) * np.repeat(np.repeat(wst.astype(np.float64), 128, 0), 128, 1)
    d_w = np.abs(w64 - wt_hat.T)
    bound = d_dy @ np.abs(w64) + np.abs(dy64) @ d_w + d_dy @ d_w
    slack = 1e-12 * (np.abs(dy64) @ np.abs(w64)) + 1e-12
    assert np.all(np.abs(c64 - exact) <= bound + slack)
