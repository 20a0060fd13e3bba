"""Pins of the oracle's block-scaled GEMM (dense and grouped).

The pages (dtcms.com §三.1/三.3, codingmall.com "Tăng độ chính xác tích lũy") fix the result
C = A W^T on the FP8 operands with their scales applied per 128-wide K block and the sum kept
in high precision. These tests check the oracle against:
  * an exact closed form: E4M3-valued inputs with tile max 448 quantize to themselves (s == 1),
    so C must equal the plain FP64 matrix product of those values (exact at these magnitudes);
  * the single-K-block case K=128, where C = s_a[m] * s_w[n/128] * (A_hat W_hat^T) exactly;
  * the unquantized FP64 product of the BF16 inputs, within the bound the quantization errors
    imply (a transposed operand, a wrong scale index or a dropped block fails it);
  * the FP32-partial variant within its rounding bound, and points == whole matrix;
  * for groups: each expert's rows equal the dense GEMM with that expert's weights.
"""
import numpy as np
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.helpers import bf16_to_f64, bits_of, dequant_act, dequant_weight, e4m3_values


def _quantized(M, N, K, seed, w_outliers=0.0):
    g = W.generator(seed, "cpu")
    a = W.activations(M, K, g, "cpu")
    w = W.weights(N, K, g, "cpu", outlier_p=w_outliers)
    ab, wb = bits_of(a), bits_of(w)
    aq, a_s = O.quant_act_1x128(ab)
    wq, w_s = O.quant_weight_128x128(wb)
    return ab, wb, aq, a_s, wq, w_s


def test_exact_product_when_quantization_is_identity():
    rng = np.random.default_rng(3)
    M, N, K = 48, 160, 512

    def codes(rows):
        c = rng.choice(np.arange(0x28, 0x7F), size=(rows, K)).astype(np.uint8)
        c |= (rng.integers(0, 2, (rows, K)) << 7).astype(np.uint8)
        for kb in range(K // 128):
            c[np.arange(rows), kb * 128 + rng.integers(0, 128, rows)] = 0x7E
        return c

    ca, cw = codes(M), codes(N)
    a = torch.from_numpy(e4m3_values(ca)).to(torch.bfloat16)
    w = torch.from_numpy(e4m3_values(cw)).to(torch.bfloat16)
    aq, a_s = O.quant_act_1x128(bits_of(a))
    wq, w_s = O.quant_weight_128x128(bits_of(w))
    assert np.all(a_s == 1) and np.all(w_s == 1)
    c64, cabs = O.gemm_f64(aq, a_s, wq, w_s)
    exact = e4m3_values(ca) @ e4m3_values(cw).T
    assert np.array_equal(c64, exact)
    assert np.array_equal(cabs, np.abs(e4m3_values(ca)) @ np.abs(e4m3_values(cw)).T)


def test_single_k_block_closed_form():
    _, _, aq, a_s, wq, w_s = _quantized(64, 300, 128, seed=4)
    c64, _ = O.gemm_f64(aq, a_s, wq, w_s)
    block = e4m3_values(aq) @ e4m3_values(wq).T              # exact (51-bit span at K=128)
    sc = a_s[0].astype(np.float64)[:, None] * np.repeat(w_s[:, 0].astype(np.float64), 128)[None, :300]
    assert np.array_equal(c64, sc * block)


def test_within_quantization_bound_of_unquantized_product():
    ab, wb, aq, a_s, wq, w_s = _quantized(40, 272, 640, seed=8, w_outliers=0.003)
    c64, cabs = O.gemm_f64(aq, a_s, wq, w_s)
    x, w = bf16_to_f64(ab), bf16_to_f64(wb)
    cu = O.gemm_unquantized_f64(ab, wb)
    assert np.allclose(cu, x @ w.T, rtol=1e-12, atol=1e-9)    # the unquantized reference itself
    da = np.abs(x - dequant_act(aq, a_s))
    dw = np.abs(w - dequant_weight(wq, w_s))
    bound = da @ np.abs(w).T + np.abs(x) @ dw.T + da @ dw.T
    slack = 1e-12 * (np.abs(x) @ np.abs(w).T) + 1e-12
    assert np.all(np.abs(c64 - cu) <= bound + slack)
    # and the bound is not vacuous: the error is far below the size of the product
    assert np.median(np.abs(c64 - cu) / (np.abs(x) @ np.abs(w).T)) < 0.05


def test_f32_partials_and_points_agree_with_f64():
    _, _, aq, a_s, wq, w_s = _quantized(33, 256, 1024, seed=9)
    c64, cabs = O.gemm_f64(aq, a_s, wq, w_s)
    mm, nn = np.meshgrid(np.arange(33), np.arange(256), indexing="ij")
    p64, pabs, p32 = O.gemm_points(aq, a_s, wq, w_s, mm.ravel(), nn.ravel(), want_f32=True)
    assert np.array_equal(p64, c64.ravel()) and np.array_equal(pabs, cabs.ravel())
    KB = 1024 // 128
    assert np.all(np.abs(p32 - p64) <= (128 + KB + 2) * 2.0 ** -24 * pabs + 1e-30)


def test_grouped_equals_dense_per_group():
    G, N, K = 5, 144, 256
    counts = [0, 1, 130, 37, 128]
    off = W.synthetic_offsets(counts)
    R = int(off[-1])
    g = W.generator(13, "cpu")
    a = W.activations(R, K, g, "cpu")
    ws = [W.weights(N, K, g, "cpu") for _ in range(G)]
    aq, a_s = O.quant_act_1x128(bits_of(a))
    wq_all, ws_all = zip(*[O.quant_weight_128x128(bits_of(w)) for w in ws])
    wq, wsc = np.stack(wq_all), np.stack(ws_all)
    pr = np.repeat(np.arange(R), N)
    pn = np.tile(np.arange(N), R)
    c, cabs = O.grouped_gemm_points(aq, a_s, wq, wsc, off, pr, pn)
    c = c.reshape(R, N)
    for e in range(G):
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            continue
        ce, _ = O.gemm_f64(aq[lo:hi], a_s[:, lo:hi], wq[e], wsc[e])
        assert np.array_equal(c[lo:hi], ce)
    # a row outside every group has no defined value
    c_out, _ = O.grouped_gemm_points(aq, a_s, wq[:2], wsc[:2], W.synthetic_offsets([1, 1]),
                                     np.array([R - 1]), np.array([0]))
    assert np.isnan(c_out[0])
