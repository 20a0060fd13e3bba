"""Pins of the oracle's 1x128 activation and 128x128 weight quantizers.

What the pages fix (codingmall.com "Định lượng hạt mịn", "Định lượng trực tuyến";
risenshineclean.com §三): activations are scaled per 1x128 tile (one token, 128 channels),
weights per 128x128 block, each from its own current maximum. What the mathematics then fixes,
and what these tests check without re-running the oracle's formula:
  * every non-zero tile reaches the top code: max |value(code)| == 448;
  * an all-zero tile gets scale 1 and zero codes (this project's reading);
  * the scale is amax / 448 in FP32, with amax found here by NumPy;
  * the round trip x -> code -> value * s is within half an E4M3 step (plus the FP32
    roundings of s and of x * r);
  * an outlier changes only its own tile (the point of fine-grained scaling);
  * inputs that already are E4M3 values with tile max 448 come back unchanged (s == 1);
  * scaling a tile by 2^k leaves its codes unchanged, down to BF16's smallest normals (this
    exercises the tiny-amax path).
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.helpers import (bf16_to_f64, bits_of, dequant_act, dequant_weight, e4m3_half_ulp,
                           e4m3_values)


def _tiny_a():
    a, _ = W.gemm_inputs(W.TINY, "cpu")
    return bits_of(a)


def _act_tiles(x64):
    M, K = x64.shape
    return x64.reshape(M, K // 128, 128)


def test_act_invariants_tiny_config():
    xb = _tiny_a()
    q, s = O.quant_act_1x128(xb)
    x = bf16_to_f64(xb)
    tiles = _act_tiles(x)
    amax = np.abs(tiles).max(axis=2)                     # [M][KB]
    vals = e4m3_values(q).reshape(tiles.shape)
    nz = amax > 0
    assert np.all(np.abs(vals).max(axis=2)[nz] == 448.0)
    m, kb = W.TINY_ZERO_TILE
    assert not nz[m, kb] and nz.sum() == nz.size - 1
    assert s[kb, m] == 1.0 and np.all(q[m, kb * 128:(kb + 1) * 128] == 0)
    expect_s = (amax.astype(np.float32) / np.float32(448.0)).T
    assert np.array_equal(s[nz.T], expect_s[nz.T])


def test_act_round_trip_bound():
    xb = _tiny_a()
    q, s = O.quant_act_1x128(xb)
    x = bf16_to_f64(xb)
    xh = dequant_act(q, s)
    s_full = np.repeat(s.astype(np.float64).T, 128, axis=1)
    y = x / s_full                                       # ~ x * r, the encoded quantity
    bound = e4m3_half_ulp(y) * s_full + np.abs(x) * 4 * 2.0 ** -24
    assert np.all(np.abs(x - xh) <= bound)


def test_outlier_changes_only_its_tile():
    g = W.generator(11, "cpu")
    a = W.activations(8, 1024, g, "cpu", outlier_p=0.0)
    q0, s0 = O.quant_act_1x128(bits_of(a))
    a2 = a.clone()
    a2[3, 5 * 128 + 7] = 1000.0
    q1, s1 = O.quant_act_1x128(bits_of(a2))
    changed_tiles = {(m, k // 128) for m, k in zip(*np.nonzero(q0 != q1))}
    assert changed_tiles == {(3, 5)}
    ds = np.argwhere(s0 != s1)
    assert ds.tolist() == [[5, 3]]


def _e4m3_valued_tiles(rng, rows, cols):
    """Random E4M3 values (|v| >= 2^-3) with +-448 somewhere in every 1x128 tile."""
    pos_codes = np.arange(0x28, 0x7F)                     # 2^-3 .. 448
    codes = rng.choice(pos_codes, size=(rows, cols)).astype(np.uint8)
    codes |= (rng.integers(0, 2, (rows, cols)) << 7).astype(np.uint8)
    for kb in range(cols // 128):
        codes[np.arange(rows), kb * 128 + rng.integers(0, 128, rows)] = 0x7E
    return codes


def test_act_identity_on_e4m3_values():
    rng = np.random.default_rng(5)
    codes = _e4m3_valued_tiles(rng, 64, 512)
    x = torch.from_numpy(e4m3_values(codes)).to(torch.bfloat16)    # exact in BF16
    q, s = O.quant_act_1x128(bits_of(x))
    assert np.all(s == 1.0)
    assert np.array_equal(q, codes)


def test_weight_identity_on_e4m3_values():
    rng = np.random.default_rng(6)
    codes = _e4m3_valued_tiles(rng, 256, 384)
    x = torch.from_numpy(e4m3_values(codes)).to(torch.bfloat16)
    q, s = O.quant_weight_128x128(bits_of(x))
    assert np.all(s == 1.0) and np.array_equal(q, codes)


@pytest.mark.parametrize("k", [-125, -100, -70, -64, -63, -20, 0, 40, 100])
def test_power_of_two_scaling_keeps_codes(k):
    rng = np.random.default_rng(7)
    mag = rng.uniform(1.0, 448.0, (16, 256)) * rng.choice([-1, 1], (16, 256))
    base = torch.from_numpy(mag).to(torch.bfloat16)
    scaled = base.double() * 2.0 ** k
    sb = scaled.to(torch.bfloat16)
    assert torch.equal(sb.double(), scaled)              # the scaling is exact in BF16
    q0, s0 = O.quant_act_1x128(bits_of(base))
    q1, s1 = O.quant_act_1x128(bits_of(sb))
    assert np.array_equal(q0, q1)
    s_expect = s0.astype(np.float64) * 2.0 ** k
    normal = np.abs(s_expect) >= 2.0 ** -126
    assert np.array_equal(s1.astype(np.float64)[normal], s_expect[normal])
    assert np.all(s1 > 0)


def test_weight_invariants_ragged_rows():
    g = W.generator(21, "cpu")
    w = W.weights(200, 384, g, "cpu", outlier_p=0.01)     # 2 row blocks, the last 72 rows
    wb = bits_of(w)
    q, s = O.quant_weight_128x128(wb)
    x = bf16_to_f64(wb)
    assert s.shape == (2, 3)
    for nb in range(2):
        for kb in range(3):
            blk = x[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            amax = np.abs(blk).max()
            assert s[nb, kb] == np.float32(amax) / np.float32(448.0)
            vals = e4m3_values(q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128])
            assert np.abs(vals).max() == 448.0
    xh = dequant_weight(q, s)
    s_full = np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)[:200, :384]
    bound = e4m3_half_ulp(x / s_full) * s_full + np.abs(x) * 4 * 2.0 ** -24
    assert np.all(np.abs(x - xh) <= bound)


def test_weight_zero_block_and_padding_rows():
    g = W.generator(22, "cpu")
    w = W.weights(130, 256, g, "cpu")
    w[0:128, 128:256] = 0.0
    q, s = O.quant_weight_128x128(bits_of(w))
    assert s[0, 1] == 1.0 and np.all(q[0:128, 128:256] == 0)
    # Zero rows appended below N do not change any code or scale (amax covers real rows only).
    wp = torch.cat([w, torch.zeros(126, 256, dtype=w.dtype)])
    qp, sp = O.quant_weight_128x128(bits_of(wp))
    assert np.array_equal(qp[:130], q) and np.array_equal(sp, s)
    assert np.all(qp[130:] == 0)


def test_subnormal_only_tile():
    x = torch.zeros(2, 128, dtype=torch.bfloat16)
    x[0, :] = torch.tensor([2.0 ** -133] * 64 + [-(2.0 ** -130)] * 64, dtype=torch.float64).to(
        torch.bfloat16)
    x[1, 5] = -(2.0 ** -126)
    q, s = O.quant_act_1x128(bits_of(x))
    vals = e4m3_values(q)
    assert np.abs(vals[0]).max() == 448.0 and np.abs(vals[1]).max() == 448.0
    assert 0 < s[0, 0] < 2.0 ** -126 and s[0, 1] > 0
    assert vals[0, 0] == 56.0                            # 2^-133 is 1/8 of the amax 2^-130
