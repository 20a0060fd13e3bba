"""Pins of the oracle's power-of-two (UE8M0) tile scales, a variant that is not on the pages
(the pages' scale is amax/448; Blackwell's block-scaled MMAs take power-of-two scales).

  * the exponent rule by brute force: 448 * 2^e >= amax > 448 * 2^(e-1) for maxima across the
    whole BF16 range, at the boundaries amax = 448 * 2^k and one ulp either side, and the clamp
    at 2^-127;
  * the codes are the E4M3 encoding of the exact quotient x / 2^e (PyTorch's float8 cast, an
    independent routine), no tile saturates, and each non-zero tile's largest code is at least 224;
  * the activation and weight quantizers agree where a 128x128 block is one row of 1x128 tiles
    repeated, and with FP32 scales on inputs whose tile maxima are 448 * 2^k (where both give
    the same scale).
"""
import numpy as np
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.helpers import bf16_to_f64, bits_of, e4m3_values


def test_exponent_rule_brute_force():
    rng = np.random.default_rng(41)
    vals = list(np.float32(2.0) ** rng.uniform(-133, 127, 4000).astype(np.float32))
    for k in range(-140, 120, 7):
        b = np.float32(448.0) * np.float32(2.0) ** k if k > -150 else None
        if b is None or not np.isfinite(b) or b == 0:
            continue
        vals += [b, np.nextafter(b, np.float32(0)), np.nextafter(b, np.float32(np.inf))]
    for a in vals:
        a = float(np.float32(a))
        if a == 0 or not np.isfinite(a):
            continue
        e = O.ue8m0_exponent(a)
        if e > -127:
            assert 448.0 * 2.0 ** e >= a > 448.0 * 2.0 ** (e - 1), (a, e)
        else:
            assert 448.0 * 2.0 ** -127 >= a


def test_codes_are_the_exact_quotient():
    g = W.generator(42, "cpu")
    x = W.activations(64, 512, g, "cpu", zero_tile=(3, 1))
    x[7, 0:128] *= 1e-35                       # a tile whose scale clamps near 2^-127
    xb = bits_of(x)
    q, s = O.quant_act_1x128_ue8m0(xb)
    x64 = bf16_to_f64(xb)
    for kb in range(4):
        tile = x64[:, kb * 128:(kb + 1) * 128]
        sc = s[kb].astype(np.float64)
        assert np.all(np.log2(sc) == np.round(np.log2(sc)))              # powers of two
        quot = torch.from_numpy((tile / sc[:, None]).astype(np.float32))
        ref = quot.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        nz = np.abs(tile).max(axis=1) > 0
        assert np.array_equal(q[nz, kb * 128:(kb + 1) * 128], ref[nz])
        vmax = np.abs(e4m3_values(q[:, kb * 128:(kb + 1) * 128])).max(axis=1)
        assert np.all(vmax[nz] <= 448)
        big = np.abs(tile).max(axis=1) > 448 * 2.0 ** -126
        assert np.all(vmax[big] >= 224)        # amax / s > 224 rounds to at least 224
    assert s[1][3] == 1 and np.all(q[3, 128:256] == 0)


def test_agrees_with_fp32_scales_on_power_of_two_maxima():
    rng = np.random.default_rng(43)
    v = rng.uniform(-1, 1, (8, 256)).astype(np.float32)
    v[:, 0] = 1.0
    v[:, 128] = -1.0
    x = torch.from_numpy(v * np.float32(448.0 * 2.0 ** -3)).to(torch.bfloat16)
    qa, sa = O.quant_act_1x128(bits_of(x))
    qb, sb = O.quant_act_1x128_ue8m0(bits_of(x))
    assert np.array_equal(sa, sb) and np.array_equal(qa, qb)
    w = torch.from_numpy(np.tile(v[:1], (128, 1)) * np.float32(448.0 * 2.0 ** 5)).to(torch.bfloat16)
    qw, sw = O.quant_weight_128x128_ue8m0(bits_of(w))
    qr, sr = O.quant_act_1x128_ue8m0(bits_of(w))
    assert np.array_equal(qw, qr) and np.all(sw[0] == sr[:, 0])
