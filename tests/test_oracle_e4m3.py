"""Pins of the oracle's E4M3 codec against things other than itself.

* hand-derived fixed points of the E4M3FN bit definition (tests/golden/e4m3_fixed_points.txt);
* PyTorch's independent ``float8_e4m3fn`` conversion (a library routine) for decode, and for
  encode inside the finite range (PyTorch does not saturate above 448, the oracle does);
* brute-force nearest-of-all-codes search over every finite BF16 value, every midpoint between
  adjacent codes +-1 FP32 ulp, and random FP32 values.
The pages only name the format (codingmall.com "Định dạng E4M3 hợp nhất"); saturation and
ties-to-even are this project's reading of "E4M3" (the OCP definition).
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_fixed_points.txt")


def _golden():
    dec, enc = [], []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        kind, a, b = line.split()
        if kind == "decode":
            dec.append((int(a, 16), float(b)))
        else:
            enc.append((float(a), int(b, 16)))
    return dec, enc


def _torch_table() -> np.ndarray:
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _brute_encode(x: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 code by exhaustive search; ties to the even code; |x| >= 448 -> 448;
    the sign bit follows the input's sign (also when the result is zero)."""
    table = _torch_table()
    pos = table[:0x7F]                       # codes 0x00..0x7E, increasing values
    x = np.asarray(x, np.float32)
    a = np.abs(x.astype(np.float64))
    out = np.empty(x.shape, np.uint8)
    for s in range(0, x.size, 8192):
        aa = a.ravel()[s:s + 8192]
        d = np.abs(aa[:, None] - pos[None, :])
        dmin = d.min(axis=1, keepdims=True)
        cand = d == dmin
        # among tied candidates prefer the even code (even mantissa)
        even = cand & (np.arange(0x7F)[None, :] % 2 == 0)
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        pick = np.where(aa >= 448.0, 0x7E, pick)
        out.ravel()[s:s + 8192] = pick
    sign = np.signbit(x).astype(np.uint8) << 7
    return out | sign


def test_golden_fixed_points():
    dec, enc = _golden()
    for code, val in dec:
        got = O.e4m3_decode(np.array([code], np.uint8))[0]
        assert got == val and math.copysign(1, got) == math.copysign(1, val), (hex(code), got)
    for val, code in enc:
        got = int(O.e4m3_encode(np.array([val], np.float32))[0])
        assert got == code, (val, hex(got), hex(code))


def test_decode_matches_torch_all_codes():
    ours = O.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = _torch_table()
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.isnan(ours[nan]).all()
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_encode_all_bf16_bruteforce():
    bits = np.arange(65536, dtype=np.uint32)
    x = (bits << 16).view(np.float32)
    x = x[~np.isnan(x)]
    assert np.array_equal(O.e4m3_encode(x), _brute_encode(x))


def test_encode_midpoints_and_neighbours():
    table = _torch_table()[:0x7F]
    mids = ((table[:-1] + table[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (table[:-1] + table[1:]) / 2)   # exact
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(-np.inf))
    xs = np.concatenate([mids, up, dn, -mids, -up, -dn, table.astype(np.float32),
                         -table.astype(np.float32),
                         np.array([448, 448.5, 463.99, 464, 465, 1e30, 3.4e38], np.float32)])
    got = O.e4m3_encode(xs)
    assert np.array_equal(got, _brute_encode(xs))
    c = np.arange(0x7E)
    assert np.array_equal(O.e4m3_encode(up), c + 1)            # just above a midpoint: upper
    assert np.array_equal(O.e4m3_encode(dn), c)                # just below: lower
    tie = O.e4m3_encode(mids)
    assert np.array_equal(tie, np.where(c % 2 == 0, c, c + 1))  # exact midpoint: even code


def test_encode_random_against_bruteforce_and_torch():
    rng = np.random.default_rng(1234)
    mag = np.exp2(rng.uniform(-14, 10, 300_000))
    x = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    ours = O.e4m3_encode(x)
    assert np.array_equal(ours, _brute_encode(x))
    inr = np.abs(x) < 448
    ref = torch.from_numpy(x[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours[inr], ref)
    assert np.all((ours[~inr] & 0x7F) == 0x7E)


@pytest.mark.parametrize("v,code", [(0.0, 0x00), (-0.0, 0x80), (1e-30, 0x00), (-1e-30, 0x80),
                                    (float("inf"), 0x7E)])
def test_encode_zero_sign_and_saturation(v, code):
    assert O.e4m3_encode(np.array([v], np.float32))[0] == code
