"""Pins of the oracle's SwiGLU (the activation between the two expert GEMMs; a reading, since
the pages name the routed experts but not their activation) and of its gate/up interleaving.

  * silu(x) * u against scipy's logistic function, an independent library routine, and at
    closed-form points (0, large positive, large negative);
  * the fused reference for whole rows equals the grouped GEMM oracle's columns picked by the
    interleaving rule (gate rows 256 j .. 256 j + 127, up rows 256 j + 128 .. 256 j + 255).
"""
import numpy as np
from scipy.special import expit

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.helpers import bits_of


def test_swiglu_against_logistic():
    rng = np.random.default_rng(31)
    g = np.concatenate([rng.normal(0, 3, 5000), rng.normal(0, 30, 1000), [0.0, -0.0, 1e-300]])
    u = rng.normal(0, 2, g.size)
    h = O.swiglu_f64(g, u)
    ref = g * expit(g) * u
    assert np.allclose(h, ref, rtol=1e-14, atol=0)


def test_swiglu_closed_forms():
    g = np.array([0.0, 50.0, 800.0, -50.0, -800.0, 1.0])
    u = np.array([3.0, 2.0, 1.0, 5.0, 5.0, 1.0])
    h = O.swiglu_f64(g, u)
    assert h[0] == 0.0
    assert abs(h[1] - 100.0) <= 1e-18 * 100 + 100 * np.exp(-50.0)
    assert h[2] == 800.0                      # e^-800 underflows: silu(x) = x
    assert abs(h[3]) < 1e-19 and h[4] == 0.0  # e^800 overflows: silu(x) = -0
    assert abs(h[5] - 1.0 / (1.0 + np.exp(-1.0))) < 1e-16


def test_fused_reference_picks_interleaved_columns():
    G, N2, K = 3, 512, 256
    off = W.synthetic_offsets([5, 0, 9])
    R = int(off[-1])
    g = W.generator(32, "cpu")
    a = W.activations(R, K, g, "cpu")
    aq, a_s = O.quant_act_1x128(bits_of(a))
    ws = [O.quant_weight_128x128(bits_of(W.weights(N2, K, g, "cpu"))) for _ in range(G)]
    wq = np.stack([w[0] for w in ws])
    w_s = np.stack([w[1] for w in ws])
    rows = np.arange(R)
    h, gg, _, uu, _ = O.grouped_swiglu_rows(aq, a_s, wq, w_s, off, rows)
    full, _ = O.grouped_gemm_points(aq, a_s, wq, w_s, off, np.repeat(rows, N2),
                                    np.tile(np.arange(N2), R))
    full = full.reshape(R, N2)
    for c in (0, 5, 127, 128, 200, 255):
        j, i = divmod(c, 128)
        assert np.array_equal(gg[:, c], full[:, 256 * j + i])
        assert np.array_equal(uu[:, c], full[:, 256 * j + 128 + i])
    assert np.array_equal(h, O.swiglu_f64(gg, uu))
