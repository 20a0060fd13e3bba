"""Pins of the oracle's MoE dispatch (the token side of routing each token to 8 experts):
permute (gather token rows into expert-sorted order) and combine (routing-weighted sum of a
token's expert outputs, FP32 fma chain, BF16 out).

  * permute equals NumPy fancy indexing, and gathering with the inverse order restores the
    token rows (a permutation of the 8 copies);
  * combine with one-hot weights returns the selected row exactly; with the weights of a
    token all 1/8 and equal rows it returns the row; against an FP64 sum it is within the
    FP32 chain's rounding bound plus half a BF16 ulp.
"""
import numpy as np

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.helpers import bf16_to_f64

SMALL = W.MoEShape(name="small", tokens=64, hidden=256, experts=16, topk=4, zipf=1.1,
                   n_gate_up=256, k_down=128, seed=3)


def test_permute_is_fancy_indexing_and_invertible():
    rng = np.random.default_rng(1)
    T, K = 64, 384
    q = rng.integers(0, 256, (T, K), dtype=np.uint8)
    s = rng.random((K // 128, T), dtype=np.float32)
    off, tok = W.moe_routing(SMALL)
    qp, sp = O.moe_permute(q, s, tok)
    assert np.array_equal(qp, q[tok]) and np.array_equal(sp, s[:, tok])
    rows = W.moe_row_of_token(tok, SMALL.tokens, SMALL.topk)
    assert np.all(tok[rows] == np.arange(T)[:, None])
    for j in range(SMALL.topk):
        assert np.array_equal(qp[rows[:, j]], q)


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    b = np.asarray(x, np.float32).view(np.uint32)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def test_combine_one_hot_and_uniform():
    rng = np.random.default_rng(2)
    R, N, T, topk = 40, 256, 10, 4
    y = _bf16_bits(rng.standard_normal((R, N)))
    row = np.stack([rng.choice(R, topk, replace=False) for _ in range(T)]).astype(np.int32)
    w = np.zeros((T, topk), np.float32)
    w[np.arange(T), rng.integers(0, topk, T)] = 1.0
    out = O.moe_combine(y, row, w)
    pick = row[np.arange(T), np.argmax(w, axis=1)]
    assert np.array_equal(out, y[pick])
    same = np.repeat(np.arange(T, dtype=np.int32)[:, None], topk, axis=1)
    out2 = O.moe_combine(y, same, np.full((T, topk), 1.0 / topk, np.float32))
    assert np.array_equal(out2, y[:T])


def test_combine_within_rounding_bound():
    off, tok = W.moe_routing(SMALL)
    rows = W.moe_row_of_token(tok, SMALL.tokens, SMALL.topk)
    w = W.moe_gate_weights(SMALL)
    assert np.allclose(w.sum(axis=1), 1, atol=1e-6) and np.all(w > 0)
    rng = np.random.default_rng(3)
    y = _bf16_bits(rng.standard_normal((tok.size, 192)))
    out = bf16_to_f64(O.moe_combine(y, rows, w))
    yv = bf16_to_f64(y)
    exact = np.einsum("tj,tjn->tn", w.astype(np.float64), yv[rows])
    mag = np.einsum("tj,tjn->tn", np.abs(w).astype(np.float64), np.abs(yv[rows]))
    bound = SMALL.topk * 2.0 ** -24 * mag + 2.0 ** -8 * np.abs(exact) + 1e-30
    assert np.all(np.abs(out - exact) <= bound)
