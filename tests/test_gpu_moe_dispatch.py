"""GPU parity of the MoE dispatch kernels (token permute and weighted combine) against the
oracle: both are bit-exact (gathers; the combine's FP32 fma chain runs in the same order).
Small routings, the full MoE workload (4096 tokens x top-8 of 256 experts, hidden 7168), and
the edges: empty inputs, leading dimensions, out-of-range indices (skipped, nothing faults)."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.gpu_common import F  # noqa: F401

pytestmark = pytest.mark.gpu

SMALL = W.MoEShape(name="small", tokens=64, hidden=384, experts=16, topk=4, zipf=1.1,
                   n_gate_up=256, k_down=128, seed=3)


def _codes(T, K, seed):
    rng = np.random.default_rng(seed)
    return (rng.integers(0, 256, (T, K), dtype=np.uint8),
            rng.random((K // 128, T), dtype=np.float32) + np.float32(0.01))


def _bf16(rows, cols, seed):
    g = W.generator(seed, "cpu")
    return W.activations(rows, cols, g, "cpu")


@pytest.mark.parametrize("shape", [SMALL, W.MOE], ids=["small", "moe_full"])
def test_permute_bit_exact(F, shape):
    off, tok = W.moe_routing(shape)
    q, s = _codes(shape.tokens, shape.hidden, seed=shape.tokens)
    qp, sp = F.fp8_moe_permute(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(),
                               torch.from_numpy(tok.astype(np.int32)).cuda())
    oq, os_ = O.moe_permute(q, s, tok)
    assert np.array_equal(qp.cpu().numpy(), oq)
    assert np.array_equal(sp.cpu().numpy().view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("shape,N", [(SMALL, 256), (W.MOE, W.MOE.hidden)], ids=["small", "moe_full"])
def test_combine_bit_exact(F, shape, N):
    off, tok = W.moe_routing(shape)
    rows = W.moe_row_of_token(tok, shape.tokens, shape.topk)
    wts = W.moe_gate_weights(shape)
    y = _bf16(tok.size, N, seed=N)
    out = F.fp8_moe_combine(y.cuda(), torch.from_numpy(rows).cuda(), torch.from_numpy(wts).cuda())
    ybits = y.view(torch.int16).numpy().view(np.uint16)
    ref = O.moe_combine(ybits, rows, wts)
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), ref)


def test_dispatch_edges(F):
    T, K = 16, 256
    q, s = _codes(T, K, seed=5)
    qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    tok = np.array([3, 0, 15, -1, 16, 7], np.int32)          # two indices out of range
    qp = torch.full((6, K + 32), 0xA5, dtype=torch.uint8, device="cuda")
    sp = torch.full((K // 128, 6), -1.0, dtype=torch.float32, device="cuda")
    F.fp8_moe_permute(qd, sd, torch.from_numpy(tok).cuda(), qp=qp[:, :K], sp=sp)
    assert F.fp8bs_last_error() == F.FP8BS_OK
    g = qp.cpu().numpy()
    for r, t in enumerate(tok):
        if 0 <= t < T:
            assert np.array_equal(g[r, :K], q[t]) and np.array_equal(sp.cpu().numpy()[:, r], s[:, t])
        else:
            assert np.all(g[r, :K] == 0xA5) and np.all(sp.cpu().numpy()[:, r] == -1.0)
    assert np.all(g[:, K:] == 0xA5)
    # combine: an out-of-range row adds nothing
    y = _bf16(4, 64, seed=6)
    rows = torch.tensor([[0, 9], [1, 2]], dtype=torch.int32, device="cuda")
    wts = torch.tensor([[1.0, 5.0], [0.5, 0.5]], dtype=torch.float32, device="cuda")
    out = F.fp8_moe_combine(y.cuda(), rows, wts)
    ref = O.moe_combine(y.view(torch.int16).numpy().view(np.uint16),
                        np.array([[0, 0], [1, 2]], np.int32), np.array([[1.0, 0.0], [0.5, 0.5]], np.float32))
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), ref)
    # empty inputs are no-ops
    F.fp8_moe_permute(qd, sd, torch.empty(0, dtype=torch.int32, device="cuda"))
    F.fp8_moe_combine(y.cuda(), torch.empty(0, 2, dtype=torch.int32, device="cuda"),
                      torch.empty(0, 2, dtype=torch.float32, device="cuda"))
