"""GPU parity of the grouped block-scaled GEMM (routed MoE experts) against the oracle.

Small synthetic groupings (empty groups, one-row groups, groups of exactly 128 rows, a single
group) compare every element; the full MoE workload (4096 tokens, top-8 of 256 experts with
Zipf(1.1) popularity; gate+up N=4096 K=7168 and down N=7168 K=2048) compares sampled rows and
columns of eight experts, including the largest and the smallest.
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.gpu_common import (F, assert_codes_equal, assert_scales_equal,  # noqa: F401
                              assert_within_tolerance, oracle_quant_act, oracle_quant_weight)
from tests.helpers import bits_of

pytestmark = pytest.mark.gpu


def run_grouped(F, a, ws, counts, out_dtype):
    G, N, K = len(ws), ws[0].shape[0], ws[0].shape[1]
    off = W.synthetic_offsets(counts)
    ag = a.cuda()
    aq, a_s = F.fp8_quant_act_1x128(ag)
    # per-expert quantization (a stacked [G*N][K] call needs N % 128 == 0)
    wq = torch.empty(G, N, K, dtype=torch.uint8, device="cuda")
    w_s = torch.empty(G, (N + 127) // 128, K // 128, dtype=torch.float32, device="cuda")
    for g_, w_ in enumerate(ws):
        F.fp8_quant_weight_128x128(w_.cuda(), wq[g_], w_s[g_])
    offs = torch.from_numpy(off).cuda()
    c = F.fp8_blockscaled_grouped_gemm(aq, a_s, wq, w_s, offs, out_dtype=out_dtype)
    assert F.fp8bs_last_error() == F.FP8BS_OK
    return off, aq, a_s, wq, w_s, c


@pytest.mark.parametrize("counts,N,K", [
    ([0, 1, 130, 37, 128], 144, 256),
    ([300], 256, 512),
    ([0, 0, 5, 0, 0], 32, 128),
    ([128, 256, 0, 1, 127, 129], 512, 384),
    ([7] * 40, 64, 128),
])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_small_groupings(F, counts, N, K, out):
    R = int(sum(counts))
    g = W.generator(500 + R + N, "cpu")
    a = W.activations(R, K, g, "cpu")
    ws = [W.weights(N, K, g, "cpu", outlier_p=0.002) for _ in counts]
    dt = torch.float32 if out == "f32" else torch.bfloat16
    off, aq, a_s, wq, w_s, c = run_grouped(F, a, ws, counts, dt)
    qa, sa = O.quant_act_1x128(bits_of(a))
    assert_codes_equal(aq, qa)
    assert_scales_equal(a_s, sa)
    qws = [O.quant_weight_128x128(bits_of(w)) for w in ws]
    wq_o = np.stack([q for q, _ in qws])
    ws_o = np.stack([s for _, s in qws])
    pr = np.repeat(np.arange(R), N)
    pn = np.tile(np.arange(N), R)
    c64, cabs = O.grouped_gemm_points(qa, sa, wq_o, ws_o, off, pr, pn)
    assert_within_tolerance(c.float().cpu().numpy().ravel(), c64, cabs, out, f"groups {counts}")


def test_rows_outside_groups_untouched(F):
    """Rows past off[G] (R > off[G]) belong to no group and are not written."""
    g = W.generator(77, "cpu")
    K, N = 256, 128
    a = W.activations(300, K, g, "cpu").cuda()
    ws = torch.stack([W.weights(N, K, g, "cpu") for _ in range(2)]).cuda()
    aq, a_s = F.fp8_quant_act_1x128(a)
    wq, w_s = F.fp8_quant_weight_128x128(ws.view(2 * N, K))
    off = torch.tensor([0, 100, 250], dtype=torch.int32, device="cuda")
    c = torch.full((300, N), 5.0, dtype=torch.float32, device="cuda")
    F.fp8_blockscaled_grouped_gemm(aq, a_s, wq.view(2, N, K), w_s.view(2, 1, 2), off, out=c)
    assert F.fp8bs_last_error() == F.FP8BS_OK
    assert torch.all(c[250:] == 5.0)
    assert not torch.any(c[:250] == 5.0)


def _moe_check(F, which: str):
    shape = W.MOE
    off, token_of_row = W.moe_routing(shape)
    R = int(off[-1])
    if which == "gate_up":
        N, K = shape.n_gate_up, shape.hidden
        tokens = W.moe_tokens(shape, "cuda")
        a = tokens[torch.from_numpy(token_of_row).cuda()]
    else:
        N, K = shape.hidden, shape.k_down
        a = W.moe_down_input(shape, R, "cuda")
    wts = W.moe_expert_weights(shape, N, K, which, "cuda")
    aq, a_s = F.fp8_quant_act_1x128(a)
    wq, w_s = F.fp8_quant_weight_128x128(wts.view(-1, K))
    offs = torch.from_numpy(off).cuda()
    c = F.fp8_blockscaled_grouped_gemm(aq, a_s, wq.view(shape.experts, N, K),
                                       w_s.view(shape.experts, N // 128, K // 128), offs)
    assert F.fp8bs_last_error() == F.FP8BS_OK

    counts = np.diff(off)
    rng = np.random.default_rng(shape.seed)
    experts = {int(np.argmax(counts)), int(np.argmin(counts))}
    while len(experts) < 8:
        experts.add(int(rng.integers(shape.experts)))
    experts = sorted(experts)
    # oracle: quantize these experts' weights and their rows from the BF16 inputs
    wsub = W.moe_expert_weights(shape, N, K, which, "cuda", experts=experts)
    rows = np.concatenate([np.arange(off[e], off[e + 1]) for e in experts])
    qa, sa = oracle_quant_act(bits_of(a[torch.from_numpy(rows).cuda()].cpu()))
    sub_off = W.synthetic_offsets(counts[experts])
    qw_list = [oracle_quant_weight(bits_of(wsub[i].cpu())) for i in range(len(experts))]
    qw = np.stack([q for q, _ in qw_list])
    sw = np.stack([s for _, s in qw_list])
    pr_l, pn_l = [], []
    for i, e in enumerate(experts):
        local = np.arange(sub_off[i], sub_off[i + 1])
        pick = local if local.size <= 48 else rng.choice(local, 48, replace=False)
        cols = rng.choice(N, 48, replace=False)
        pr_l.append(np.repeat(pick, cols.size))
        pn_l.append(np.tile(cols, pick.size))
    pr, pn = np.concatenate(pr_l), np.concatenate(pn_l)
    c64, cabs = O.grouped_gemm_points(qa, sa, qw, sw, sub_off, pr, pn)
    got = c[torch.from_numpy(rows[pr]).cuda(), torch.from_numpy(pn).cuda()].float().cpu().numpy()
    assert_within_tolerance(got, c64, cabs, "bf16", f"moe {which}")


def test_full_moe_gate_up_sampled(F):
    _moe_check(F, "gate_up")


def test_full_moe_down_sampled(F):
    _moe_check(F, "down")
