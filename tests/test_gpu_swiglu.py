"""GPU parity of the grouped gate/up GEMM with the fused SwiGLU and 1x128 re-quantization.

gate and up are FP32 accumulations and silu uses CUDA's expf, so the codes cannot be compared
bit for bit with an FP64 reference. Each 1x128 tile of h is checked against the oracle's FP64
h = silu(gate) * up (grouped GEMM oracle, interleaved gate/up rows) with the error the GEMM
tolerance implies: |gate_gpu - gate| <= 1e-5 * sum|a_hat w_hat| + 1 FP32 ulp (likewise up),
propagated through h (|d silu / dg| <= 1.1) plus a few FP32 roundings, delta_h. Then:
  * scale: |448 s - amax(h)| <= max delta_h over the tile (+ FP32 rounding);
  * every non-degenerate tile holds a code of magnitude 448 (the tile maximum);
  * every value: |decode(q) s - h| <= half an E4M3 step at |h| / s, times s, + delta_h.
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.gpu_common import F, oracle_grouped_swiglu_rows  # noqa: F401
from tests.helpers import bits_of, e4m3_half_ulp, e4m3_values, gemm_tolerance

pytestmark = pytest.mark.gpu


def check_tiles(hq_rows, hs_rows, h, g, gabs, u, uabs, what):
    """hq_rows [n][I] codes, hs_rows [n][I/128] scales of the same rows as the oracle arrays."""
    eg, eu = gemm_tolerance(g, gabs, "f32"), gemm_tolerance(u, uabs, "f32")
    silu = O.swiglu_f64(g, np.ones_like(g))
    delta = 1.1 * eg * (np.abs(u) + eu) + np.abs(silu) * eu + 2.0 ** -20 * np.abs(h) + 1e-35
    n, I = h.shape
    T = I // 128
    ht = h.reshape(n, T, 128)
    dt = delta.reshape(n, T, 128)
    amax = np.abs(ht).max(axis=2)
    dmax = dt.max(axis=2)
    s = hs_rows.astype(np.float64)
    err_s = np.abs(448.0 * s - amax)
    bad = err_s > dmax + 2.0 ** -21 * amax + 1e-35
    assert not bad.any(), (f"{what}: {int(bad.sum())} scales off; worst "
                           f"{np.unravel_index(np.argmax(err_s - dmax), err_s.shape)}")
    vals = e4m3_values(hq_rows).reshape(n, T, 128)
    live = amax > 4 * dmax
    assert np.all(np.abs(vals).max(axis=2)[live] == 448), f"{what}: a tile without its 448 code"
    sx = s[:, :, None]
    hu = (np.abs(ht) + dt) / np.maximum(sx, 1e-300)
    bound = e4m3_half_ulp(hu) * sx * (1 + 2.0 ** -20) + dt + 1e-35
    err = np.abs(vals * sx - ht)
    badv = err > bound
    assert not badv.any(), (f"{what}: {int(badv.sum())} of {badv.size} values outside the bound; "
                            f"worst {np.unravel_index(np.argmax(err - bound), err.shape)}")


def _inputs(counts, N2, K, seed):
    G = len(counts)
    off = W.synthetic_offsets(counts)
    R = int(off[-1])
    g = W.generator(seed, "cpu")
    a = W.activations(R, K, g, "cpu")
    ws = [W.weights(N2, K, g, "cpu") for _ in range(G)]
    aq, a_s = O.quant_act_1x128(bits_of(a))
    qs = [O.quant_weight_128x128(bits_of(w)) for w in ws]
    return off, R, a, torch.stack(ws), aq, a_s, np.stack([q[0] for q in qs]), np.stack([q[1] for q in qs])


@pytest.mark.parametrize("counts,N2,K", [([0, 130, 37, 200], 512, 384), ([1, 128, 3], 256, 128),
                                         ([129, 0, 255], 1024, 1024)])
def test_fused_swiglu_small(F, counts, N2, K):
    off, R, a, ws, aq_o, as_o, wq_o, ws_o = _inputs(counts, N2, K, seed=sum(counts) + N2)
    G = len(counts)
    aq, a_s = F.fp8_quant_act_1x128(a.cuda())
    wq, w_s = F.fp8_quant_weight_128x128(ws.view(-1, K).cuda())
    hq, hs = F.fp8_blockscaled_grouped_gemm_swiglu_quant(
        aq, a_s, wq.view(G, N2, K), w_s.view(G, N2 // 128, K // 128),
        torch.from_numpy(off).cuda())
    assert F.fp8bs_last_error() == F.FP8BS_OK
    # the GPU quantized the same inputs bit for bit like the oracle (checked elsewhere)
    assert np.array_equal(aq.cpu().numpy(), aq_o)
    rows = np.arange(R)
    h, g, gabs, u, uabs = O.grouped_swiglu_rows(aq_o, as_o, wq_o, ws_o, off, rows)
    check_tiles(hq.cpu().numpy(), hs.cpu().numpy().T, h, g, gabs, u, uabs,
                f"groups {counts} N2={N2} K={K}")


def test_fused_swiglu_leading_dimension_and_determinism(F):
    off, R, a, ws, *_ = _inputs([64, 200], 512, 256, seed=9)
    aq, a_s = F.fp8_quant_act_1x128(a.cuda())
    wq, w_s = F.fp8_quant_weight_128x128(ws.view(-1, 256).cuda())
    offs = torch.from_numpy(off).cuda()
    wq3, ws3 = wq.view(2, 512, 256), w_s.view(2, 4, 2)
    buf = torch.full((R, 256 + 48), 0xA5, dtype=torch.uint8, device="cuda")
    hq1, hs1 = F.fp8_blockscaled_grouped_gemm_swiglu_quant(aq, a_s, wq3, ws3, offs, h_q=buf[:, :256])
    hq2, hs2 = F.fp8_blockscaled_grouped_gemm_swiglu_quant(aq, a_s, wq3, ws3, offs)
    assert torch.equal(hq1, hq2) and torch.equal(hs1, hs2)
    assert torch.all(buf[:, 256:] == 0xA5)


def test_fused_swiglu_full_size_moe_sampled(F):
    """The MoE gate/up workload (4096 tokens x top-8 of 256 experts, N2 = 4096, K = 7168) in
    the benchmark's launch configuration; whole rows of 8 experts (the largest and the
    smallest included) against the oracle."""
    shape = W.MOE
    off, token_of_row = W.moe_routing(shape)
    R = int(off[-1])
    N2, K, E = shape.n_gate_up, shape.hidden, shape.experts
    x = W.moe_tokens(shape, "cuda")[torch.from_numpy(token_of_row).cuda()]
    wts = W.moe_expert_weights(shape, N2, K, "gate_up", "cuda")
    aq, a_s = F.fp8_quant_act_1x128(x)
    wq, w_s = F.fp8_quant_weight_128x128(wts.view(-1, K))
    hq, hs = F.fp8_blockscaled_grouped_gemm_swiglu_quant(
        aq, a_s, wq.view(E, N2, K), w_s.view(E, N2 // 128, K // 128), torch.from_numpy(off).cuda())
    assert F.fp8bs_last_error() == F.FP8BS_OK
    counts = np.diff(off)
    rng = np.random.default_rng(7)
    experts = sorted({int(np.argmax(counts)), int(np.argmin(counts))} |
                     set(rng.choice(E, 6, replace=False).tolist()))
    rows = np.concatenate([off[e] + np.sort(rng.choice(counts[e], min(24, counts[e]),
                                                       replace=False)) for e in experts])
    # the oracle quantizes the same BF16 inputs itself (codes checked equal to the GPU's)
    sel_exp = torch.tensor(experts, device="cuda")
    wq_o = np.zeros((E, N2, K), np.uint8)
    ws_o = np.ones((E, N2 // 128, K // 128), np.float32)
    for e in experts:
        q, s = O.quant_weight_128x128(bits_of(wts[e]))
        wq_o[e], ws_o[e] = q, s
    assert np.array_equal(wq.view(E, N2, K)[sel_exp].cpu().numpy(), wq_o[experts])
    xa = bits_of(x[torch.from_numpy(rows).cuda()])
    aq_rows, as_rows = O.quant_act_1x128(xa)
    assert np.array_equal(aq[torch.from_numpy(rows).cuda()].cpu().numpy(), aq_rows)
    # oracle A operand: the sampled rows' codes placed at their row indices
    aq_o = np.zeros((R, K), np.uint8)
    as_o = np.ones((K // 128, R), np.float32)
    aq_o[rows], as_o[:, rows] = aq_rows, as_rows
    h, g, gabs, u, uabs = oracle_grouped_swiglu_rows(aq_o, as_o, wq_o, ws_o, off, rows)
    check_tiles(hq[torch.from_numpy(rows).cuda()].cpu().numpy(),
                hs[:, torch.from_numpy(rows).cuda()].cpu().numpy().T, h, g, gabs, u, uabs,
                "MoE gate/up sampled")
