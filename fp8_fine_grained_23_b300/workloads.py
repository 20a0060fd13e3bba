"""Seeded synthetic inputs for the FP8 quantize + block-scaled GEMM path.

This module generates inputs only; it holds none of the method's arithmetic. The tests, the
oracle side of the tests and ``bench.py`` all take their inputs from here.

Recipe (every workload):
  * a ``torch.Generator`` on the requested device, seeded with the workload's seed, draws in a
    fixed order: activations, outlier mask, zero-tile mask, then weights;
  * activations are FP32 N(0, 1); each element is multiplied by 100 with probability 0.001
    (outliers); optionally whole 1x128 tiles are zeroed;
  * weights are FP32 N(0, 0.02^2); optionally whole 128x128 blocks are zeroed;
  * BF16 is made from the FP32 draw by round-to-nearest-even (``Tensor.to(torch.bfloat16)``).
The CPU and CUDA generators give different streams for the same seed: a test that compares
the GPU path with the oracle draws once and hands the same BF16 tensor to both.

Backward pass (dense workloads): the output gradient dY [M][N] is drawn like activations and
scaled by 2^-12, from its own generator (the workload's seed + 1000).

MoE routing (grouped workload): expert popularity is proportional to rank^-1.1 with the rank a
seeded permutation of the experts; every token picks 8 distinct experts by Gumbel-top-8 on the
log-popularity (sampling without replacement); the routed rows are sorted by expert and the
group offsets are the prefix sums of the per-expert row counts.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

# --------------------------------------------------------------------------------------
# Workload shapes (the hot path's configurations)
# --------------------------------------------------------------------------------------


@dataclass(frozen=True)
class GemmShape:
    name: str
    M: int
    N: int
    K: int
    seed: int
    out_f32: bool = False
    n_padded: int | None = None   # weight rows padded with zeros to this count


# Tiny quantize + GEMM: A 256x512, W 512x512, FP32 output, one all-zero activation tile.
TINY = GemmShape("tiny_256x512x512", M=256, N=512, K=512, seed=0, out_f32=True)
TINY_ZERO_TILE = (17, 2)          # (row, K block) of the all-zero 1x128 activation tile

# Dense projection: M=4096 tokens, N=18432, K=7168 (hidden), BF16 output.
DENSE = GemmShape("dense_4096x18432x7168", M=4096, N=18432, K=7168, seed=1)

# MLA-style low-rank projections, 8192 tokens, three separate GEMMs to BF16.
MLA = (
    GemmShape("mla_q_down_8192x1536x7168", M=8192, N=1536, K=7168, seed=2),
    GemmShape("mla_kv_down_8192x576x7168", M=8192, N=576, K=7168, seed=3, n_padded=640),
    GemmShape("mla_q_up_8192x24576x1536", M=8192, N=24576, K=1536, seed=4),
)


@dataclass(frozen=True)
class MoEShape:
    name: str = "moe_4096tok_256e_top8"
    tokens: int = 4096
    hidden: int = 7168
    experts: int = 256
    topk: int = 8
    zipf: float = 1.1
    n_gate_up: int = 4096          # gate+up GEMM: K = hidden, N = 4096
    k_down: int = 2048             # down GEMM: K = 2048, N = hidden
    seed: int = 5


MOE = MoEShape()

# Quantizer bandwidth sweep: activations M x 7168, weights 7168 x 18432 (N x K).
SWEEP_ACT_M = (1024, 4096, 16384, 65536)
SWEEP_K = 7168
SWEEP_W_N, SWEEP_W_K = 7168, 18432
SWEEP_SEED = 6
SWEEP_ZERO_TILE_P = 0.01

OUTLIER_P = 1e-3
OUTLIER_MULT = 100.0
W_SIGMA = 0.02


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


# --------------------------------------------------------------------------------------
# Tensors
# --------------------------------------------------------------------------------------


def activations(M: int, K: int, gen: torch.Generator, device, *, outlier_p: float = OUTLIER_P,
                zero_tile_p: float = 0.0, zero_tile: tuple[int, int] | None = None,
                sigma: float = 1.0) -> torch.Tensor:
    """BF16 [M][K]: N(0, sigma^2), outliers x100 with probability outlier_p, zero tiles."""
    a = torch.randn(M, K, generator=gen, device=device, dtype=torch.float32)
    if sigma != 1.0:
        a.mul_(sigma)
    if outlier_p > 0:
        mask = torch.rand(M, K, generator=gen, device=device) < outlier_p
        a = torch.where(mask, a * OUTLIER_MULT, a)
    if zero_tile_p > 0:
        zt = torch.rand(M, K // 128, generator=gen, device=device) < zero_tile_p
        a.view(M, K // 128, 128).masked_fill_(zt.unsqueeze(-1), 0.0)
    if zero_tile is not None:
        m, kb = zero_tile
        a[m, kb * 128:(kb + 1) * 128] = 0.0
    return a.to(torch.bfloat16)


def weights(N: int, K: int, gen: torch.Generator, device, *, sigma: float = W_SIGMA,
            zero_block_p: float = 0.0, outlier_p: float = 0.0) -> torch.Tensor:
    """BF16 [N][K]: N(0, sigma^2), optional outliers x100 and all-zero 128x128 blocks."""
    w = torch.randn(N, K, generator=gen, device=device, dtype=torch.float32).mul_(sigma)
    if outlier_p > 0:
        mask = torch.rand(N, K, generator=gen, device=device) < outlier_p
        w = torch.where(mask, w * OUTLIER_MULT, w)
    if zero_block_p > 0:
        nb, kb = (N + 127) // 128, K // 128
        zb = torch.rand(nb, kb, generator=gen, device=device) < zero_block_p
        rows = zb.repeat_interleave(128, dim=0)[:N]            # [N][KB]
        w.view(N, kb, 128).masked_fill_(rows.unsqueeze(-1), 0.0)
    return w.to(torch.bfloat16)


def gemm_inputs(shape: GemmShape, device) -> tuple[torch.Tensor, torch.Tensor]:
    """(A [M][K], W [N or n_padded][K]) for a dense workload; padded weight rows are zero."""
    g = generator(shape.seed, device)
    zero_tile = TINY_ZERO_TILE if shape is TINY else None
    a = activations(shape.M, shape.K, g, device, zero_tile=zero_tile)
    w = weights(shape.N, shape.K, g, device)
    if shape.n_padded is not None and shape.n_padded > shape.N:
        pad = torch.zeros(shape.n_padded - shape.N, shape.K, dtype=w.dtype, device=device)
        w = torch.cat([w, pad], dim=0)
    return a, w


# Backward pass of a dense projection: X [M][K] and W [N][K] as in the forward workload of the
# same shape, and the output gradient dY [M][N] drawn like activations (N(0, 1), 0.1% x100
# outliers) then scaled by 2^-12 (exact in BF16), from its own generator (seed + 1000).
GRAD_SIGMA = 2.0 ** -12
GRAD_SEED_OFFSET = 1000


def backward_inputs(shape: GemmShape, device) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """(X [M][K], W [N][K], dY [M][N]) for the backward pass of a dense workload."""
    x, w = gemm_inputs(shape, device)
    g = generator(shape.seed + GRAD_SEED_OFFSET, device)
    dy = activations(shape.M, shape.N, g, device, sigma=GRAD_SIGMA)
    return x, w, dy


def sweep_activations(M: int, device) -> torch.Tensor:
    g = generator(SWEEP_SEED + M, device)
    return activations(M, SWEEP_K, g, device, zero_tile_p=SWEEP_ZERO_TILE_P)


def sweep_weight(device) -> torch.Tensor:
    g = generator(SWEEP_SEED, device)
    return weights(SWEEP_W_N, SWEEP_W_K, g, device, sigma=1.0, outlier_p=OUTLIER_P,
                   zero_block_p=SWEEP_ZERO_TILE_P)


# --------------------------------------------------------------------------------------
# MoE routing and grouped inputs
# --------------------------------------------------------------------------------------


def moe_routing(shape: MoEShape = MOE) -> tuple[np.ndarray, np.ndarray]:
    """Returns (offsets int32 [E+1], token_of_row int64 [tokens*topk]) with rows sorted by expert."""
    rng = np.random.default_rng(shape.seed)
    rank = rng.permutation(shape.experts) + 1
    log_pop = -shape.zipf * np.log(rank.astype(np.float64))
    gumbel = rng.gumbel(size=(shape.tokens, shape.experts))
    choice = np.argsort(-(log_pop[None, :] + gumbel), axis=1, kind="stable")[:, :shape.topk]
    expert_of_row = choice.reshape(-1)
    token_of_row = np.repeat(np.arange(shape.tokens, dtype=np.int64), shape.topk)
    order = np.argsort(expert_of_row, kind="stable")
    counts = np.bincount(expert_of_row, minlength=shape.experts)
    offsets = np.zeros(shape.experts + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    return offsets, token_of_row[order]


def moe_row_of_token(token_of_row: np.ndarray, tokens: int, topk: int) -> np.ndarray:
    """Inverse of the routing's row order: int32 [tokens][topk], the sorted rows that hold each
    token, in increasing row (= expert) order."""
    order = np.argsort(token_of_row, kind="stable")        # rows grouped by token, rows ascending
    return order.astype(np.int32).reshape(tokens, topk)


def moe_gate_weights(shape: MoEShape = MOE) -> np.ndarray:
    """Routing weights float32 [tokens][topk]: a seeded softmax over each token's selected
    experts (positive, summing to 1 per token), in the order of moe_row_of_token."""
    rng = np.random.default_rng(shape.seed + 2)
    logits = rng.standard_normal((shape.tokens, shape.topk))
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def synthetic_offsets(counts) -> np.ndarray:
    """Group offsets from explicit per-group row counts (edge-case tests)."""
    counts = np.asarray(counts, np.int64)
    off = np.zeros(counts.size + 1, np.int32)
    off[1:] = np.cumsum(counts)
    return off


def moe_tokens(shape: MoEShape, device) -> torch.Tensor:
    """Token activations [tokens][hidden] BF16 (routed rows are gathered from these)."""
    g = generator(shape.seed, device)
    return activations(shape.tokens, shape.hidden, g, device)


def moe_down_input(shape: MoEShape, rows: int, device) -> torch.Tensor:
    """Input of the down GEMM: an independent seeded [rows][k_down] BF16 tensor."""
    g = generator(shape.seed + 1000, device)
    return activations(rows, shape.k_down, g, device)


def moe_expert_weights(shape: MoEShape, n: int, k: int, which: str, device,
                       experts=None) -> torch.Tensor:
    """Per-expert weights [E][n][k] BF16 ~N(0, 0.02^2); expert e is drawn from its own seed so
    that any subset of experts can be regenerated alone."""
    ids = range(shape.experts) if experts is None else experts
    salt = {"gate_up": 1, "down": 2}[which]
    out = torch.empty(len(ids), n, k, dtype=torch.bfloat16, device=device)
    for i, e in enumerate(ids):
        g = generator(shape.seed * 1_000_003 + salt * 100_003 + int(e), device)
        out[i] = weights(n, k, g, device)
    return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host uint16 bit patterns of a BF16 tensor (for the oracle)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
