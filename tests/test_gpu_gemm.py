"""GPU parity of the block-scaled FP8 GEMM against the oracle.

Bar (per element): |C_gpu - C_oracle| <= 1e-5 * sum_k |a_hat_k w_hat_k| + 1 ulp of the output type
at |C_oracle|, with C_oracle the FP64 block-scaled product of the oracle's own quantization of the
same BF16 inputs (whose codes and scales are also checked bit-exact against the GPU's).
Small cases compare every element; the full-size dense and MLA workloads compare sampled rows and
columns, in the launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.gpu_common import (F, assert_codes_equal, assert_scales_equal,  # noqa: F401
                              assert_within_tolerance, oracle_points, oracle_quant_act,
                              oracle_quant_weight)
from tests.helpers import bits_of, e4m3_values

pytestmark = pytest.mark.gpu


def gpu_path(F, a, w, out_dtype):
    ag, wg = a.to("cuda"), w.to("cuda")
    aq, a_s = F.fp8_quant_act_1x128(ag)
    wq, w_s = F.fp8_quant_weight_128x128(wg)
    c = F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out_dtype=out_dtype)
    assert F.fp8bs_last_error() == F.FP8BS_OK
    return aq, a_s, wq, w_s, c


def check_full(F, a, w, out_dtype=torch.float32):
    aq, a_s, wq, w_s, c = gpu_path(F, a, w, out_dtype)
    qa, sa = oracle_quant_act(bits_of(a))
    qw, sw = oracle_quant_weight(bits_of(w))
    assert_codes_equal(aq, qa)
    assert_scales_equal(a_s, sa)
    assert_codes_equal(wq, qw)
    assert_scales_equal(w_s, sw)
    c64, cabs = O.gemm_f64(qa, sa, qw, sw)
    name = "f32" if out_dtype == torch.float32 else "bf16"
    return assert_within_tolerance(c.float().cpu().numpy(), c64, cabs, name,
                                   f"{tuple(a.shape)}x{tuple(w.shape)} {name}")


def test_tiny_workload_f32(F):
    a, w = W.gemm_inputs(W.TINY, "cpu")
    check_full(F, a, w, torch.float32)


def test_tiny_workload_bf16(F):
    a, w = W.gemm_inputs(W.TINY, "cpu")
    check_full(F, a, w, torch.bfloat16)


@pytest.mark.parametrize("M,N,K", [
    (1, 16, 128), (1, 256, 256), (3, 272, 384), (129, 144, 128), (130, 512, 640),
    (257, 400, 1024), (128, 768, 512), (383, 1040, 256),
])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_ragged_shapes(F, M, N, K, out):
    g = W.generator(1000 + M + N + K, "cpu")
    a = W.activations(M, K, g, "cpu", zero_tile_p=0.02)
    w = W.weights(N, K, g, "cpu", outlier_p=0.001)
    check_full(F, a, w, torch.float32 if out == "f32" else torch.bfloat16)


def test_identity_quantization_exact_product(F):
    """E4M3-valued inputs with tile max 448 quantize to themselves (s == 1): the GEMM must
    reproduce the plain product of those values within the same bar."""
    rng = np.random.default_rng(17)
    M, N, K = 200, 320, 768

    def codes(rows):
        c = rng.choice(np.arange(0x28, 0x7F), size=(rows, K)).astype(np.uint8)
        c |= (rng.integers(0, 2, (rows, K)) << 7).astype(np.uint8)
        for kb in range(K // 128):
            c[np.arange(rows), kb * 128 + rng.integers(0, 128, rows)] = 0x7E
        return c

    va, vw = e4m3_values(codes(M)), e4m3_values(codes(N))
    a = torch.from_numpy(va).to(torch.bfloat16)
    w = torch.from_numpy(vw).to(torch.bfloat16)
    _, a_s, _, w_s, c = gpu_path(F, a, w, torch.float32)
    assert torch.all(a_s == 1) and torch.all(w_s == 1)
    exact = va @ vw.T
    assert_within_tolerance(c.cpu().numpy(), exact, np.abs(va) @ np.abs(vw).T, "f32", "identity")


def test_cancellation_and_wide_range(F):
    """Rows whose K blocks have scales 2^40 apart, and products that cancel."""
    g = W.generator(23, "cpu")
    a = W.activations(64, 1024, g, "cpu").float()
    a[:, :128] *= 2.0 ** 20
    a[:, 512:640] *= 2.0 ** -20
    w = W.weights(256, 1024, g, "cpu").float()
    w[128:, 256:384] = -w[128:, 256:384]
    a[::2, 256:384] = a[1::2, 256:384]
    check_full(F, a.to(torch.bfloat16), w.to(torch.bfloat16), torch.float32)


def test_repeated_calls_deterministic(F):
    a, w = W.gemm_inputs(W.TINY, "cpu")
    r1 = gpu_path(F, a, w, torch.bfloat16)[-1].clone()
    r2 = gpu_path(F, a, w, torch.bfloat16)[-1]
    assert torch.equal(r1, r2)


def sampled_check(F, shape: W.GemmShape, n_rows=256, n_cols=256):
    a, w = W.gemm_inputs(shape, "cuda")
    aq, a_s = F.fp8_quant_act_1x128(a)
    wq, w_s = F.fp8_quant_weight_128x128(w)
    c = F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out_dtype=torch.bfloat16)
    assert F.fp8bs_last_error() == F.FP8BS_OK
    M, N = a.shape[0], w.shape[0]
    rng = np.random.default_rng(shape.seed)
    rows = np.unique(np.concatenate([np.arange(0, M, max(1, M // n_rows)), [M - 1]]))
    cols = np.unique(np.concatenate([rng.choice(N, min(N, n_cols), replace=False), [0, N - 1]]))
    pm = np.repeat(rows, cols.size)
    pn = np.tile(cols, rows.size)
    qa, sa = oracle_quant_act(bits_of(a.cpu()))
    qw, sw = oracle_quant_weight(bits_of(w.cpu()))
    c64, cabs = oracle_points(qa, sa, qw, sw, pm, pn)
    got = c[torch.from_numpy(pm).cuda(), torch.from_numpy(pn).cuda()].float().cpu().numpy()
    assert_within_tolerance(got, c64, cabs, "bf16", shape.name)
    return c


def test_full_size_dense_sampled(F):
    sampled_check(F, W.DENSE)


def store_warp_case(F):
    """A ragged shape with K loops of 32 blocks and 304 tiles for 74 CTA pairs: the launch the
    host gives the store-warp variant (BF16 output written by a dedicated warp from a staged
    tile). Returns (a, w, BF16 result, FP32 result)."""
    M, N, K = 4000, 4752, 4096
    g = W.generator(4242, "cuda")
    a = W.activations(M, K, g, "cuda")
    w = W.weights(N, K, g, "cuda")
    aq, a_s = F.fp8_quant_act_1x128(a)
    wq, w_s = F.fp8_quant_weight_128x128(w)
    c16 = F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out_dtype=torch.bfloat16)
    c32 = F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out_dtype=torch.float32)
    assert F.fp8bs_last_error() == F.FP8BS_OK
    return a, w, c16, c32


def test_store_warp_variant(F):
    """Every element: the BF16 output equals the FP32 output (another kernel variant, plain
    stores) rounded to BF16, since both form the same FP32 sums; sampled rows and columns,
    among them the ragged last ones, against the oracle."""
    a, w, c16, c32 = store_warp_case(F)
    assert torch.equal(c16, c32.to(torch.bfloat16))
    M, N = c16.shape
    # the same launch into rows of a wider buffer (ldc = N + 64): the 64 extra columns stay put
    aq, a_s = F.fp8_quant_act_1x128(a)
    wq, w_s = F.fp8_quant_weight_128x128(w)
    wide = torch.full((M, N + 64), 3.0, dtype=torch.bfloat16, device="cuda")
    F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out=wide[:, :N])
    assert F.fp8bs_last_error() == F.FP8BS_OK
    assert torch.equal(wide[:, :N], c16)
    assert bool((wide[:, N:] == 3.0).all())
    rows = np.unique(np.concatenate([np.arange(0, M, 61), np.arange(M - 40, M)]))
    cols = np.unique(np.concatenate([np.arange(0, N, 97), np.arange(N - 40, N)]))
    pm, pn = np.repeat(rows, cols.size), np.tile(cols, rows.size)
    qa, sa = oracle_quant_act(bits_of(a.cpu()))
    qw, sw = oracle_quant_weight(bits_of(w.cpu()))
    c64, cabs = oracle_points(qa, sa, qw, sw, pm, pn)
    got = c16[torch.from_numpy(pm).cuda(), torch.from_numpy(pn).cuda()].float().cpu().numpy()
    assert_within_tolerance(got, c64, cabs, "bf16", "store-warp 4000x4752x4096")


def test_full_size_mla_sampled(F):
    for shape in W.MLA:
        sampled_check(F, shape)


def test_mla_padded_and_unpadded_agree(F):
    """kv down-proj N=576 run unpadded (masked tail tile) and padded to 640 with zero rows:
    the first 576 columns must be bit-identical."""
    shape = W.MLA[1]
    a, w = W.gemm_inputs(shape, "cuda")
    assert w.shape[0] == 640
    aq, a_s = F.fp8_quant_act_1x128(a)
    wq_p, ws_p = F.fp8_quant_weight_128x128(w)
    wq_u, ws_u = F.fp8_quant_weight_128x128(w[:576].contiguous())
    c_p = F.fp8_blockscaled_gemm(aq, a_s, wq_p, ws_p, out_dtype=torch.bfloat16)
    c_u = F.fp8_blockscaled_gemm(aq, a_s, wq_u, ws_u, out_dtype=torch.bfloat16)
    assert F.fp8bs_last_error() == F.FP8BS_OK
    assert torch.equal(c_p[:, :576], c_u)


def test_output_leading_dimension(F):
    g = W.generator(41, "cpu")
    a = W.activations(100, 256, g, "cpu").cuda()
    w = W.weights(160, 256, g, "cpu").cuda()
    aq, a_s = F.fp8_quant_act_1x128(a)
    wq, w_s = F.fp8_quant_weight_128x128(w)
    big = torch.full((100, 200), 7.0, dtype=torch.float32, device="cuda")
    F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out=big[:, :160])
    ref = F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out_dtype=torch.float32)
    assert torch.equal(big[:, :160], ref)
    assert torch.all(big[:, 160:] == 7.0)
