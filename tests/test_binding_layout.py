"""The Python binding checks every tensor's layout against what the C ABI reads before it
passes a pointer: a view with other strides (a column slice, a transpose) or a wrong shape is
rejected with an exception and nothing is launched. Runs without a GPU."""
import pytest
import torch


@pytest.fixture(scope="module")
def F():
    from fp8_fine_grained_23_b300 import build
    build.build()
    from fp8_fine_grained_23_b300 import fp8bs
    return fp8bs


M, N, K = 256, 256, 512


def _gemm_operands():
    a_q = torch.zeros(M, K, dtype=torch.uint8)
    a_s = torch.ones(K // 128, M)
    w_q = torch.zeros(N, K, dtype=torch.uint8)
    w_s = torch.ones(N // 128, K // 128)
    return a_q, a_s, w_q, w_s


def test_gemm_rejects_column_sliced_codes(F):
    a_q, a_s, w_q, w_s = _gemm_operands()
    wide = torch.zeros(M, 2 * K, dtype=torch.uint8)
    with pytest.raises(ValueError, match="a_q must be contiguous"):
        F.fp8_blockscaled_gemm(wide[:, :K], a_s, w_q, w_s)
    with pytest.raises(ValueError, match="w_q must be contiguous"):
        F.fp8_blockscaled_gemm(a_q, a_s, torch.zeros(N, 2 * K, dtype=torch.uint8)[:, K:], w_s)


def test_gemm_rejects_transposed_scales(F):
    a_q, a_s, w_q, w_s = _gemm_operands()
    with pytest.raises(ValueError, match="a_s must have shape"):
        F.fp8_blockscaled_gemm(a_q, torch.ones(M, K // 128), w_q, w_s)
    with pytest.raises(ValueError, match="a_s must be contiguous"):
        F.fp8_blockscaled_gemm(a_q, torch.ones(M, K // 128).t(), w_q, w_s)
    with pytest.raises(ValueError, match="w_s must be contiguous"):
        F.fp8_blockscaled_gemm(a_q, a_s, w_q, torch.ones(K // 128, N // 128).t())
    with pytest.raises(ValueError, match="w_s must have shape"):
        F.fp8_blockscaled_gemm(a_q, a_s, w_q, torch.ones(N // 128 + 1, K // 128))


def test_gemm_rejects_wrong_dtypes_and_output(F):
    a_q, a_s, w_q, w_s = _gemm_operands()
    with pytest.raises(TypeError, match="a_q must be torch.uint8"):
        F.fp8_blockscaled_gemm(a_q.to(torch.int8), a_s, w_q, w_s)
    with pytest.raises(TypeError, match="a_s must be torch.float32"):
        F.fp8_blockscaled_gemm(a_q, a_s.double(), w_q, w_s)
    with pytest.raises(ValueError, match="out must have shape"):
        F.fp8_blockscaled_gemm(a_q, a_s, w_q, w_s, out=torch.empty(M, N + 16, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="unit column stride"):
        F.fp8_blockscaled_gemm(a_q, a_s, w_q, w_s, out=torch.empty(N, M, dtype=torch.bfloat16).t())


def test_correct_layouts_reach_the_device_check(F):
    """Well-formed host tensors pass every layout check and are then refused because the
    library dereferences device pointers only."""
    a_q, a_s, w_q, w_s = _gemm_operands()
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        F.fp8_blockscaled_gemm(a_q, a_s, w_q, w_s)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        F.fp8_quant_act_1x128(torch.zeros(M, K, dtype=torch.bfloat16))


def test_quantizers_check_outputs(F):
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="scales must be contiguous"):
        F.fp8_quant_act_1x128(x, scales=torch.empty(M, K // 128).t())
    with pytest.raises(ValueError, match="q must have shape"):
        F.fp8_quant_act_1x128(x, q=torch.empty(M, K + 128, dtype=torch.uint8))
    with pytest.raises(ValueError, match="unit column stride"):
        F.fp8_quant_act_1x128(torch.zeros(K, M, dtype=torch.bfloat16).t())
    with pytest.raises(TypeError, match="x must be torch.bfloat16"):
        F.fp8_quant_act_1x128(x.float())
    with pytest.raises(ValueError, match="scales must have shape"):
        F.fp8_quant_weight_128x128(x, scales=torch.empty(M // 128, K // 128 + 1))
    with pytest.raises(ValueError, match="scales must have shape"):
        F.fp8_quant_act_128x1(x, scales=torch.empty(K, M // 128))


def test_grouped_checks_stacked_layouts(F):
    G = 2
    a_q = torch.zeros(M, K, dtype=torch.uint8)
    a_s = torch.ones(K // 128, M)
    w_q = torch.zeros(G, N, K, dtype=torch.uint8)
    w_s = torch.ones(G, N // 128, K // 128)
    off = torch.tensor([0, 100, M], dtype=torch.int32)
    with pytest.raises(ValueError, match="w_q must be a 3-D tensor"):
        F.fp8_blockscaled_grouped_gemm(a_q, a_s, w_q.view(G * N, K), w_s, off)
    with pytest.raises(ValueError, match="w_q must be contiguous"):
        F.fp8_blockscaled_grouped_gemm(a_q, a_s, w_q.transpose(0, 1), w_s, off)
    with pytest.raises(ValueError, match="group_offsets must have shape"):
        F.fp8_blockscaled_grouped_gemm(a_q, a_s, w_q, w_s, off[:2])
    with pytest.raises(TypeError, match="group_offsets must be torch.int32"):
        F.fp8_blockscaled_grouped_gemm(a_q, a_s, w_q, w_s, off.long())
    with pytest.raises(ValueError, match="h_s must have shape"):
        F.fp8_blockscaled_grouped_gemm_swiglu_quant(a_q, a_s, w_q, w_s, off,
                                                    h_s=torch.empty(M, N // 256))
    with pytest.raises(ValueError, match="h_s must be contiguous"):
        F.fp8_blockscaled_grouped_gemm_swiglu_quant(a_q, a_s, w_q, w_s, off,
                                                    h_s=torch.empty(M, 2)[:, :1].t())


def test_moe_dispatch_checks(F):
    q = torch.zeros(8, K, dtype=torch.uint8)
    s = torch.ones(K // 128, 8)
    tok = torch.zeros(16, dtype=torch.int32)
    with pytest.raises(ValueError, match="s must be contiguous"):
        F.fp8_moe_permute(q, torch.ones(8, K // 128).t(), tok)
    with pytest.raises(ValueError, match="token_of_row must be contiguous"):
        F.fp8_moe_permute(q, s, torch.zeros(32, dtype=torch.int32)[::2])
    y = torch.zeros(16, K, dtype=torch.bfloat16)
    rows = torch.zeros(4, 8, dtype=torch.int32)
    with pytest.raises(ValueError, match="weights must have shape"):
        F.fp8_moe_combine(y, rows, torch.ones(4, 4))
    with pytest.raises(ValueError, match="row_of_token must be contiguous"):
        F.fp8_moe_combine(y, torch.zeros(8, 4, dtype=torch.int32).t(), torch.ones(4, 8))
