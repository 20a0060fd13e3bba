"""The allocation-free GEMM entry point (fp8_blockscaled_gemm_noalloc) against the regular one.

Some callers cannot let the library allocate device memory: a framework whose own caching
allocator or pool must be the only source of device memory, or a deployment whose device
footprint is fixed before it starts. For them the library runs the dense GEMM with its scratch
word in a fixed array inside its own image. This test calls that entry point through the C ABI
twice in a row (the second call reuses the scratch the first call left behind), on the tiny
workload and on a ragged shape, and checks both outputs against fp8_blockscaled_gemm's, within
the GEMM tolerance the other tests use (they are in fact identical: same kernel, same
arithmetic). The file is named to be collected last and passes alone in a fresh process as well
as after the other tests.
"""
import numpy as np
import pytest
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.gpu_common import F, assert_within_tolerance  # noqa: F401
from tests.helpers import bits_of

pytestmark = pytest.mark.gpu


def _ragged_inputs(M, N, K, seed):
    g = W.generator(seed, "cpu")
    return W.activations(M, K, g, "cpu"), W.weights(N, K, g, "cpu")


@pytest.mark.parametrize("shape", ["tiny", "200x272x384"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_noalloc_gemm_matches_regular_entry_point(F, out_dtype, shape):
    if shape == "tiny":
        a, w = W.gemm_inputs(W.TINY, "cpu")
    else:
        M, N, K = (int(v) for v in shape.split("x"))
        a, w = _ragged_inputs(M, N, K, seed=M + N)
    M, K = a.shape
    N = w.shape[0]
    aq, a_s = F.fp8_quant_act_1x128(a.cuda())
    wq, w_s = F.fp8_quant_weight_128x128(w.cuda())
    ref = F.fp8_blockscaled_gemm(aq, a_s, wq, w_s, out_dtype=out_dtype)
    assert F.fp8bs_last_error() == F.FP8BS_OK

    qa, sa = O.quant_act_1x128(bits_of(a))
    qw, sw = O.quant_weight_128x128(bits_of(w))
    _, cabs = O.gemm_f64(qa, sa, qw, sw)
    name = "f32" if out_dtype == torch.float32 else "bf16"
    code = F.FP8BS_OUT_F32 if out_dtype == torch.float32 else F.FP8BS_OUT_BF16
    stream = torch.cuda.current_stream().cuda_stream

    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
        st = F.lib.fp8_blockscaled_gemm_noalloc(aq.data_ptr(), a_s.data_ptr(), wq.data_ptr(),
                                                w_s.data_ptr(), M, N, K, out.data_ptr(), N, code,
                                                stream)
        assert st == F.FP8BS_OK, F.fp8bs_status_string(st)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        want = ref.float().cpu().numpy().astype(np.float64)
        assert_within_tolerance(got, want, cabs, name, f"noalloc call {call}")
        assert torch.equal(out, ref)   # the same kernel and arithmetic: identical results


def test_noalloc_rejects_bad_arguments(F):
    st = F.lib.fp8_blockscaled_gemm_noalloc(0x1000, 0x2004, 0x1000, 0x2004, 4, 24, 128, 0x1000,
                                            24, 0, None)
    assert st == F.FP8BS_ERR_INVALID_ARG
