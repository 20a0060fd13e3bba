"""The allocation-free GEMM entry point (fp8_blockscaled_gemm_noalloc) against the regular one.

Some callers cannot let the library allocate device memory: a framework whose own caching
allocator or pool must be the only source of device memory, or a deployment whose device
footprint is fixed before it starts. For them the library runs the dense GEMM with its scratch
word in a fixed array inside its own image. These tests call that entry point through the C ABI
twice in a row (the second call reuses the scratch the first call left behind) on the tiny
workload, a ragged shape and few-row shapes that take the split-K kernel, and check both outputs
against fp8_blockscaled_gemm's within the GEMM tolerance the other tests use (they are in fact
identical: same dispatch, kernels and arithmetic). A fresh process shows that the first calls
allocate nothing: the device's free memory is the same before and after them. The file is named
to be collected last and passes alone in a fresh process as well as after the other tests.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from fp8_fine_grained_23_b300 import workloads as W
from oracle import oracle as O
from tests.gpu_common import F, assert_within_tolerance  # noqa: F401
from tests.helpers import bits_of

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _ragged_inputs(M, N, K, seed):
    g = W.generator(seed, "cpu")
    return W.activations(M, K, g, "cpu"), W.weights(N, K, g, "cpu")


# few-row shapes (M <= 64) take the swap-AB split-K kernel; the others the CTA-pair kernel
@pytest.mark.parametrize("shape", ["tiny", "200x272x384", "1x1536x7168", "16x1536x7168",
                                   "64x400x1024"])
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
        assert F.fp8bs_last_error() == F.FP8BS_OK   # no timeout in either error word
        got = out.float().cpu().numpy().astype(np.float64)
        want = ref.float().cpu().numpy().astype(np.float64)
        assert_within_tolerance(got, want, cabs, name, f"noalloc call {call}")
        assert torch.equal(out, ref)   # the same dispatch, kernel and arithmetic


def test_noalloc_rejects_bad_arguments(F):
    st = F.lib.fp8_blockscaled_gemm_noalloc(0x1000, 0x2004, 0x1000, 0x2004, 4, 24, 128, 0x1000,
                                            24, 0, None)
    assert st == F.FP8BS_ERR_INVALID_ARG


# Run in a fresh process: every tensor is made first (E4M3 codes and scales drawn directly, so
# that no regular library call, which allocates its error word, runs before the measurement);
# one allocation-free library call (fp8bs_last_error) initialises the library's CUDA runtime and,
# with eager module loading, loads its kernels; then the device's free memory is read around the
# two first GEMM calls, one per kernel (M = 16: split-K; M = 256: CTA pairs).
_CHILD = r"""
import json, os, sys
import torch
sys.path.insert(0, os.environ["FP8BS_ROOT"])
from fp8_fine_grained_23_b300 import fp8bs as F
torch.cuda.init()
dev = torch.device("cuda", 0)
g = torch.Generator(device=dev).manual_seed(11)

def codes(r, c):
    q = torch.randint(0, 256, (r, c), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
    return torch.where((q & 0x7F) == 0x7F, q ^ 1, q)      # no NaN codes

K, N = 1024, 512
cases = []
for M in (16, 256):
    aq, wq = codes(M, K), codes(N, K)
    a_s = torch.rand(K // 128, M, generator=g, device=dev) + 0.5
    w_s = torch.rand(N // 128, K // 128, generator=g, device=dev) + 0.5
    outs = [torch.empty(M, N, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    cases.append((M, aq, a_s, wq, w_s, outs))
stream = torch.cuda.current_stream(dev).cuda_stream
assert F.lib.fp8bs_last_error(stream) == 0
torch.cuda.synchronize(dev)
free0 = torch.cuda.mem_get_info(dev)[0]
for M, aq, a_s, wq, w_s, outs in cases:
    for out in outs:
        st = F.lib.fp8_blockscaled_gemm_noalloc(aq.data_ptr(), a_s.data_ptr(), wq.data_ptr(),
                                                w_s.data_ptr(), M, N, K, out.data_ptr(), N, 0,
                                                stream)
        assert st == 0, st
torch.cuda.synchronize(dev)
free1 = torch.cuda.mem_get_info(dev)[0]
same = []
for M, aq, a_s, wq, w_s, outs in cases:
    ref = F.fp8_blockscaled_gemm(aq, a_s, wq, w_s)
    same.append(bool(torch.equal(outs[0], ref) and torch.equal(outs[1], ref)))
torch.cuda.synchronize(dev)
free2 = torch.cuda.mem_get_info(dev)[0]
print(json.dumps({"free0": free0, "free1": free1, "free2": free2, "same": same,
                  "status": F.fp8bs_last_error()}))
"""


def test_noalloc_first_calls_allocate_nothing(F):
    env = dict(os.environ, FP8BS_ROOT=ROOT, CUDA_MODULE_LOADING="EAGER")
    res = subprocess.run([sys.executable, "-c", _CHILD], env=env, capture_output=True, text=True,
                         timeout=300)
    assert res.returncode == 0, res.stderr[-3000:]
    got = json.loads(res.stdout.strip().splitlines()[-1])
    assert got["status"] == F.FP8BS_OK
    assert got["same"] == [True, True]
    assert got["free1"] == got["free0"], (
        f"free device memory changed across the first allocation-free calls: {got}")
