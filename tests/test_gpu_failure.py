"""Failure detection on the GPU without faulting it: a pipeline wait that runs out.

A one-shot test hook (fp8bs_debug_skip_release) makes one epilogue warp of the grouped GEMM skip
one release of a TMEM accumulator. The MMA issuer's wait for that release never completes, so it
runs past its clock budget (about a second): the kernel records FP8BS_ERR_TIMEOUT in the device
error word, every role stops and drains its in-flight copies and MMAs, and the kernel returns.
The test checks the status the host reads and that the same process can run the GEMM again with
correct results (the CUDA context stays usable). No trap, assert or invalid access is involved.
"""
import time

import numpy as np
import pytest
import torch

from fp8_fine_grained_23_b300 import workloads as W
from tests.gpu_common import F  # noqa: F401

pytestmark = pytest.mark.gpu


def _grouped_problem():
    counts = [200, 300]
    K, N = 1024, 256
    g = W.generator(91, "cpu")
    a = W.activations(sum(counts), K, g, "cpu").cuda()
    w = torch.stack([W.weights(N, K, g, "cpu") for _ in counts]).cuda()
    return counts, a, w, N, K


def test_timeout_is_reported_and_context_survives(F):
    counts, a, w, N, K = _grouped_problem()
    G = len(counts)
    aq, a_s = F.fp8_quant_act_1x128(a)
    wq, w_s = F.fp8_quant_weight_128x128(w.view(G * N, K))
    offs = torch.from_numpy(W.synthetic_offsets(counts)).cuda()
    run = lambda: F.fp8_blockscaled_grouped_gemm(  # noqa: E731
        aq, a_s, wq.view(G, N, K), w_s.view(G, N // 128, K // 128), offs)
    ref = run()
    assert F.fp8bs_last_error() == F.FP8BS_OK

    assert F.lib.fp8bs_debug_skip_release(3) == F.FP8BS_OK
    t0 = time.time()
    run()
    status = F.fp8bs_last_error()
    waited = time.time() - t0
    assert status == F.FP8BS_ERR_TIMEOUT, F.fp8bs_status_string(status)
    assert 0.1 < waited < 30.0

    again = run()                                 # the hook was one-shot
    assert F.fp8bs_last_error() == F.FP8BS_OK
    assert torch.equal(again, ref)
    x = torch.randn(1024, 1024, device="cuda")
    assert np.isfinite((x @ x).sum().item())      # the context still runs other work
