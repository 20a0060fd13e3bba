"""The guard-band wrapper the GPU tests put around the binding catches writes past either end of
an output it allocated (checked on the CPU with a stand-in module and planted overruns)."""
import types

import pytest
import torch

from tests.gpu_common import GuardedBinding


def _fake_module(overrun):
    mod = types.SimpleNamespace(torch=torch)

    def fp8_fake(n):
        out = mod.torch.empty(n, 4, dtype=torch.float32, device="cpu")
        out.fill_(1.0)
        if overrun == "after":
            torch.as_strided(out, (out.numel() + 1,), (1,), out.storage_offset())[-1] = 2.0
        elif overrun == "before":
            torch.as_strided(out, (1,), (1,), out.storage_offset() - 1)[0] = 2.0
        return out
    mod.fp8_fake = fp8_fake
    mod.OTHER = 7
    return mod


def test_clean_call_passes_and_returns_the_output():
    g = GuardedBinding(_fake_module(None))
    out = g.fp8_fake(3)
    assert out.shape == (3, 4) and torch.all(out == 1.0)
    assert g.OTHER == 7


@pytest.mark.parametrize("where", ["after", "before"])
def test_overrun_is_caught(where):
    g = GuardedBinding(_fake_module(where))
    with pytest.raises(AssertionError, match="guard-band bytes"):
        g.fp8_fake(3)


def test_binding_module_is_restored():
    mod = _fake_module("after")
    g = GuardedBinding(mod)
    with pytest.raises(AssertionError):
        g.fp8_fake(2)
    assert mod.torch is torch
