"""Shared pieces of the GPU parity tests: the library fixture and oracle runners that split big
inputs into row slabs over host threads (the oracle's C calls release the GIL)."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests.helpers import bits_of, gemm_tolerance

THREADS = max(1, min(32, os.cpu_count() or 1))


GUARD_BYTES = 4096   # canary band on each side of every output the binding allocates
GUARD_FILL = 0xA5


class _GuardTorch:
    """Stands in for `torch` inside the binding during one call: its `empty` returns a view into
    a buffer with GUARD_BYTES of canary bytes before and after it, and records the buffer."""

    def __init__(self, real, records):
        self._real = real
        self._records = records

    def __getattr__(self, name):
        return getattr(self._real, name)

    def empty(self, *size, dtype=None, device=None):
        if len(size) == 1 and isinstance(size[0], (tuple, list, torch.Size)):
            size = tuple(size[0])
        dtype = dtype or torch.float32
        elem = torch.empty((), dtype=dtype).element_size()
        pad = GUARD_BYTES // elem
        numel = int(np.prod(size)) if size else 1
        buf = self._real.empty(numel + 2 * pad, dtype=dtype, device=device)
        buf.view(torch.uint8).fill_(GUARD_FILL)
        self._records.append((buf, pad * elem))
        return buf[pad:pad + numel].view(size)


class GuardedBinding:
    """The binding with guard bands around every output it allocates: each fp8_* call runs with
    its outputs inside canary bands, and after the call (synchronized) both bands must still
    hold the canary bytes, so a kernel that writes past either end of an output fails the test
    that called it. Other attributes pass through."""

    def __init__(self, mod):
        self._mod = mod

    def __getattr__(self, name):
        v = getattr(self._mod, name)
        if name.startswith("fp8_") and callable(v):
            def call(*args, **kw):
                records = []
                real = self._mod.torch
                self._mod.torch = _GuardTorch(real, records)
                try:
                    out = v(*args, **kw)
                finally:
                    self._mod.torch = real
                if records:
                    if torch.cuda.is_available():
                        torch.cuda.synchronize()
                    for buf, pad in records:
                        b = buf.view(torch.uint8)
                        bad = int((b[:pad] != GUARD_FILL).sum() + (b[b.numel() - pad:] != GUARD_FILL).sum())
                        assert bad == 0, f"{name}: {bad} guard-band bytes around an output were written"
                return out
            return call
        return v


@pytest.fixture(scope="session")
def F():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from fp8_fine_grained_23_b300 import build
    build.build()
    from fp8_fine_grained_23_b300 import fp8bs
    return GuardedBinding(fp8bs)


def oracle_quant_act(x_bits: np.ndarray):
    """Oracle 1x128 quantization of [M][K] BF16 bits, row slabs on host threads."""
    M = x_bits.shape[0]
    if M < 4096:
        return O.quant_act_1x128(x_bits)
    cuts = np.linspace(0, M, THREADS + 1).astype(int)
    with ThreadPoolExecutor(THREADS) as ex:
        parts = list(ex.map(lambda i: O.quant_act_1x128(x_bits[cuts[i]:cuts[i + 1]]),
                            range(THREADS)))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts], axis=1)


def oracle_quant_weight(w_bits: np.ndarray):
    """Oracle 128x128 quantization; slabs are whole 128-row blocks."""
    N = w_bits.shape[0]
    nb = (N + 127) // 128
    if nb < 16:
        return O.quant_weight_128x128(w_bits)
    cuts = np.linspace(0, nb, min(THREADS, nb) + 1).astype(int) * 128
    cuts[-1] = N
    with ThreadPoolExecutor(THREADS) as ex:
        parts = list(ex.map(lambda i: O.quant_weight_128x128(w_bits[cuts[i]:cuts[i + 1]]),
                            range(len(cuts) - 1)))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts], axis=0)


def oracle_points(aq, a_s, wq, w_s, pm, pn):
    """Oracle GEMM elements at (pm[i], pn[i]) split over host threads."""
    n = pm.size
    cuts = np.linspace(0, n, THREADS + 1).astype(int)
    with ThreadPoolExecutor(THREADS) as ex:
        parts = list(ex.map(
            lambda i: O.gemm_points(aq, a_s, wq, w_s, pm[cuts[i]:cuts[i + 1]],
                                    pn[cuts[i]:cuts[i + 1]]), range(THREADS)))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def assert_codes_equal(q_gpu: torch.Tensor, q_orc: np.ndarray):
    g = q_gpu.cpu().numpy()
    if not np.array_equal(g, q_orc):
        bad = np.argwhere(g != q_orc)
        i = tuple(bad[0])
        raise AssertionError(f"{len(bad)} codes differ; first at {i}: gpu {g[i]:#04x} "
                             f"oracle {q_orc[i]:#04x}")


def assert_scales_equal(s_gpu: torch.Tensor, s_orc: np.ndarray):
    g = s_gpu.cpu().numpy().view(np.uint32)
    o = np.ascontiguousarray(s_orc).view(np.uint32)
    if not np.array_equal(g, o):
        bad = np.argwhere(g != o)
        i = tuple(bad[0])
        raise AssertionError(f"{len(bad)} scales differ; first at {i}: gpu "
                             f"{g[i].view(np.float32)!r} oracle {o[i].view(np.float32)!r}")


def assert_within_tolerance(c_gpu: np.ndarray, c64: np.ndarray, cabs: np.ndarray, out_dtype: str,
                            what: str = ""):
    tol = gemm_tolerance(c64, cabs, out_dtype)
    err = np.abs(c_gpu.astype(np.float64) - c64)
    bad = err > tol
    if bad.any() or not np.isfinite(c_gpu).all():
        i = np.argmax(err - tol)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside |gpu-oracle| <= 1e-5*sum|ab| + 1 ulp; "
            f"worst index {i}: gpu {c_gpu.ravel()[i]!r} oracle {c64.ravel()[i]!r} "
            f"tol {tol.ravel()[i]!r}")
    return float((err / np.maximum(cabs, 1e-300)).max())


def gpu_bits_pair(a: torch.Tensor, w: torch.Tensor):
    return bits_of(a), bits_of(w)


def _column_cuts(n_blocks: int) -> np.ndarray:
    return np.linspace(0, n_blocks, min(THREADS, n_blocks) + 1).astype(int) * 128


def oracle_quant_act_128x1(x_bits: np.ndarray):
    """Oracle 128x1 quantization of [M][K] BF16 bits; column slabs of 128 on host threads.
    Returns (codes [K][M], scales [M/128][K])."""
    K = x_bits.shape[1]
    if x_bits.size < (1 << 22):
        return O.quant_act_128x1(x_bits)
    cuts = _column_cuts(K // 128)
    with ThreadPoolExecutor(THREADS) as ex:
        parts = list(ex.map(lambda i: O.quant_act_128x1(x_bits[:, cuts[i]:cuts[i + 1]]),
                            range(len(cuts) - 1)))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts], axis=1)


def oracle_quant_weight_t(w_bits: np.ndarray):
    """Oracle transposed 128x128 quantization of [N][K]; row-block slabs on host threads.
    Returns (codes [K][N], scales [K/128][N/128])."""
    N = w_bits.shape[0]
    if w_bits.size < (1 << 22):
        return O.quant_weight_128x128_t(w_bits)
    cuts = _column_cuts(N // 128)
    with ThreadPoolExecutor(THREADS) as ex:
        parts = list(ex.map(lambda i: O.quant_weight_128x128_t(w_bits[cuts[i]:cuts[i + 1]]),
                            range(len(cuts) - 1)))
    return (np.concatenate([p[0] for p in parts], axis=1),
            np.concatenate([p[1] for p in parts], axis=1))


def oracle_points_1d1d(aq, a_s, bq, b_s, pm, pn):
    """Oracle per-row-scaled GEMM elements at (pm[i], pn[i]) split over host threads."""
    n = pm.size
    cuts = np.linspace(0, n, THREADS + 1).astype(int)
    with ThreadPoolExecutor(THREADS) as ex:
        parts = list(ex.map(
            lambda i: O.gemm_1d1d_points(aq, a_s, bq, b_s, pm[cuts[i]:cuts[i + 1]],
                                         pn[cuts[i]:cuts[i + 1]]), range(THREADS)))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def oracle_grouped_swiglu_rows(aq, a_s, wq, w_s, offsets, rows):
    """O.grouped_swiglu_rows split over host threads by rows."""
    rows = np.asarray(rows, np.int64)
    cuts = np.linspace(0, rows.size, min(THREADS, rows.size) + 1).astype(int)
    with ThreadPoolExecutor(THREADS) as ex:
        parts = list(ex.map(lambda i: O.grouped_swiglu_rows(aq, a_s, wq, w_s, offsets,
                                                            rows[cuts[i]:cuts[i + 1]]),
                            range(len(cuts) - 1)))
    return tuple(np.concatenate([p[k] for p in parts]) for k in range(5))


def check_requant_tiles(codes, scales, ref, delta, what):
    """Codes [n][N] and scales [n][N/128] of an FP32 result re-quantized in 1x128 tiles, against
    the FP64 reference `ref` [n][N] of that result with error bound `delta` [n][N]: per tile,
    |448 s - amax(ref)| <= max delta (+ FP32 rounding), a +-448 code in every tile clearly above
    zero, and |decode(q) s - ref| <= half an E4M3 step at the value / s, times s, + delta."""
    from tests.helpers import e4m3_half_ulp, e4m3_values
    n, N = ref.shape
    T = N // 128
    rt, dt = ref.reshape(n, T, 128), delta.reshape(n, T, 128)
    amax = np.abs(rt).max(axis=2)
    dmax = dt.max(axis=2)
    s = scales.astype(np.float64)
    bad = np.abs(448.0 * s - amax) > dmax + 2.0 ** -21 * amax + 1e-35
    assert not bad.any(), f"{what}: {int(bad.sum())} scales outside the bound"
    vals = e4m3_values(codes).reshape(n, T, 128)
    live = amax > 4 * dmax
    assert np.all(np.abs(vals).max(axis=2)[live] == 448), f"{what}: a tile without its 448 code"
    sx = s[:, :, None]
    bound = e4m3_half_ulp((np.abs(rt) + dt) / np.maximum(sx, 1e-300)) * sx * (1 + 2.0 ** -20) + dt + 1e-35
    badv = np.abs(vals * sx - rt) > bound
    assert not badv.any(), f"{what}: {int(badv.sum())} of {badv.size} values outside the bound"
