"""Test-side helpers: dequantization, the GEMM tolerance, and BF16 conversions.

Nothing here is used by the CUDA path; the oracle-pin tests and the GPU parity tests share it.
"""
from __future__ import annotations

import numpy as np
import torch


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    """E4M3FN code values through PyTorch's own float8 type (independent of the oracle)."""
    c = torch.from_numpy(np.ascontiguousarray(codes, np.uint8))
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def dequant_act(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """x_hat[m, k] = value(q[m, k]) * s[k // 128, m]."""
    v = e4m3_values(q)
    M, K = q.shape
    return v * np.repeat(s.astype(np.float64).T, 128, axis=1)[:, :K]


def dequant_weight(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """w_hat[n, k] = value(q[n, k]) * s[n // 128, k // 128]."""
    v = e4m3_values(q)
    N, K = q.shape
    full = np.repeat(np.repeat(s.astype(np.float64), 128, axis=0), 128, axis=1)
    return v * full[:N, :K]


def e4m3_half_ulp(y: np.ndarray) -> np.ndarray:
    """Half the E4M3 grid spacing at |y| (spacing 2^-9 below 2^-6, 2^(e-3) in [2^e, 2^(e+1)))."""
    a = np.abs(np.asarray(y, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return 0.5 * np.exp2(e - 3)


def ulp(x: np.ndarray, out_dtype: str) -> np.ndarray:
    """One unit in the last place of the output type at |x| (the smallest subnormal at 0)."""
    a = np.abs(np.asarray(x, np.float64))
    if out_dtype == "bf16":
        mant, emin = 7, -126
        tiny = 2.0 ** -133
    else:
        mant, emin = 23, -126
        tiny = 2.0 ** -149
    e = np.floor(np.log2(np.maximum(a, 2.0 ** emin)))
    return np.maximum(np.exp2(e - mant), tiny)


GEMM_REL_TOL = 1e-5


def gemm_tolerance(c64: np.ndarray, cabs: np.ndarray, out_dtype: str) -> np.ndarray:
    """|gpu - oracle| <= 1e-5 * sum_k |a_hat_k w_hat_k| + 1 ulp of the output type at |C64|."""
    return GEMM_REL_TOL * cabs + ulp(c64, out_dtype)
