"""NumPy front end of the CPU oracle (``fp8_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg use this module; the CUDA library never does. It builds ``liboracle.so`` from
``fp8_oracle.c`` with gcc (no fast-math, no FP contraction) on first use.

What each function computes, and the pages it follows, is documented in ``fp8_oracle.c``:
fine-grained E4M3 quantization with one FP32 scale per 1x128 activation tile and per
128x128 weight block (codingmall.com, "Định lượng hạt mịn" / "Định lượng trực tuyến"), and
the block-scaled GEMM whose per-128-K-block partials are rescaled and accumulated in high
precision (codingmall.com, "Tăng độ chính xác tích lũy"; dtcms.com, section 三.3).

Arrays: BF16 tensors are passed as their uint16 bit patterns; codes are uint8 E4M3FN bytes;
activation scales are float32 [K/128][M]; weight scales float32 [ceil(N/128)][K/128].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile fp8_oracle.c into liboracle.so (strict IEEE: no fast-math, no contraction)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-fno-fast-math", "-ffp-contract=off",
             "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_encode.argtypes = [ctypes.c_float]
            L.orc_e4m3_encode_array.argtypes = [_p, _i64, _p]
            L.orc_e4m3_decode_array.argtypes = [_p, _i64, _p]
            L.orc_quant_act_1x128.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p]
            L.orc_quant_weight_128x128.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p]
            L.orc_gemm_points.argtypes = [_p, _i64, _p, _p, _i64, _p, _i64, _i64, _i64,
                                          _i64, _p, _p, _p, _p, _p]
            L.orc_gemm_f64.argtypes = [_p, _i64, _p, _p, _i64, _p, _i64, _i64, _i64, _p, _p]
            L.orc_grouped_gemm_points.argtypes = [_p, _i64, _p, _p, _i64, _p, _p, _i64, _i64,
                                                  _i64, _i64, _i64, _p, _p, _p, _p]
            L.orc_gemm_unquantized_f64.argtypes = [_p, _i64, _p, _i64, _i64, _i64, _i64, _p]
            L.orc_quant_act_128x1.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p]
            L.orc_quant_weight_128x128_t.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p]
            L.orc_gemm_1d1d_points.argtypes = [_p, _i64, _p, _p, _i64, _p, _i64, _i64, _i64,
                                               _i64, _p, _p, _p, _p, _p]
            L.orc_swiglu_f64.argtypes = [_p, _p, _i64, _p]
            L.orc_quant_act_1x128_ue8m0.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p]
            L.orc_quant_weight_128x128_ue8m0.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p]
            L.orc_ue8m0_exponent.argtypes = [ctypes.c_float]
            L.orc_ue8m0_exponent.restype = ctypes.c_int
            L.orc_moe_permute.argtypes = [_p, _i64, _p, _i64, _p, _i64, _i64, _p, _i64, _p]
            L.orc_moe_combine.argtypes = [_p, _i64, _p, _p, _i64, _i64, _i64, _p, _i64]
            for f in (L.orc_e4m3_encode_array, L.orc_e4m3_decode_array, L.orc_quant_act_1x128,
                      L.orc_quant_weight_128x128, L.orc_gemm_points, L.orc_gemm_f64,
                      L.orc_grouped_gemm_points, L.orc_gemm_unquantized_f64,
                      L.orc_quant_act_128x1, L.orc_quant_weight_128x128_t,
                      L.orc_gemm_1d1d_points, L.orc_swiglu_f64, L.orc_moe_permute,
                      L.orc_moe_combine, L.orc_quant_act_1x128_ue8m0,
                      L.orc_quant_weight_128x128_ue8m0):
                f.restype = None
            _lib = L
        return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------------------
# E4M3
# --------------------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().orc_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_encode(x) -> np.ndarray:
    v = _c(x, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


# --------------------------------------------------------------------------------------
# Quantizers
# --------------------------------------------------------------------------------------

def quant_act_1x128(x_bits) -> tuple[np.ndarray, np.ndarray]:
    """x_bits: uint16 BF16 bits [M][K]. Returns (codes uint8 [M][K], scales f32 [K/128][M])."""
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    assert K % 128 == 0
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // 128, M), np.float32)
    lib().orc_quant_act_1x128(_ptr(x), M, K, K, _ptr(q), K, _ptr(s))
    return q, s


def quant_weight_128x128(w_bits) -> tuple[np.ndarray, np.ndarray]:
    """w_bits: uint16 BF16 bits [N][K]. Returns (codes [N][K], scales f32 [ceil(N/128)][K/128])."""
    w = _c(w_bits, np.uint16)
    N, K = w.shape
    assert K % 128 == 0
    q = np.empty((N, K), np.uint8)
    s = np.empty(((N + 127) // 128, K // 128), np.float32)
    lib().orc_quant_weight_128x128(_ptr(w), N, K, K, _ptr(q), K, _ptr(s))
    return q, s


def ue8m0_exponent(amax: float) -> int:
    """e of the power-of-two tile scale 2^e for a tile maximum amax > 0 (see fp8_oracle.c)."""
    return int(lib().orc_ue8m0_exponent(ctypes.c_float(amax)))


def quant_act_1x128_ue8m0(x_bits) -> tuple[np.ndarray, np.ndarray]:
    """quant_act_1x128 with power-of-two (UE8M0) tile scales; same layouts."""
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    assert K % 128 == 0
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // 128, M), np.float32)
    lib().orc_quant_act_1x128_ue8m0(_ptr(x), M, K, K, _ptr(q), K, _ptr(s))
    return q, s


def quant_weight_128x128_ue8m0(w_bits) -> tuple[np.ndarray, np.ndarray]:
    """quant_weight_128x128 with power-of-two (UE8M0) block scales; same layouts."""
    w = _c(w_bits, np.uint16)
    N, K = w.shape
    assert K % 128 == 0
    q = np.empty((N, K), np.uint8)
    s = np.empty(((N + 127) // 128, K // 128), np.float32)
    lib().orc_quant_weight_128x128_ue8m0(_ptr(w), N, K, K, _ptr(q), K, _ptr(s))
    return q, s


def quant_act_128x1(x_bits) -> tuple[np.ndarray, np.ndarray]:
    """Backward (weight-gradient) tiles of 128 rows x 1 column. x_bits: uint16 BF16 bits
    [M][K], M % 128 == 0. Returns (codes uint8 [K][M], transposed; scales f32 [M/128][K])."""
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    assert M % 128 == 0
    qt = np.empty((K, M), np.uint8)
    s = np.empty((M // 128, K), np.float32)
    lib().orc_quant_act_128x1(_ptr(x), M, K, K, _ptr(qt), M, _ptr(s))
    return qt, s


def quant_weight_128x128_t(w_bits) -> tuple[np.ndarray, np.ndarray]:
    """128x128 blocks of w [N][K] (N, K % 128 == 0) with the codes written as W^T. Returns
    (codes uint8 [K][N], scales f32 [K/128][N/128])."""
    w = _c(w_bits, np.uint16)
    N, K = w.shape
    assert N % 128 == 0 and K % 128 == 0
    qt = np.empty((K, N), np.uint8)
    st = np.empty((K // 128, N // 128), np.float32)
    lib().orc_quant_weight_128x128_t(_ptr(w), N, K, K, _ptr(qt), N, _ptr(st))
    return qt, st


# --------------------------------------------------------------------------------------
# GEMMs
# --------------------------------------------------------------------------------------

def gemm_f64(aq, a_s, wq, w_s) -> tuple[np.ndarray, np.ndarray]:
    """Whole C = A W^T in FP64 on the quantized operands, and sum_k |a_hat w_hat| per element."""
    aq, wq = _c(aq, np.uint8), _c(wq, np.uint8)
    a_s, w_s = _c(a_s, np.float32), _c(w_s, np.float32)
    M, K = aq.shape
    N = wq.shape[0]
    c = np.empty((M, N), np.float64)
    cabs = np.empty((M, N), np.float64)
    lib().orc_gemm_f64(_ptr(aq), K, _ptr(a_s), _ptr(wq), K, _ptr(w_s), M, N, K,
                       _ptr(c), _ptr(cabs))
    return c, cabs


def gemm_points(aq, a_s, wq, w_s, pm, pn, want_f32: bool = False):
    """Selected elements (pm[i], pn[i]): returns (c64, cabs) or (c64, cabs, c32)."""
    aq, wq = _c(aq, np.uint8), _c(wq, np.uint8)
    a_s, w_s = _c(a_s, np.float32), _c(w_s, np.float32)
    pm, pn = _c(pm, np.int64), _c(pn, np.int64)
    M, K = aq.shape
    N = wq.shape[0]
    n = pm.size
    c = np.empty(n, np.float64)
    cabs = np.empty(n, np.float64)
    c32 = np.empty(n, np.float32) if want_f32 else None
    lib().orc_gemm_points(_ptr(aq), K, _ptr(a_s), _ptr(wq), K, _ptr(w_s), M, N, K,
                          n, _ptr(pm), _ptr(pn), _ptr(c), _ptr(cabs), _ptr(c32))
    return (c, cabs, c32) if want_f32 else (c, cabs)


def gemm_1d1d_points(aq, a_s, bq, b_s, pm, pn, want_f32: bool = False):
    """Per-row scales on both operands: aq [M][K], a_s [K/128][M]; bq [N][K], b_s [K/128][N].
    Returns (c64, cabs) or (c64, cabs, c32) at (pm[i], pn[i])."""
    aq, bq = _c(aq, np.uint8), _c(bq, np.uint8)
    a_s, b_s = _c(a_s, np.float32), _c(b_s, np.float32)
    pm, pn = _c(pm, np.int64), _c(pn, np.int64)
    M, K = aq.shape
    N = bq.shape[0]
    assert a_s.shape == (K // 128, M) and b_s.shape == (K // 128, N)
    n = pm.size
    c = np.empty(n, np.float64)
    cabs = np.empty(n, np.float64)
    c32 = np.empty(n, np.float32) if want_f32 else None
    lib().orc_gemm_1d1d_points(_ptr(aq), K, _ptr(a_s), _ptr(bq), K, _ptr(b_s), M, N, K,
                               n, _ptr(pm), _ptr(pn), _ptr(c), _ptr(cabs), _ptr(c32))
    return (c, cabs, c32) if want_f32 else (c, cabs)


def gemm_1d1d_f64(aq, a_s, bq, b_s) -> tuple[np.ndarray, np.ndarray]:
    """Whole output of gemm_1d1d_points, (C64 [M][N], Cabs [M][N])."""
    M, N = aq.shape[0], bq.shape[0]
    mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    c, cabs = gemm_1d1d_points(aq, a_s, bq, b_s, mm.ravel(), nn.ravel())
    return c.reshape(M, N), cabs.reshape(M, N)


def grouped_gemm_points(aq, a_s, wq, w_s, offsets, pr, pn):
    """Grouped GEMM elements. aq [R][K]; a_s [K/128][R]; wq [G][N][K]; w_s [G][NB][KB];
    offsets int32 [G+1]. Returns (c64, cabs) at (pr[i], pn[i])."""
    aq, wq = _c(aq, np.uint8), _c(wq, np.uint8)
    a_s, w_s = _c(a_s, np.float32), _c(w_s, np.float32)
    off = _c(offsets, np.int32)
    pr, pn = _c(pr, np.int64), _c(pn, np.int64)
    R, K = aq.shape
    G, N = off.size - 1, wq.shape[1]
    assert wq.shape[0] == G and w_s.shape[0] == G, "one weight matrix per group"
    n = pr.size
    c = np.empty(n, np.float64)
    cabs = np.empty(n, np.float64)
    lib().orc_grouped_gemm_points(_ptr(aq), K, _ptr(a_s), _ptr(wq), K, _ptr(w_s), _ptr(off),
                                  G, R, N, K, n, _ptr(pr), _ptr(pn), _ptr(c), _ptr(cabs))
    return c, cabs


def swiglu_f64(g, u) -> np.ndarray:
    """h = silu(g) * u elementwise in FP64 (the expert FFN activation, a reading)."""
    g, u = _c(g, np.float64), _c(u, np.float64)
    assert g.shape == u.shape
    h = np.empty(g.shape, np.float64)
    lib().orc_swiglu_f64(_ptr(g), _ptr(u), g.size, _ptr(h))
    return h


def gate_up_columns(I: int) -> tuple[np.ndarray, np.ndarray]:
    """Columns of the gate and up outputs of channel c (0 <= c < I) in a gate/up GEMM whose
    weight rows are interleaved in blocks of 128: gate 256 (c // 128) + c % 128, up + 128."""
    c = np.arange(I, dtype=np.int64)
    gate = 256 * (c // 128) + c % 128
    return gate, gate + 128


def grouped_swiglu_rows(aq, a_s, wq, w_s, offsets, rows):
    """FP64 reference of the fused grouped gate/up GEMM + SwiGLU for whole rows: returns
    (h, g, gabs, u, uabs), each [len(rows)][I], from the grouped GEMM oracle."""
    rows = _c(rows, np.int64)
    I = wq.shape[1] // 2
    gc, uc = gate_up_columns(I)
    pr = np.repeat(rows, I)
    g, gabs = grouped_gemm_points(aq, a_s, wq, w_s, offsets, pr, np.tile(gc, rows.size))
    u, uabs = grouped_gemm_points(aq, a_s, wq, w_s, offsets, pr, np.tile(uc, rows.size))
    shape = (rows.size, I)
    g, gabs, u, uabs = (x.reshape(shape) for x in (g, gabs, u, uabs))
    return swiglu_f64(g, u), g, gabs, u, uabs


def moe_permute(q, s, tok) -> tuple[np.ndarray, np.ndarray]:
    """Rows of (codes q [T][K], scales s [K/128][T]) gathered in the order tok [R]:
    (qp [R][K], sp [K/128][R])."""
    q, s, tok = _c(q, np.uint8), _c(s, np.float32), _c(tok, np.int32)
    T, K = q.shape
    R = tok.size
    qp = np.empty((R, K), np.uint8)
    sp = np.empty((K // 128, R), np.float32)
    lib().orc_moe_permute(_ptr(q), K, _ptr(s), T, _ptr(tok), R, K, _ptr(qp), K, _ptr(sp))
    return qp, sp


def moe_combine(y_bits, row, w) -> np.ndarray:
    """out[t] = sum_j w[t][j] * y[row[t][j]] (FP32 fma chain in j order, then BF16 RNE).
    y_bits uint16 [R][N]; row int32 [T][topk]; w float32 [T][topk]. Returns uint16 [T][N]."""
    y, row, w = _c(y_bits, np.uint16), _c(row, np.int32), _c(w, np.float32)
    R, N = y.shape
    T, topk = row.shape
    out = np.empty((T, N), np.uint16)
    lib().orc_moe_combine(_ptr(y), N, _ptr(row), _ptr(w), T, topk, N, _ptr(out), N)
    return out


def gemm_unquantized_f64(x_bits, w_bits) -> np.ndarray:
    x, w = _c(x_bits, np.uint16), _c(w_bits, np.uint16)
    M, K = x.shape
    N = w.shape[0]
    c = np.empty((M, N), np.float64)
    lib().orc_gemm_unquantized_f64(_ptr(x), K, _ptr(w), K, M, N, K, _ptr(c))
    return c
