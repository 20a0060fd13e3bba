"""Python binding of libfp8bs (the C ABI in ``include/fp8bs.h``).

Argument marshalling only: every step of the quantize + GEMM path runs in the library's CUDA
kernels. PyTorch supplies device memory and the current stream. Importing this module fails
loudly when ``libfp8bs.so`` has not been built (``python -m fp8_fine_grained_23_b300.build``);
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8bs.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libfp8bs.so is not built ({LIB_PATH}); run `python -m fp8_fine_grained_23_b300.build`")

lib = ctypes.CDLL(LIB_PATH)

_i64, _p, _int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
lib.fp8_quant_act_1x128.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p, _p]
lib.fp8_quant_weight_128x128.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p, _p]
lib.fp8_quant_act_1x128_ue8m0.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p, _p]
lib.fp8_quant_weight_128x128_ue8m0.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p, _p]
lib.fp8_blockscaled_gemm.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _p, _i64, _int, _p]
lib.fp8_blockscaled_gemm_noalloc.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _p, _i64, _int,
                                             _p]
lib.fp8_blockscaled_grouped_gemm.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _p,
                                             _i64, _int, _p]
lib.fp8_quant_act_128x1.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p, _p]
lib.fp8_quant_weight_128x128_t.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p, _p]
lib.fp8_blockscaled_gemm_1d1d.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _p, _i64, _int, _p]
lib.fp8_blockscaled_grouped_gemm_swiglu_quant.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64,
                                                         _i64, _p, _i64, _p, _p]
lib.fp8_moe_permute.argtypes = [_p, _i64, _p, _i64, _p, _i64, _i64, _p, _i64, _p, _p]
lib.fp8_moe_combine.argtypes = [_p, _i64, _i64, _p, _p, _i64, _i64, _i64, _p, _i64, _p]
lib.fp8_blockscaled_gemm_quant.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _p, _i64, _p, _p]
lib.fp8bs_status_string.argtypes = [_int]
lib.fp8bs_status_string.restype = ctypes.c_char_p
lib.fp8bs_last_error.argtypes = [_p]
lib.fp8bs_debug_skip_release.argtypes = [_int]
for _f in (lib.fp8_quant_act_1x128, lib.fp8_quant_weight_128x128, lib.fp8_blockscaled_gemm,
           lib.fp8_blockscaled_gemm_noalloc, lib.fp8_blockscaled_grouped_gemm,
           lib.fp8bs_last_error, lib.fp8bs_debug_skip_release, lib.fp8_quant_act_128x1,
           lib.fp8_quant_weight_128x128_t, lib.fp8_blockscaled_gemm_1d1d,
           lib.fp8_blockscaled_grouped_gemm_swiglu_quant, lib.fp8_moe_permute,
           lib.fp8_moe_combine, lib.fp8_quant_act_1x128_ue8m0,
           lib.fp8_quant_weight_128x128_ue8m0, lib.fp8_blockscaled_gemm_quant):
    _f.restype = _int

FP8BS_OK = 0
FP8BS_ERR_INVALID_ARG = -1
FP8BS_ERR_MISALIGNED = -2
FP8BS_ERR_UNSUPPORTED_DEVICE = -3
FP8BS_ERR_CUDA = -4
FP8BS_ERR_TIMEOUT = -5
FP8BS_OUT_BF16 = 0
FP8BS_OUT_F32 = 1


class Fp8bsError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call} failed: {fp8bs_status_string(status)} ({status})")


def fp8bs_status_string(status: int) -> str:
    return lib.fp8bs_status_string(status).decode()


def _check(call: str, status: int) -> None:
    if status != FP8BS_OK:
        raise Fp8bsError(call, status)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _rows_ld(t: torch.Tensor, name: str, shape=None, dtype=None) -> tuple[int, int]:
    """Rows and leading dimension of a row-major matrix argument that may be a row slice of a
    wider buffer (unit column stride, row stride >= its width); shape and dtype when given."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != 2 or t.stride(1) != 1 or (t.shape[0] > 1 and t.stride(0) < t.shape[1]):
        raise ValueError(f"{name} must be a 2-D row-major tensor with unit column stride "
                         f"(got shape {tuple(t.shape)}, strides {t.stride()})")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.shape[0], max(t.stride(0), t.shape[1]) if t.shape[0] > 1 else t.shape[1]


def _dense(t: torch.Tensor, name: str, shape, dtype) -> None:
    """A densely packed argument of the layout the C ABI reads with no leading dimension."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major {tuple(shape)}), got strides "
                         f"{t.stride()}")


def _matrix(t: torch.Tensor, name: str, dim: int = 2) -> tuple[int, ...]:
    if not isinstance(t, torch.Tensor) or t.dim() != dim:
        raise ValueError(f"{name} must be a {dim}-D tensor")
    return tuple(t.shape)


def _on_device(*named) -> None:
    """Every tensor argument on one CUDA device: the library dereferences device pointers only."""
    devs = {t.device for _, t in named}
    for name, t in named:
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor, got device {t.device}")
    if len(devs) > 1:
        raise ValueError("all tensor arguments must be on the same device, got "
                         + ", ".join(f"{n}: {t.device}" for n, t in named))


def fp8_quant_act_1x128(x: torch.Tensor, q: torch.Tensor | None = None,
                        scales: torch.Tensor | None = None, stream=None, _fn=None):
    """E4M3 codes [M][K] (uint8) and FP32 scales [K/128][M] of BF16 activations x [M][K]."""
    M, ldx = _rows_ld(x, "x", dtype=torch.bfloat16)
    K = x.shape[1]
    if q is None:
        q = torch.empty(M, K, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(K // 128, M, dtype=torch.float32, device=x.device)
    _, ldq = _rows_ld(q, "q", (M, K), torch.uint8)
    _dense(scales, "scales", (K // 128, M), torch.float32)
    _on_device(("x", x), ("q", q), ("scales", scales))
    fn = _fn or lib.fp8_quant_act_1x128
    _check(fn.__name__, fn(x.data_ptr(), M, K, ldx, q.data_ptr(), ldq, scales.data_ptr(),
                           _stream(stream)))
    return q, scales


def fp8_quant_act_1x128_ue8m0(x: torch.Tensor, q: torch.Tensor | None = None,
                              scales: torch.Tensor | None = None, stream=None):
    """fp8_quant_act_1x128 with power-of-two (UE8M0) tile scales."""
    return fp8_quant_act_1x128(x, q, scales, stream, _fn=lib.fp8_quant_act_1x128_ue8m0)


def fp8_quant_weight_128x128(w: torch.Tensor, q: torch.Tensor | None = None,
                             scales: torch.Tensor | None = None, stream=None, _fn=None):
    """E4M3 codes [N][K] and FP32 scales [ceil(N/128)][K/128] of BF16 weights w [N][K]."""
    N, ldw = _rows_ld(w, "w", dtype=torch.bfloat16)
    K = w.shape[1]
    if q is None:
        q = torch.empty(N, K, dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((N + 127) // 128, K // 128, dtype=torch.float32, device=w.device)
    _, ldq = _rows_ld(q, "q", (N, K), torch.uint8)
    _dense(scales, "scales", ((N + 127) // 128, K // 128), torch.float32)
    _on_device(("w", w), ("q", q), ("scales", scales))
    fn = _fn or lib.fp8_quant_weight_128x128
    _check(fn.__name__, fn(w.data_ptr(), N, K, ldw, q.data_ptr(), ldq, scales.data_ptr(),
                           _stream(stream)))
    return q, scales


def fp8_quant_weight_128x128_ue8m0(w: torch.Tensor, q: torch.Tensor | None = None,
                                   scales: torch.Tensor | None = None, stream=None):
    """fp8_quant_weight_128x128 with power-of-two (UE8M0) block scales."""
    return fp8_quant_weight_128x128(w, q, scales, stream, _fn=lib.fp8_quant_weight_128x128_ue8m0)


def fp8_quant_act_128x1(x: torch.Tensor, qt: torch.Tensor | None = None,
                        scales: torch.Tensor | None = None, stream=None):
    """Backward 128x1 tiles of BF16 x [M][K] (M % 128 == 0): codes transposed, qt [K][M], and
    FP32 scales [M/128][K]."""
    M, ldx = _rows_ld(x, "x", dtype=torch.bfloat16)
    K = x.shape[1]
    if qt is None:
        qt = torch.empty(K, M, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(M // 128, K, dtype=torch.float32, device=x.device)
    _, ldqt = _rows_ld(qt, "qt", (K, M), torch.uint8)
    _dense(scales, "scales", (M // 128, K), torch.float32)
    _on_device(("x", x), ("qt", qt), ("scales", scales))
    _check("fp8_quant_act_128x1",
           lib.fp8_quant_act_128x1(x.data_ptr(), M, K, ldx, qt.data_ptr(), ldqt,
                                   scales.data_ptr(), _stream(stream)))
    return qt, scales


def fp8_quant_weight_128x128_t(w: torch.Tensor, qt: torch.Tensor | None = None,
                               scales_t: torch.Tensor | None = None, stream=None):
    """128x128 blocks of BF16 w [N][K] with the codes written as W^T: qt [K][N] and FP32
    scales_t [K/128][N/128]."""
    N, ldw = _rows_ld(w, "w", dtype=torch.bfloat16)
    K = w.shape[1]
    if qt is None:
        qt = torch.empty(K, N, dtype=torch.uint8, device=w.device)
    if scales_t is None:
        scales_t = torch.empty(K // 128, N // 128, dtype=torch.float32, device=w.device)
    _, ldqt = _rows_ld(qt, "qt", (K, N), torch.uint8)
    _dense(scales_t, "scales_t", (K // 128, N // 128), torch.float32)
    _on_device(("w", w), ("qt", qt), ("scales_t", scales_t))
    _check("fp8_quant_weight_128x128_t",
           lib.fp8_quant_weight_128x128_t(w.data_ptr(), N, K, ldw, qt.data_ptr(), ldqt,
                                          scales_t.data_ptr(), _stream(stream)))
    return qt, scales_t


def _out_code(dtype) -> int:
    if dtype == torch.bfloat16:
        return FP8BS_OUT_BF16
    if dtype == torch.float32:
        return FP8BS_OUT_F32
    raise TypeError("output dtype must be bfloat16 or float32")


def _gemm_operands(a_q, a_s, w_q, w_s, w_scale_shape=None):
    """M, N, K of C = A W^T after checking the operand layouts the C ABI reads: codes
    [M][K] and [N][K] with contiguous rows, activation scales [K/128][M], weight scales
    [ceil(N/128)][K/128] (or `w_scale_shape`)."""
    M, K = _matrix(a_q, "a_q")
    N = _matrix(w_q, "w_q")[0]
    _dense(a_q, "a_q", (M, K), torch.uint8)
    _dense(w_q, "w_q", (N, K), torch.uint8)
    _dense(a_s, "a_s", (K // 128, M), torch.float32)
    _dense(w_s, "w_s", w_scale_shape or ((N + 127) // 128, K // 128), torch.float32)
    return M, N, K


def fp8_blockscaled_gemm(a_q: torch.Tensor, a_s: torch.Tensor, w_q: torch.Tensor,
                         w_s: torch.Tensor, out: torch.Tensor | None = None,
                         out_dtype=torch.bfloat16, stream=None) -> torch.Tensor:
    """C [M][N] = A W^T with per-(1x128) activation and per-(128x128) weight scales."""
    M, N, K = _gemm_operands(a_q, a_s, w_q, w_s)
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype, device=a_q.device)
    _, ldc = _rows_ld(out, "out", (M, N))
    _on_device(("a_q", a_q), ("a_s", a_s), ("w_q", w_q), ("w_s", w_s), ("out", out))
    _check("fp8_blockscaled_gemm",
           lib.fp8_blockscaled_gemm(a_q.data_ptr(), a_s.data_ptr(), w_q.data_ptr(),
                                    w_s.data_ptr(), M, N, K, out.data_ptr(), ldc,
                                    _out_code(out.dtype), _stream(stream)))
    return out


def fp8_blockscaled_gemm_1d1d(a_q: torch.Tensor, a_s: torch.Tensor, b_q: torch.Tensor,
                              b_s: torch.Tensor, out: torch.Tensor | None = None,
                              out_dtype=torch.bfloat16, stream=None) -> torch.Tensor:
    """C [M][N] = A B^T with per-row scales on both operands: a_s [K/128][M], b_s [K/128][N]."""
    N, K = _matrix(b_q, "b_q")
    M = _matrix(a_q, "a_q")[0]
    _dense(b_q, "b_q", (N, K), torch.uint8)
    _dense(a_q, "a_q", (M, K), torch.uint8)
    _dense(a_s, "a_s", (K // 128, M), torch.float32)
    _dense(b_s, "b_s", (K // 128, N), torch.float32)
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype, device=a_q.device)
    _, ldc = _rows_ld(out, "out", (M, N))
    _on_device(("a_q", a_q), ("a_s", a_s), ("b_q", b_q), ("b_s", b_s), ("out", out))
    _check("fp8_blockscaled_gemm_1d1d",
           lib.fp8_blockscaled_gemm_1d1d(a_q.data_ptr(), a_s.data_ptr(), b_q.data_ptr(),
                                         b_s.data_ptr(), M, N, K, out.data_ptr(), ldc,
                                         _out_code(out.dtype), _stream(stream)))
    return out


def fp8_blockscaled_gemm_quant(a_q: torch.Tensor, a_s: torch.Tensor, w_q: torch.Tensor,
                               w_s: torch.Tensor, c_q: torch.Tensor | None = None,
                               c_s: torch.Tensor | None = None, stream=None):
    """C = A W^T re-quantized in the epilogue: E4M3 codes c_q [M][N] and 1x128 scales
    c_s [N/128][M] (N % 128 == 0), the layout of fp8_quant_act_1x128."""
    M, N, K = _gemm_operands(a_q, a_s, w_q, w_s)
    if c_q is None:
        c_q = torch.empty(M, N, dtype=torch.uint8, device=a_q.device)
    if c_s is None:
        c_s = torch.empty(N // 128, M, dtype=torch.float32, device=a_q.device)
    _, ldcq = _rows_ld(c_q, "c_q", (M, N), torch.uint8)
    _dense(c_s, "c_s", (N // 128, M), torch.float32)
    _on_device(("a_q", a_q), ("a_s", a_s), ("w_q", w_q), ("w_s", w_s), ("c_q", c_q),
               ("c_s", c_s))
    _check("fp8_blockscaled_gemm_quant",
           lib.fp8_blockscaled_gemm_quant(a_q.data_ptr(), a_s.data_ptr(), w_q.data_ptr(),
                                          w_s.data_ptr(), M, N, K, c_q.data_ptr(), ldcq,
                                          c_s.data_ptr(), _stream(stream)))
    return c_q, c_s


def fp8_blockscaled_gemm_noalloc(a_q: torch.Tensor, a_s: torch.Tensor, w_q: torch.Tensor,
                                 w_s: torch.Tensor, out: torch.Tensor, stream=None) -> torch.Tensor:
    """fp8_blockscaled_gemm for callers that must not allocate device memory: the library uses a
    fixed scratch word inside its own image instead of allocating one. `out` is required (this
    wrapper allocates nothing either). Calls that may overlap on the GPU must be ordered."""
    M, N, K = _gemm_operands(a_q, a_s, w_q, w_s)
    _, ldc = _rows_ld(out, "out", (M, N))
    _on_device(("a_q", a_q), ("a_s", a_s), ("w_q", w_q), ("w_s", w_s), ("out", out))
    _check("fp8_blockscaled_gemm_noalloc",
           lib.fp8_blockscaled_gemm_noalloc(a_q.data_ptr(), a_s.data_ptr(), w_q.data_ptr(),
                                            w_s.data_ptr(), M, N, K, out.data_ptr(), ldc,
                                            _out_code(out.dtype), _stream(stream)))
    return out


def _grouped_operands(a_q, a_s, w_q, w_s, group_offsets):
    """G, R, N, K of a grouped GEMM after checking its layouts: a_q [R][K], a_s [K/128][R],
    w_q [G][N][K], w_s [G][ceil(N/128)][K/128], all contiguous; group_offsets int32 [G+1]."""
    R, K = _matrix(a_q, "a_q")
    G, N = _matrix(w_q, "w_q", 3)[:2]
    _dense(a_q, "a_q", (R, K), torch.uint8)
    _dense(a_s, "a_s", (K // 128, R), torch.float32)
    _dense(w_q, "w_q", (G, N, K), torch.uint8)
    _dense(w_s, "w_s", (G, (N + 127) // 128, K // 128), torch.float32)
    _dense(group_offsets, "group_offsets", (G + 1,), torch.int32)
    return G, R, N, K


def fp8_blockscaled_grouped_gemm(a_q: torch.Tensor, a_s: torch.Tensor, w_q: torch.Tensor,
                                 w_s: torch.Tensor, group_offsets: torch.Tensor,
                                 out: torch.Tensor | None = None, out_dtype=torch.bfloat16,
                                 stream=None) -> torch.Tensor:
    """Per-group C rows: rows [off[g], off[g+1]) of A use weights w_q[g] ([G][N][K])."""
    G, R, N, K = _grouped_operands(a_q, a_s, w_q, w_s, group_offsets)
    if out is None:
        out = torch.empty(R, N, dtype=out_dtype, device=a_q.device)
    _, ldc = _rows_ld(out, "out", (R, N))
    _on_device(("a_q", a_q), ("a_s", a_s), ("w_q", w_q), ("w_s", w_s),
               ("group_offsets", group_offsets), ("out", out))
    _check("fp8_blockscaled_grouped_gemm",
           lib.fp8_blockscaled_grouped_gemm(a_q.data_ptr(), a_s.data_ptr(), w_q.data_ptr(),
                                            w_s.data_ptr(), group_offsets.data_ptr(), G, R, N, K,
                                            out.data_ptr(), ldc, _out_code(out.dtype),
                                            _stream(stream)))
    return out


def fp8_blockscaled_grouped_gemm_swiglu_quant(a_q: torch.Tensor, a_s: torch.Tensor,
                                              w_q: torch.Tensor, w_s: torch.Tensor,
                                              group_offsets: torch.Tensor,
                                              h_q: torch.Tensor | None = None,
                                              h_s: torch.Tensor | None = None, stream=None):
    """Grouped gate/up GEMM (w_q [G][N2][K], gate and up rows interleaved per 128) with the
    SwiGLU h = silu(gate) * up re-quantized in 1x128 tiles: codes h_q [R][N2/2], scales
    h_s [N2/256][R]."""
    G, R, N2, K = _grouped_operands(a_q, a_s, w_q, w_s, group_offsets)
    if h_q is None:
        h_q = torch.empty(R, N2 // 2, dtype=torch.uint8, device=a_q.device)
    if h_s is None:
        h_s = torch.empty(N2 // 256, R, dtype=torch.float32, device=a_q.device)
    _, ldh = _rows_ld(h_q, "h_q", (R, N2 // 2), torch.uint8)
    _dense(h_s, "h_s", (N2 // 256, R), torch.float32)
    _on_device(("a_q", a_q), ("a_s", a_s), ("w_q", w_q), ("w_s", w_s),
               ("group_offsets", group_offsets), ("h_q", h_q), ("h_s", h_s))
    _check("fp8_blockscaled_grouped_gemm_swiglu_quant",
           lib.fp8_blockscaled_grouped_gemm_swiglu_quant(
               a_q.data_ptr(), a_s.data_ptr(), w_q.data_ptr(), w_s.data_ptr(),
               group_offsets.data_ptr(), G, R, N2, K, h_q.data_ptr(), ldh, h_s.data_ptr(),
               _stream(stream)))
    return h_q, h_s


def fp8_moe_permute(q: torch.Tensor, s: torch.Tensor, token_of_row: torch.Tensor,
                    qp: torch.Tensor | None = None, sp: torch.Tensor | None = None, stream=None):
    """Gather token rows (codes q [T][K], scales s [K/128][T]) into sorted order:
    qp [R][K] = q[token_of_row], sp [K/128][R]."""
    T, ldq = _rows_ld(q, "q", dtype=torch.uint8)
    K = q.shape[1]
    _dense(s, "s", (K // 128, T), torch.float32)
    if not isinstance(token_of_row, torch.Tensor) or token_of_row.dtype != torch.int32:
        raise TypeError("token_of_row must be int32")
    R = token_of_row.numel()
    _dense(token_of_row, "token_of_row", (R,), torch.int32)
    if qp is None:
        qp = torch.empty(R, K, dtype=torch.uint8, device=q.device)
    if sp is None:
        sp = torch.empty(K // 128, R, dtype=torch.float32, device=q.device)
    _, ldqp = _rows_ld(qp, "qp", (R, K), torch.uint8)
    _dense(sp, "sp", (K // 128, R), torch.float32)
    _on_device(("q", q), ("s", s), ("token_of_row", token_of_row), ("qp", qp), ("sp", sp))
    _check("fp8_moe_permute",
           lib.fp8_moe_permute(q.data_ptr(), ldq, s.data_ptr(), T, token_of_row.data_ptr(), R, K,
                               qp.data_ptr(), ldqp, sp.data_ptr(), _stream(stream)))
    return qp, sp


def fp8_moe_combine(y: torch.Tensor, row_of_token: torch.Tensor, weights: torch.Tensor,
                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[t] = sum_j weights[t][j] * y[row_of_token[t][j]] (FP32, BF16 out); y BF16 [R][N]."""
    R, ldy = _rows_ld(y, "y", dtype=torch.bfloat16)
    N = y.shape[1]
    if row_of_token.dtype != torch.int32 or weights.dtype != torch.float32:
        raise TypeError("row_of_token must be int32 and weights float32")
    T, topk = _matrix(row_of_token, "row_of_token")
    _dense(row_of_token, "row_of_token", (T, topk), torch.int32)
    _dense(weights, "weights", (T, topk), torch.float32)
    if out is None:
        out = torch.empty(T, N, dtype=torch.bfloat16, device=y.device)
    _, ldo = _rows_ld(out, "out", (T, N), torch.bfloat16)
    _on_device(("y", y), ("row_of_token", row_of_token), ("weights", weights), ("out", out))
    _check("fp8_moe_combine",
           lib.fp8_moe_combine(y.data_ptr(), ldy, R, row_of_token.data_ptr(), weights.data_ptr(),
                               T, topk, N, out.data_ptr(), ldo, _stream(stream)))
    return out


def fp8bs_last_error(stream=None) -> int:
    """Synchronize the stream; return (and clear) the device error word's status."""
    return lib.fp8bs_last_error(_stream(stream))
