"""Python binding of libbsq.so: block-scaled quantization (MXFP8, NVFP4, MXFP4) and the
block-scaled GEMM with a fused bias + bf16 epilogue on GB300 (sm_103a).

The functions named like the C ABI (``bsq_quantize``, ``bsq_gemm``, ...) only marshal
arguments: torch tensors are passed as device pointers, the current torch stream as the
CUDA stream. ``quantize`` / ``gemm`` / ``linear`` add output allocation with torch (device
memory is the only thing torch provides here). Every step of the computation runs in the
library's CUDA kernels; there is no other implementation, and importing this package
raises if libbsq.so is missing.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional, Union

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# BSQ_LIBRARY=checked selects the checked build (device-side index checks, status
# BSQ_ERR_DEVICE_CHECK on a failed check); the default is the normal build
LIB_PATH = os.path.join(_HERE, "libbsq_checked.so" if os.environ.get("BSQ_LIBRARY") == "checked" else "libbsq.so")

MXFP8, NVFP4, MXFP4 = 1, 2, 3
FLAG_SRC_F32 = 0x100
FLAG_GLOBAL_GIVEN = 0x200
FLAG_STOCHASTIC = 0x400
FORMATS = {"mxfp8": MXFP8, "nvfp4": NVFP4, "mxfp4": MXFP4}

OK, ERR_ARG, ERR_SHAPE, ERR_ALIGN, ERR_ARCH, ERR_LAUNCH, ERR_TIMEOUT, ERR_DEVICE_CHECK = 0, -1, -2, -3, -4, -5, -6, -7

if not os.path.exists(LIB_PATH):
    raise ImportError("%s is not built (run block_scaled_precision_bsq_gb300.build.build() "
                      "or __graft_entry__.build()); there is no fallback implementation" % os.path.basename(LIB_PATH))

_lib = ctypes.CDLL(LIB_PATH)
_i64, _vp, _int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
_lib.bsq_codes_bytes.restype = ctypes.c_size_t
_lib.bsq_codes_bytes.argtypes = [_int, _i64, _i64]
_lib.bsq_scales_bytes.restype = ctypes.c_size_t
_lib.bsq_scales_bytes.argtypes = [_int, _i64, _i64]
_lib.bsq_quantize.restype = _int
_lib.bsq_quantize.argtypes = [_int, _vp, _i64, _i64, _vp, _vp, _vp, _vp]
MAX_BATCH = 8


class QuantItem(ctypes.Structure):
    """bsq_quant_item of bsq.h."""
    _fields_ = [("src", _vp), ("rows", _i64), ("cols", _i64), ("codes", _vp), ("scales", _vp),
                ("global_scale", ctypes.POINTER(ctypes.c_float))]


_lib.bsq_quantize_batch.restype = _int
_lib.bsq_quantize_batch.argtypes = [_int, _int, ctypes.POINTER(QuantItem), _vp]
_lib.bsq_layernorm_quantize.restype = _int
_lib.bsq_layernorm_quantize.argtypes = [_int, _vp, _vp, _vp, ctypes.c_float, _i64, _i64, _vp, _vp, _vp]
_lib.bsq_gemm.restype = _int
_lib.bsq_quantize_dual.argtypes = [_int, _vp, _i64, _i64, ctypes.c_uint64, _vp, _vp, _vp, _vp, _vp, _vp]
_lib.bsq_quantize_dual.restype = _int
_lib.bsq_delayed_global_scale.argtypes = [_vp, _i64, _i64, ctypes.c_float, _vp, _vp]
_lib.bsq_delayed_global_scale.restype = _int
_lib.bsq_convt2x2.argtypes = [_int, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _int, _vp]
_lib.bsq_convt2x2.restype = _int
_lib.bsq_gemm.argtypes = [_int, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp]
_lib.bsq_gemm_splitk.restype = _int
_lib.bsq_gemm_splitk.argtypes = [_int, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, ctypes.c_size_t, _vp]
_lib.bsq_gemm_splitk_scratch.restype = _int
_lib.bsq_gemm_splitk_scratch.argtypes = [_int, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]
_lib.bsq_gemm_splitk_splits.restype = _int
_lib.bsq_gemm_splitk_splits.argtypes = [_int, _i64, _i64, _i64]
_lib.bsq_gemm_gelu.restype = _int
_lib.bsq_gemm_gelu.argtypes = [_int, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp]
_lib.bsq_gemm_gelu_quantize.restype = _int
_lib.bsq_gemm_gelu_quantize.argtypes = [_int, _vp, _vp, _vp, _vp, _vp, _int, _vp, _vp, _i64, _i64, _i64, _vp]
_lib.bsq_get_device_status.restype = _int
_lib.bsq_get_device_status.argtypes = [_vp]
_lib.bsq_selftest_timeout.restype = _int
_lib.bsq_selftest_timeout.argtypes = [_i64, _vp]
_lib.bsq_selftest_device_check.restype = _int
_lib.bsq_selftest_device_check.argtypes = [_vp]
_lib.bsq_test_inject_stall.restype = _int
_lib.bsq_test_inject_stall.argtypes = [_int, _i64, _i64]
KERNEL_GEMM, KERNEL_DUAL, KERNEL_LAYERNORM = 1, 2, 3
_lib.bsq_last_error.restype = _int
_lib.bsq_strerror.restype = ctypes.c_char_p
_lib.bsq_strerror.argtypes = [_int]

EXPORTS = ("bsq_codes_bytes", "bsq_scales_bytes", "bsq_quantize", "bsq_quantize_batch", "bsq_layernorm_quantize",
           "bsq_quantize_dual", "bsq_delayed_global_scale", "bsq_gemm", "bsq_gemm_splitk", "bsq_gemm_splitk_splits",
           "bsq_gemm_splitk_scratch",
           "bsq_gemm_gelu", "bsq_gemm_gelu_quantize", "bsq_convt2x2", "bsq_get_device_status", "bsq_selftest_timeout",
           "bsq_selftest_device_check", "bsq_test_inject_stall",
           "bsq_last_error", "bsq_strerror")

Ptr = Union[int, None, torch.Tensor]


class BsqError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__("%s failed: %d (%s)" % (what, code, bsq_strerror(code)))
        self.code = code


def _p(x: Ptr) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr() if x.numel() > 0 else None
    return int(x)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


# ---------------------------------------------------------------- C ABI, one to one
def bsq_codes_bytes(fmt, rows: int, cols: int) -> int:
    return int(_lib.bsq_codes_bytes(_fmt(fmt), rows, cols))


def bsq_scales_bytes(fmt, rows: int, cols: int) -> int:
    return int(_lib.bsq_scales_bytes(_fmt(fmt), rows, cols))


def bsq_quantize(fmt_flags: int, src: Ptr, rows: int, cols: int, codes: Ptr, scales: Ptr,
                 global_scale: Ptr = None, stream=None) -> int:
    return int(_lib.bsq_quantize(int(fmt_flags), _p(src), rows, cols, _p(codes), _p(scales), _p(global_scale),
                                 _stream(stream)))


def bsq_quantize_batch(fmt_flags: int, items, stream=None) -> int:
    """items: sequence of (src, rows, cols, codes, scales, global_scale) tuples (pointers or
    tensors, as bsq_quantize takes them)."""
    arr = (QuantItem * max(1, len(items)))()
    for i, (src, rows, cols, codes, scales, gs) in enumerate(items):
        g = _p(gs)
        arr[i] = QuantItem(_p(src), rows, cols, _p(codes), _p(scales),
                           ctypes.cast(g, ctypes.POINTER(ctypes.c_float)) if g else None)
    return int(_lib.bsq_quantize_batch(int(fmt_flags), len(items), arr, _stream(stream)))


def bsq_layernorm_quantize(fmt_flags: int, src: Ptr, gamma: Ptr, beta: Ptr, eps: float, rows: int, cols: int,
                           codes: Ptr, scales: Ptr, stream=None) -> int:
    return int(_lib.bsq_layernorm_quantize(int(fmt_flags), _p(src), _p(gamma), _p(beta), float(eps), rows, cols,
                                           _p(codes), _p(scales), _stream(stream)))


def bsq_quantize_dual(fmt_flags: int, src: Ptr, rows: int, cols: int, seed: int, row_codes: Ptr, row_scales: Ptr,
                      col_codes: Ptr, col_scales: Ptr, global_scale: Ptr = None, stream=None) -> int:
    return int(_lib.bsq_quantize_dual(int(fmt_flags), _p(src), rows, cols, int(seed) & (2 ** 64 - 1), _p(row_codes),
                                      _p(row_scales), _p(col_codes), _p(col_scales), _p(global_scale),
                                      _stream(stream)))


def bsq_delayed_global_scale(prev_scales: Ptr, rows: int, cols: int, headroom: float, g_out: Ptr,
                             stream=None) -> int:
    return int(_lib.bsq_delayed_global_scale(_p(prev_scales), rows, cols, float(headroom), _p(g_out),
                                             _stream(stream)))


def bsq_gemm(fmt, A: Ptr, A_scales: Ptr, B: Ptr, B_scales: Ptr, bias: Ptr, out: Ptr, M: int, N: int, K: int,
             stream=None) -> int:
    return int(_lib.bsq_gemm(_fmt(fmt), _p(A), _p(A_scales), _p(B), _p(B_scales), _p(bias), _p(out), M, N, K,
                             _stream(stream)))


def bsq_gemm_splitk(fmt, A: Ptr, A_scales: Ptr, B: Ptr, B_scales: Ptr, bias: Ptr, out: Ptr, M: int, N: int, K: int,
                    splits: int, workspace: Ptr, workspace_bytes: int, stream=None) -> int:
    return int(_lib.bsq_gemm_splitk(_fmt(fmt), _p(A), _p(A_scales), _p(B), _p(B_scales), _p(bias), _p(out), M, N, K,
                                    splits, _p(workspace), workspace_bytes, _stream(stream)))


def bsq_gemm_splitk_scratch(fmt, A: Ptr, A_scales: Ptr, B: Ptr, B_scales: Ptr, bias: Ptr, out: Ptr, M: int, N: int,
                            K: int, splits: int, stream=None) -> int:
    return int(_lib.bsq_gemm_splitk_scratch(_fmt(fmt), _p(A), _p(A_scales), _p(B), _p(B_scales), _p(bias), _p(out),
                                            M, N, K, splits, _stream(stream)))


def bsq_gemm_splitk_splits(fmt, M: int, N: int, K: int) -> int:
    return int(_lib.bsq_gemm_splitk_splits(_fmt(fmt), M, N, K))


def bsq_gemm_gelu(fmt, A: Ptr, A_scales: Ptr, B: Ptr, B_scales: Ptr, bias: Ptr, out: Ptr, M: int, N: int,
                  K: int, stream=None) -> int:
    return int(_lib.bsq_gemm_gelu(_fmt(fmt), _p(A), _p(A_scales), _p(B), _p(B_scales), _p(bias), _p(out), M, N, K,
                                  _stream(stream)))


def bsq_gemm_gelu_quantize(fmt, A: Ptr, A_scales: Ptr, B: Ptr, B_scales: Ptr, bias: Ptr, out_fmt, out_codes: Ptr,
                           out_scales: Ptr, M: int, N: int, K: int, stream=None) -> int:
    return int(_lib.bsq_gemm_gelu_quantize(_fmt(fmt), _p(A), _p(A_scales), _p(B), _p(B_scales), _p(bias),
                                           _fmt(out_fmt), _p(out_codes), _p(out_scales), M, N, K, _stream(stream)))


def bsq_convt2x2(fmt, A: Ptr, A_scales: Ptr, B: Ptr, B_scales: Ptr, bias: Ptr, out: Ptr, batch: int, H: int, W: int,
                 C_in: int, C_out: int, gelu: bool = False, stream=None) -> int:
    return int(_lib.bsq_convt2x2(_fmt(fmt), _p(A), _p(A_scales), _p(B), _p(B_scales), _p(bias), _p(out), batch, H, W,
                                 C_in, C_out, 1 if gelu else 0, _stream(stream)))


def bsq_get_device_status(stream=None) -> int:
    return int(_lib.bsq_get_device_status(_stream(stream)))


def bsq_selftest_timeout(limit_ns: int, stream=None) -> int:
    return int(_lib.bsq_selftest_timeout(int(limit_ns), _stream(stream)))


def bsq_selftest_device_check(stream=None) -> int:
    return int(_lib.bsq_selftest_device_check(_stream(stream)))


def bsq_test_inject_stall(kernel: int, after_stages: int, wait_limit_ns: int) -> int:
    return int(_lib.bsq_test_inject_stall(int(kernel), int(after_stages), int(wait_limit_ns)))


def bsq_last_error() -> int:
    return int(_lib.bsq_last_error())


def bsq_strerror(code: int) -> str:
    return _lib.bsq_strerror(int(code)).decode()


# ---------------------------------------------------------------- tensor-level helpers
@dataclasses.dataclass
class QTensor:
    """A quantized rows x cols matrix: packed codes, tiled scales (with the NVFP4 tail) and,
    for NVFP4, a one-element fp32 tensor holding the per-tensor scale g."""

    fmt: int
    rows: int
    cols: int
    codes: torch.Tensor
    scales: torch.Tensor
    global_scale: Optional[torch.Tensor] = None


def empty_qtensor(fmt, rows: int, cols: int, device="cuda") -> QTensor:
    f = _fmt(fmt)
    codes = torch.empty(bsq_codes_bytes(f, rows, cols), dtype=torch.uint8, device=device)
    scales = torch.empty(bsq_scales_bytes(f, rows, cols), dtype=torch.uint8, device=device)
    g = torch.empty(1, dtype=torch.float32, device=device) if f == NVFP4 else None
    return QTensor(f, rows, cols, codes, scales, g)


def quantize(fmt, x: torch.Tensor, global_scale: Optional[torch.Tensor] = None, out: Optional[QTensor] = None,
             stream=None) -> QTensor:
    """Quantize a contiguous bf16 or fp32 CUDA matrix along its last dimension."""
    f = _fmt(fmt)
    assert x.is_cuda and x.is_contiguous() and x.dim() == 2, "x must be a contiguous 2-D CUDA tensor"
    rows, cols = x.shape
    flags = f
    if x.dtype == torch.float32:
        flags |= FLAG_SRC_F32
    elif x.dtype != torch.bfloat16:
        raise TypeError("x must be bfloat16 or float32")
    q = out if out is not None else empty_qtensor(f, rows, cols, x.device)
    g = q.global_scale
    if global_scale is not None:
        flags |= FLAG_GLOBAL_GIVEN
        g = global_scale
    rc = bsq_quantize(flags, x, rows, cols, q.codes, q.scales, g, stream)
    if rc != OK:
        raise BsqError(rc, "bsq_quantize")
    if global_scale is not None:
        q.global_scale = global_scale
    return q


def quantize_many(fmt, xs, outs=None, stream=None):
    """Quantize several contiguous 2-D CUDA matrices of one dtype (bf16 or fp32) in one launch
    (bsq_quantize_batch); NVFP4 computes each matrix's own g. Returns a list of QTensor."""
    f = _fmt(fmt)
    assert 1 <= len(xs) <= MAX_BATCH, "1..%d matrices per call" % MAX_BATCH
    dt = xs[0].dtype
    for x in xs:
        assert x.is_cuda and x.is_contiguous() and x.dim() == 2 and x.dtype == dt, \
            "matrices must be contiguous 2-D CUDA tensors of one dtype"
    flags = f
    if dt == torch.float32:
        flags |= FLAG_SRC_F32
    elif dt != torch.bfloat16:
        raise TypeError("matrices must be bfloat16 or float32")
    qs = list(outs) if outs is not None else [empty_qtensor(f, x.shape[0], x.shape[1], x.device) for x in xs]
    items = [(x, x.shape[0], x.shape[1], q.codes, q.scales, q.global_scale) for x, q in zip(xs, qs)]
    rc = bsq_quantize_batch(flags, items, stream)
    if rc != OK:
        raise BsqError(rc, "bsq_quantize_batch")
    return qs


def layernorm_quantize(fmt, x: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor, eps: float = 1e-6,
                       out: Optional[QTensor] = None, stream=None) -> QTensor:
    """Row LayerNorm (gamma, beta bf16) of a contiguous bf16 / fp32 CUDA matrix, quantized along
    the row into MXFP8 / MXFP4 in the same kernel."""
    f = _fmt(fmt)
    assert x.is_cuda and x.is_contiguous() and x.dim() == 2, "x must be a contiguous 2-D CUDA tensor"
    rows, cols = x.shape
    assert gamma.dtype == torch.bfloat16 and beta.dtype == torch.bfloat16 and gamma.numel() == cols == beta.numel()
    flags = f | (FLAG_SRC_F32 if x.dtype == torch.float32 else 0)
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("x must be bfloat16 or float32")
    q = out if out is not None else empty_qtensor(f, rows, cols, x.device)
    rc = bsq_layernorm_quantize(flags, x, gamma, beta, eps, rows, cols, q.codes, q.scales, stream)
    if rc != OK:
        raise BsqError(rc, "bsq_layernorm_quantize")
    return q


def quantize_dual(fmt, x: torch.Tensor, stochastic: bool = False, seed: int = 0,
                  global_scale: Optional[torch.Tensor] = None, out=None, stream=None):
    """Both operands of a contiguous bf16 / fp32 CUDA matrix X (R x C, multiples of 32) in one
    launch: (row-wise QTensor R x C, column-wise QTensor C x R = X^T quantized along R), with
    round-to-nearest-even or Philox-keyed stochastic rounding. NVFP4 shares one per-tensor
    scale between the layouts: computed from X, or `global_scale` (a one-element fp32 tensor)."""
    f = _fmt(fmt)
    assert x.is_cuda and x.is_contiguous() and x.dim() == 2, "x must be a contiguous 2-D CUDA tensor"
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("x must be bfloat16 or float32")
    rows, cols = x.shape
    flags = f | (FLAG_SRC_F32 if x.dtype == torch.float32 else 0) | (FLAG_STOCHASTIC if stochastic else 0)
    qr, qc = out if out is not None else (empty_qtensor(f, rows, cols, x.device), empty_qtensor(f, cols, rows, x.device))
    g = qr.global_scale
    if global_scale is not None:
        flags |= FLAG_GLOBAL_GIVEN
        g = global_scale
    rc = bsq_quantize_dual(flags, x, rows, cols, seed, qr.codes, qr.scales, qc.codes, qc.scales, g, stream)
    if rc != OK:
        raise BsqError(rc, "bsq_quantize_dual")
    if f == NVFP4:
        qr.global_scale = g
        qc.global_scale = g
    return qr, qc


def delayed_global_scale(prev: QTensor, headroom: float = 32.0, out: Optional[torch.Tensor] = None,
                         stream=None) -> torch.Tensor:
    """The next step's NVFP4 per-tensor scale from an earlier quantization `prev` of the tensor:
    fp32(fp32(amax * headroom) / 2688) on the device, as a one-element fp32 tensor to pass as
    `global_scale`."""
    assert prev.fmt == NVFP4
    g = out if out is not None else torch.empty(1, dtype=torch.float32, device=prev.scales.device)
    rc = bsq_delayed_global_scale(prev.scales, prev.rows, prev.cols, headroom, g, stream)
    if rc != OK:
        raise BsqError(rc, "bsq_delayed_global_scale")
    return g


def gemm(qa: QTensor, qb: QTensor, bias: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
         stream=None) -> torch.Tensor:
    """out[M, N] = bf16(alpha * A_hat . B_hat^T + bias), A: M x K, B: N x K (weight layout)."""
    assert qa.fmt == qb.fmt and qa.cols == qb.cols
    M, K, N = qa.rows, qa.cols, qb.rows
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=qa.codes.device)
    if bias is not None:
        assert bias.dtype == torch.bfloat16 and bias.numel() == N and bias.is_contiguous()
    rc = bsq_gemm(qa.fmt, qa.codes, qa.scales, qb.codes, qb.scales, bias, out, M, N, K, stream)
    if rc != OK:
        raise BsqError(rc, "bsq_gemm")
    return out


def gemm_splitk(qa: QTensor, qb: QTensor, bias: Optional[torch.Tensor] = None, splits: Optional[int] = None,
                workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    """gemm() with K cut into `splits` ranges (default: the library's choice for the shape), the
    fp32 partial sums in `workspace` (splits x M x N fp32; allocated here when not given)."""
    assert qa.fmt == qb.fmt and qa.cols == qb.cols
    M, K, N = qa.rows, qa.cols, qb.rows
    if splits is None:
        splits = bsq_gemm_splitk_splits(qa.fmt, M, N, K)
        if splits < 0:
            raise BsqError(splits, "bsq_gemm_splitk_splits")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=qa.codes.device)
    if bias is not None:
        assert bias.dtype == torch.bfloat16 and bias.numel() == N and bias.is_contiguous()
    if workspace is None and splits > 1:
        workspace = torch.empty(splits * M * N, dtype=torch.float32, device=qa.codes.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = bsq_gemm_splitk(qa.fmt, qa.codes, qa.scales, qb.codes, qb.scales, bias, out, M, N, K, splits, workspace,
                         ws_bytes, stream)
    if rc != OK:
        raise BsqError(rc, "bsq_gemm_splitk")
    return out


def gemm_gelu(qa: QTensor, qb: QTensor, bias: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
              stream=None) -> torch.Tensor:
    """out[M, N] = bf16(GELU(alpha * A_hat . B_hat^T + bias)), GELU in its erf form."""
    assert qa.fmt == qb.fmt and qa.cols == qb.cols
    M, K, N = qa.rows, qa.cols, qb.rows
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=qa.codes.device)
    rc = bsq_gemm_gelu(qa.fmt, qa.codes, qa.scales, qb.codes, qb.scales, bias, out, M, N, K, stream)
    if rc != OK:
        raise BsqError(rc, "bsq_gemm_gelu")
    return out


def gemm_gelu_quantize(qa: QTensor, qb: QTensor, bias: Optional[torch.Tensor] = None, out_fmt="mxfp8",
                       out: Optional[QTensor] = None, stream=None) -> QTensor:
    """GELU(alpha * A_hat . B_hat^T + bias) quantized along N into out_fmt (MXFP8 / MXFP4) in the
    GEMM's epilogue: an M x N operand, laid out as quantize() lays it out."""
    assert qa.fmt == qb.fmt and qa.cols == qb.cols
    M, K, N = qa.rows, qa.cols, qb.rows
    of = _fmt(out_fmt)
    q = out if out is not None else empty_qtensor(of, M, N, qa.codes.device)
    rc = bsq_gemm_gelu_quantize(qa.fmt, qa.codes, qa.scales, qb.codes, qb.scales, bias, of, q.codes, q.scales,
                                M, N, K, stream)
    if rc != OK:
        raise BsqError(rc, "bsq_gemm_gelu_quantize")
    return q


def linear(fmt, x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The whole block-scaled linear layer: quantize x and w along K, then the GEMM."""
    return gemm(quantize(fmt, x, stream=stream), quantize(fmt, w, stream=stream), bias, stream=stream)


def linear_backward(dy: torch.Tensor, x_col: QTensor, w_col: QTensor, stochastic: bool = False, seed: int = 0,
                    stream=None):
    """The two backward GEMMs of a block-scaled linear layer: dY (M x N, bf16 / fp32) is
    quantized in both layouts in one pass, then dX = dY . W (dY row-wise against W column-wise,
    M x K) and dW = dY^T . X (dY column-wise against X column-wise, N x K), both bf16 with fp32
    accumulation. x_col / w_col are the column-wise operands of X (M x K) and W (N x K) from
    quantize_dual (K x M and K x N). dW (few output tiles, K = the token count) goes through
    gemm_splitk with the library's split count. Returns (dX, dW)."""
    dy_row, dy_col = quantize_dual(x_col.fmt, dy, stochastic=stochastic, seed=seed, stream=stream)
    return gemm(dy_row, w_col, stream=stream), gemm_splitk(dy_col, x_col, stream=stream)


def convt2x2(qx: QTensor, qw: QTensor, batch: int, H: int, W: int, bias: Optional[torch.Tensor] = None,
             gelu: bool = False, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Kernel-2 stride-2 transposed convolution of a quantized NHWC input (batch*H*W x C_in) with a
    quantized 4*C_out x C_in weight (row (2 dy + dx) C_out + co): batch x 2H x 2W x C_out bf16."""
    assert qx.fmt == qw.fmt and qx.cols == qw.cols and qx.rows == batch * H * W and qw.rows % 4 == 0
    C_in, C_out = qx.cols, qw.rows // 4
    if out is None:
        out = torch.empty((batch, 2 * H, 2 * W, C_out), dtype=torch.bfloat16, device=qx.codes.device)
    rc = bsq_convt2x2(qx.fmt, qx.codes, qx.scales, qw.codes, qw.scales, bias, out, batch, H, W, C_in, C_out, gelu,
                      stream)
    if rc != OK:
        raise BsqError(rc, "bsq_convt2x2")
    return out


def device_status(stream=None) -> int:
    return bsq_get_device_status(stream)
