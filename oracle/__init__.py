"""CPU oracle for the block-scaled quantize + GEMM path (ctypes over bsq_oracle.c).

TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU-baseline
leg import this package. The product library never does, and nothing here is shared with
the CUDA path: the two meet only through the seeded inputs of ``workloads``.

The C source states the readings it takes where the pages are silent (rounding, the
UE8M0 exponent rule, NVFP4 arithmetic order, nibble order, scale layout).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsq_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

MXFP8, NVFP4, MXFP4 = 1, 2, 3
FMT_IDS = {"mxfp8": MXFP8, "nvfp4": NVFP4, "mxfp4": MXFP4}

_lib: Optional[ctypes.CDLL] = None


def build(force: bool = False) -> str:
    """Compile bsq_oracle.c into liboracle.so next to it (gcc, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i64, u8p, f64p, vp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
        L.orc_decode_e4m3.restype = ctypes.c_double
        L.orc_decode_e4m3.argtypes = [ctypes.c_uint]
        L.orc_decode_e2m1.restype = ctypes.c_double
        L.orc_decode_e2m1.argtypes = [ctypes.c_uint]
        L.orc_decode_ue8m0.restype = ctypes.c_double
        L.orc_decode_ue8m0.argtypes = [ctypes.c_uint]
        L.orc_encode_e4m3.restype = ctypes.c_uint
        L.orc_encode_e4m3.argtypes = [ctypes.c_double]
        L.orc_encode_e2m1.restype = ctypes.c_uint
        L.orc_encode_e2m1.argtypes = [ctypes.c_double]
        L.orc_scale_tiled_offset.restype = i64
        L.orc_scale_tiled_offset.argtypes = [i64, i64, i64]
        L.orc_scales_tiled_bytes.restype = i64
        L.orc_scales_tiled_bytes.argtypes = [ctypes.c_int, i64, i64]
        L.orc_codes_bytes.restype = i64
        L.orc_codes_bytes.argtypes = [ctypes.c_int, i64, i64]
        L.orc_tile_scales.restype = ctypes.c_int
        L.orc_tile_scales.argtypes = [ctypes.c_int, u8p, i64, i64, ctypes.c_float, ctypes.c_float, u8p]
        L.orc_quantize_mx.restype = ctypes.c_int
        L.orc_quantize_mx.argtypes = [ctypes.c_int, vp, ctypes.c_int, i64, i64, u8p, u8p]
        L.orc_quantize_nvfp4.restype = ctypes.c_int
        L.orc_quantize_nvfp4.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_int, ctypes.c_float,
                                         u8p, u8p, vp, vp]
        L.orc_tensor_amax.restype = ctypes.c_float
        L.orc_tensor_amax.argtypes = [vp, ctypes.c_int, i64]
        L.orc_decode.restype = ctypes.c_int
        L.orc_decode.argtypes = [ctypes.c_int, u8p, u8p, i64, i64, f64p]
        L.orc_gemm.restype = ctypes.c_int
        L.orc_gemm.argtypes = [f64p, f64p, vp, i64, i64, i64, ctypes.c_double, i64, i64, f64p, vp]
        L.orc_gelu_erf.restype = ctypes.c_int
        L.orc_gelu_erf.argtypes = [f64p, f64p, i64]
        L.orc_quantize_mx_f64.restype = ctypes.c_int
        L.orc_quantize_mx_f64.argtypes = [ctypes.c_int, f64p, i64, i64, u8p, u8p]
        L.orc_encode_array.restype = ctypes.c_int
        L.orc_encode_array.argtypes = [ctypes.c_int, f64p, i64, u8p]
        L.orc_layernorm.restype = ctypes.c_int
        L.orc_layernorm.argtypes = [vp, ctypes.c_int, vp, vp, ctypes.c_double, i64, i64, f64p]
        L.orc_philox4x32_10.restype = None
        L.orc_philox4x32_10.argtypes = [vp, vp, vp]
        L.orc_encode_sr_array.restype = ctypes.c_int
        L.orc_encode_sr_array.argtypes = [ctypes.c_int, f64p, f64p, i64, u8p]
        L.orc_quantize_mx_dual.restype = ctypes.c_int
        L.orc_quantize_mx_dual.argtypes = [ctypes.c_int, vp, ctypes.c_int, i64, i64, ctypes.c_int, ctypes.c_uint64,
                                           u8p, u8p, u8p, u8p]
        L.orc_num_threads.restype = ctypes.c_int
        L.orc_quantize_nv_dual.restype = ctypes.c_int
        L.orc_quantize_nv_dual.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                           ctypes.c_uint64, u8p, u8p, u8p, u8p, vp, vp]
        L.orc_delayed_global_scale.restype = ctypes.c_float
        L.orc_delayed_global_scale.argtypes = [ctypes.c_float, ctypes.c_float]
        L.orc_convt2x2.restype = ctypes.c_int
        L.orc_convt2x2.argtypes = [f64p, f64p, vp, i64, i64, i64, i64, i64, ctypes.c_double, ctypes.c_int, f64p]
        L.orc_set_num_threads.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _fmt(fmt) -> int:
    return FMT_IDS[fmt] if isinstance(fmt, str) else int(fmt)


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


# --- scalar codecs -------------------------------------------------------------------------
def decode_e4m3(c: int) -> float:
    return lib().orc_decode_e4m3(int(c))


def decode_e2m1(c: int) -> float:
    return lib().orc_decode_e2m1(int(c))


def decode_ue8m0(c: int) -> float:
    return lib().orc_decode_ue8m0(int(c))


def encode_e4m3(v: float) -> int:
    return lib().orc_encode_e4m3(float(v))


def encode_e2m1(v: float) -> int:
    return lib().orc_encode_e2m1(float(v))


# --- layout --------------------------------------------------------------------------------
def codes_bytes(fmt, rows: int, cols: int) -> int:
    return int(lib().orc_codes_bytes(_fmt(fmt), rows, cols))


def scales_tiled_bytes(fmt, rows: int, cols: int) -> int:
    return int(lib().orc_scales_tiled_bytes(_fmt(fmt), rows, cols))


def scale_tiled_offset(r: int, c: int, n_scale_cols: int) -> int:
    return int(lib().orc_scale_tiled_offset(r, c, n_scale_cols))


def block_size(fmt) -> int:
    return 16 if _fmt(fmt) == NVFP4 else 32


def tile_scales(fmt, plain: np.ndarray, rows: int, cols: int, g: float = 0.0, amax: float = 0.0) -> np.ndarray:
    plain = np.ascontiguousarray(plain, dtype=np.uint8)
    out = np.empty(scales_tiled_bytes(fmt, rows, cols), dtype=np.uint8)
    st = lib().orc_tile_scales(_fmt(fmt), _ptr(plain), rows, cols, g, amax, _ptr(out))
    assert st == 0, st
    return out


# --- quantizers ----------------------------------------------------------------------------
class Quantized:
    """codes (uint8, packed), plain scales (rows x cols/bs), per-tensor g and amax (NVFP4)."""

    def __init__(self, fmt: int, rows: int, cols: int, codes: np.ndarray, scales: np.ndarray,
                 g: float = 1.0, amax: float = 0.0):
        self.fmt, self.rows, self.cols = fmt, rows, cols
        self.codes, self.scales, self.g, self.amax = codes, scales, g, amax

    def tiled_scales(self) -> np.ndarray:
        return tile_scales(self.fmt, self.scales, self.rows, self.cols, self.g if self.fmt == NVFP4 else 0.0,
                           self.amax if self.fmt == NVFP4 else 0.0)

    def decode(self) -> np.ndarray:
        return decode(self.fmt, self.codes, self.scales, self.rows, self.cols)


def _src(x: np.ndarray) -> Tuple[np.ndarray, int]:
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, 1
    assert x.dtype == np.uint16, "sources are fp32 values or bf16 bit patterns (uint16)"
    return x, 0


def quantize(fmt, x: np.ndarray, global_scale: Optional[float] = None) -> Quantized:
    f = _fmt(fmt)
    x, is_f32 = _src(x)
    rows, cols = x.shape
    codes = np.zeros(codes_bytes(f, rows, cols), dtype=np.uint8)
    bs = block_size(f)
    scales = np.zeros((rows, cols // bs), dtype=np.uint8)
    L = lib()
    if f == NVFP4:
        g = np.zeros(1, np.float32)
        amax = np.zeros(1, np.float32)
        st = L.orc_quantize_nvfp4(_ptr(x), is_f32, rows, cols, 0 if global_scale is None else 1,
                                  0.0 if global_scale is None else float(global_scale),
                                  _ptr(codes), _ptr(scales), _ptr(g), _ptr(amax))
        if st:
            raise ValueError("oracle quantize failed: %d" % st)
        return Quantized(f, rows, cols, codes, scales, float(g[0]), float(amax[0]))
    st = L.orc_quantize_mx(f, _ptr(x), is_f32, rows, cols, _ptr(codes), _ptr(scales))
    if st:
        raise ValueError("oracle quantize failed: %d" % st)
    return Quantized(f, rows, cols, codes, scales)


def tensor_amax(x: np.ndarray) -> float:
    x, is_f32 = _src(x)
    return float(lib().orc_tensor_amax(_ptr(x), is_f32, x.size))


def decode(fmt, codes: np.ndarray, scales: np.ndarray, rows: int, cols: int) -> np.ndarray:
    f = _fmt(fmt)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.empty((rows, cols), dtype=np.float64)
    st = lib().orc_decode(f, _ptr(codes), _ptr(scales), rows, cols, _ptr(out))
    assert st == 0, st
    return out


def gemm(A: np.ndarray, B: np.ndarray, bias: Optional[np.ndarray] = None, alpha: float = 1.0,
         rows: Optional[Tuple[int, int]] = None, want_abs: bool = True):
    """fp64 out = alpha * A . B^T + bias for output rows [r0, r1); returns (out, abs_sum)."""
    A = np.ascontiguousarray(A, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    r0, r1 = (0, M) if rows is None else rows
    out = np.empty((r1 - r0, N), dtype=np.float64)
    ab = np.empty((r1 - r0, N), dtype=np.float64) if want_abs else None
    bias_arr = None if bias is None else np.ascontiguousarray(bias, dtype=np.uint16)
    st = lib().orc_gemm(_ptr(A), _ptr(B), _ptr(bias_arr), M, N, K, float(alpha), r0, r1, _ptr(out), _ptr(ab))
    assert st == 0, st
    return out, ab


def reference_linear(fmt, a_src: np.ndarray, b_src: np.ndarray, bias: Optional[np.ndarray] = None,
                     rows: Optional[Tuple[int, int]] = None):
    """The whole path on the CPU: quantize A and B, decode, fp64 GEMM (+ alpha for NVFP4)."""
    qa = quantize(fmt, a_src)
    qb = quantize(fmt, b_src)
    alpha = qa.g * qb.g if qa.fmt == NVFP4 else 1.0
    out, ab = gemm(qa.decode(), qb.decode(), bias, alpha, rows)
    return qa, qb, out, ab


def gelu_erf(v: np.ndarray) -> np.ndarray:
    """Exact-erf GELU in fp64 (reading R8)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty_like(v)
    st = lib().orc_gelu_erf(_ptr(v), _ptr(out), v.size)
    if st:
        raise ValueError("oracle gelu failed: %d" % st)
    return out


def quantize_mx_f64(fmt, y: np.ndarray) -> Quantized:
    """MX quantization (rule R2) of fp64 values y (rows x cols)."""
    f = _fmt(fmt)
    assert f in (MXFP8, MXFP4)
    y = np.ascontiguousarray(y, dtype=np.float64)
    rows, cols = y.shape
    codes = np.zeros(codes_bytes(f, rows, cols), dtype=np.uint8)
    scales = np.zeros((rows, cols // 32), dtype=np.uint8)
    st = lib().orc_quantize_mx_f64(f, _ptr(y), rows, cols, _ptr(codes), _ptr(scales))
    if st:
        raise ValueError("oracle quantize failed: %d" % st)
    return Quantized(f, rows, cols, codes, scales)


def encode_array(elem: str, v: np.ndarray) -> np.ndarray:
    """Element codes (one per byte) of fp64 values: elem 'e4m3' or 'e2m1' (rule R1)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    st = lib().orc_encode_array(0 if elem == "e4m3" else 1, _ptr(v), v.size, _ptr(out))
    if st:
        raise ValueError("oracle encode failed: %d" % st)
    return out


def gelu_quantize_reference(fmt, y: np.ndarray) -> Quantized:
    """The fused fc1 step of reading R8 on the unrounded GEMM values y: MX(GELU(y))."""
    return quantize_mx_f64(fmt, gelu_erf(y))


def layernorm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float) -> np.ndarray:
    """Row LayerNorm in fp64 (reading R9): x bf16 bits (uint16) or fp32; gamma, beta bf16 bits."""
    x, is_f32 = _src(x)
    rows, cols = x.shape
    gamma = np.ascontiguousarray(gamma, dtype=np.uint16)
    beta = np.ascontiguousarray(beta, dtype=np.uint16)
    out = np.empty((rows, cols), dtype=np.float64)
    st = lib().orc_layernorm(_ptr(x), is_f32, _ptr(gamma), _ptr(beta), float(eps), rows, cols, _ptr(out))
    if st:
        raise ValueError("oracle layernorm failed: %d" % st)
    return out


def layernorm_quantize_reference(fmt, x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float) -> Quantized:
    """The fused LN step of reading R9: MX(LayerNorm(x))."""
    return quantize_mx_f64(fmt, layernorm(x, gamma, beta, eps))


def philox4x32_10(counter, key) -> Tuple[int, int, int, int]:
    """Philox4x32-10 of a 4 x 32-bit counter and a 2 x 32-bit key (reading R10)."""
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return tuple(int(v) for v in out)


def encode_sr_array(elem: str, v: np.ndarray, u: np.ndarray) -> np.ndarray:
    """Stochastically rounded element codes (reading R10): up iff frac(|v| / spacing) > u."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    u = np.ascontiguousarray(u, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    st = lib().orc_encode_sr_array(0 if elem == "e4m3" else 1, _ptr(v), _ptr(u), v.size, _ptr(out))
    if st:
        raise ValueError("oracle encode failed: %d" % st)
    return out


def quantize_dual(fmt, x: np.ndarray, stochastic: bool = False, seed: int = 0,
                  global_scale: Optional[float] = None) -> Tuple[Quantized, Quantized]:
    """Dual-layout quantization (readings R10, R11): (row-wise R x C, column-wise C x R). NVFP4
    shares one per-tensor scale between the layouts (computed, or `global_scale`)."""
    f = _fmt(fmt)
    x, is_f32 = _src(x)
    R, C = x.shape
    bs = block_size(f)
    rc = np.zeros(codes_bytes(f, R, C), dtype=np.uint8)
    rs = np.zeros((R, C // bs), dtype=np.uint8)
    cc = np.zeros(codes_bytes(f, C, R), dtype=np.uint8)
    cs = np.zeros((C, R // bs), dtype=np.uint8)
    seed = int(seed) & (2 ** 64 - 1)
    if f == NVFP4:
        g = np.zeros(1, np.float32)
        amax = np.zeros(1, np.float32)
        st = lib().orc_quantize_nv_dual(_ptr(x), is_f32, R, C, 0 if global_scale is None else 1,
                                        0.0 if global_scale is None else float(global_scale),
                                        1 if stochastic else 0, seed, _ptr(rc), _ptr(rs), _ptr(cc), _ptr(cs),
                                        _ptr(g), _ptr(amax))
        if st:
            raise ValueError("oracle dual quantize failed: %d" % st)
        return (Quantized(f, R, C, rc, rs, float(g[0]), float(amax[0])),
                Quantized(f, C, R, cc, cs, float(g[0]), float(amax[0])))
    assert global_scale is None
    st = lib().orc_quantize_mx_dual(f, _ptr(x), is_f32, R, C, 1 if stochastic else 0, seed,
                                    _ptr(rc), _ptr(rs), _ptr(cc), _ptr(cs))
    if st:
        raise ValueError("oracle dual quantize failed: %d" % st)
    return Quantized(f, R, C, rc, rs), Quantized(f, C, R, cc, cs)


def delayed_global_scale(amax_prev: float, headroom: float) -> float:
    """Delayed per-tensor NVFP4 scale (reading R12): fp32(fp32(amax_prev * headroom) / 2688)."""
    return float(lib().orc_delayed_global_scale(float(amax_prev), float(headroom)))


def convt2x2(A: np.ndarray, B: np.ndarray, bias: Optional[np.ndarray], batch: int, H: int, W: int,
             alpha: float = 1.0, gelu: bool = False) -> np.ndarray:
    """Transposed convolution, kernel 2, stride 2 (reading R13) from decoded fp64 operands:
    A (batch*H*W) x Cin, B (4*Cout) x Cin (row (2 dy + dx) Cout + co), bias Cout bf16 bits or
    None; returns batch x 2H x 2W x Cout fp64 (NHWC)."""
    A = np.ascontiguousarray(A, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    Cin = A.shape[1]
    Cout = B.shape[0] // 4
    assert A.shape[0] == batch * H * W and B.shape == (4 * Cout, Cin)
    bias_arr = None if bias is None else np.ascontiguousarray(bias, dtype=np.uint16)
    out = np.empty((batch, 2 * H, 2 * W, Cout), dtype=np.float64)
    st = lib().orc_convt2x2(_ptr(A), _ptr(B), _ptr(bias_arr), batch, H, W, Cin, Cout, float(alpha),
                            1 if gelu else 0, _ptr(out))
    assert st == 0, st
    return out
