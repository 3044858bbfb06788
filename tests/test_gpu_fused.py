"""GPU parity of the fused fc1 epilogues against the oracle's reading R8: GELU -> bf16, and
GELU -> MX codes + tiled scales (the fc2 operand).

The kernel quantizes its fp32 value of GELU(v); the oracle's is exact. A code is accepted when
it is the encoding of some value inside an error band around the exact GELU(y) -- accumulation
(2^-16 |y| + the GEMM tolerance's sum term, times GELU's largest slope 1.13) plus the stated
error of the kernel's GELU (4e-7 |y| + 2^-20 |GELU|, Abramowitz & Stegun 7.1.26 in fp32) --
and the block scale when it is the MX exponent of some block maximum inside the band. On
top of that validity check, at least 99 % of codes and scales must equal those of the exact
value (only values within the band of a rounding boundary may differ)."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import (bf16_to_f64, check_gemm_rows, check_mx_band, decode_rows, element_codes, plain_scales,
                            sample_rows, to_dev)
from workloads import f32_to_bf16_bits, random_matrix

pytestmark = pytest.mark.gpu

def _bsq():
    import block_scaled_precision_bsq_gb300 as bsq

    return bsq


def _operands(fmt, M, N, K, seed):
    """fc1-like operands: v = A W^T + bias spread over [-4, 4] where GELU bends."""
    a = random_matrix(M, K, seed, dist="normal")
    w = random_matrix(N, K, seed + 1, std=1.0 / np.sqrt(K))
    rng = np.random.default_rng(seed + 2)
    bias = f32_to_bf16_bits((rng.standard_normal(N) * 0.5).astype(np.float32))
    qa, qw = oracle.quantize(fmt, a), oracle.quantize(fmt, w)
    return a, w, bias, qa, qw


def _gpu_operands(bsq, fmt, a, w, bias):
    return bsq.quantize(fmt, to_dev(a)), bsq.quantize(fmt, to_dev(w)), to_dev(bias)


def check_fused(out_fmt, codes_el, scales_plain, y, absum):
    G = oracle.gelu_erf(y)
    band = 1.13 * (2.0 ** -16 * np.abs(y) + 1e-5 * absum) + 4e-7 * np.abs(y) + 2.0 ** -20 * np.abs(G) + 1e-30
    return check_mx_band(out_fmt, codes_el, scales_plain, G, band)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
def test_gemm_gelu_bf16(fmt):
    bsq = _bsq()
    M, N, K = 300, 640, 512
    a, w, bias, qa, qw = _operands(fmt, M, N, K, seed=60)
    ga, gw, gb = _gpu_operands(bsq, fmt, a, w, bias)
    out = bsq.gemm_gelu(ga, gw, gb)
    assert bsq.device_status() == 0
    idx = np.arange(M)
    y, absum = oracle.gemm(decode_rows(qa, idx), qw.decode(), bias, qa.g * qw.g if fmt == "nvfp4" else 1.0)
    G = oracle.gelu_erf(y)
    got = bf16_to_f64(out)
    tol = 2.0 ** -7 * np.abs(G) + 1.13 * 1e-5 * absum + 4e-7 * np.abs(y) + 1e-30
    assert (np.abs(got - G) <= tol).all()


@pytest.mark.parametrize("fmt,out_fmt", [("mxfp8", "mxfp8"), ("mxfp8", "mxfp4"), ("nvfp4", "mxfp8"), ("mxfp4", "mxfp4")])
@pytest.mark.parametrize("M,N,K", [(300, 640, 512), (128, 288, 256), (1, 32, 256)])
def test_gemm_gelu_quantize(fmt, out_fmt, M, N, K):
    bsq = _bsq()
    a, w, bias, qa, qw = _operands(fmt, M, N, K, seed=61 + M)
    ga, gw, gb = _gpu_operands(bsq, fmt, a, w, bias)
    q = bsq.gemm_gelu_quantize(ga, gw, gb, out_fmt=out_fmt)
    assert bsq.device_status() == 0
    codes = q.codes.cpu().numpy()
    tiled = q.scales.cpu().numpy()
    plain = plain_scales(tiled, M, N)
    # layout: the tiled buffer is exactly the oracle's tiling of these scales (zero padding)
    assert np.array_equal(tiled, oracle.tile_scales(out_fmt, plain, M, N))
    idx = np.arange(M)
    y, absum = oracle.gemm(decode_rows(qa, idx), qw.decode(), bias, qa.g * qw.g if fmt == "nvfp4" else 1.0)
    check_fused(out_fmt, element_codes(out_fmt, codes, M, N), plain, y, absum)


@pytest.mark.parametrize("fmt,out_fmt", [("mxfp8", "mxfp8"), ("mxfp4", "mxfp4")])
def test_fused_output_feeds_fc2(fmt, out_fmt):
    """fc1 (fused GELU quantization) -> fc2 through bsq_gemm on the fused operand: fc2 must
    match the oracle's GEMM on the decoded fused operand (layout compatibility end to end)."""
    bsq = _bsq()
    M, N1, K, N2 = 300, 768, 512, 256
    a, w1, b1, qa, qw1 = _operands(fmt, M, N1, K, seed=70)
    ga, gw1, gb1 = _gpu_operands(bsq, fmt, a, w1, b1)
    h = bsq.gemm_gelu_quantize(ga, gw1, gb1, out_fmt=out_fmt)
    w2 = random_matrix(N2, N1, 72, std=1.0 / np.sqrt(N1))
    gw2 = bsq.quantize(out_fmt, to_dev(w2))
    out = bsq.gemm(h, gw2, None)
    assert bsq.device_status() == 0
    codes = h.codes.cpu().numpy()
    plain = plain_scales(h.scales.cpu().numpy(), M, N1)
    qh = oracle.Quantized(oracle._fmt(out_fmt), M, N1, codes, plain)
    idx = sample_rows(M)
    check_gemm_rows(bf16_to_f64(out)[idx], qh, oracle.quantize(out_fmt, w2), None, idx, "fc2 on fused fc1")


def test_fused_full_size_sampled_rows():
    """ViT-L fc1 at its full size (M=7168, K=1024 -> N=4096), MXFP8 in and out, on sampled rows."""
    bsq = _bsq()
    M, N, K = 7168, 4096, 1024
    a, w, bias, qa, qw = _operands("mxfp8", M, N, K, seed=80)
    ga, gw, gb = _gpu_operands(bsq, "mxfp8", a, w, bias)
    q = bsq.gemm_gelu_quantize(ga, gw, gb, out_fmt="mxfp8")
    assert bsq.device_status() == 0
    idx = sample_rows(M)
    codes = q.codes.cpu().numpy().reshape(M, N)[idx]
    tiled = q.scales.cpu().numpy()
    nsc = N // 32
    off = np.array([[oracle.scale_tiled_offset(int(r), c, nsc) for c in range(nsc)] for r in idx])
    y, absum = oracle.gemm(decode_rows(qa, idx), qw.decode(), bias, 1.0)
    check_fused("mxfp8", codes, tiled[off], y, absum)
