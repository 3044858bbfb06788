"""GPU parity of the fused LayerNorm + MX quantization kernel against the oracle's reading R9.

The kernel quantizes its fp32 LayerNorm output; the oracle's is exact (fp64). A code is
accepted when it is the encoding of some value inside an error band around the exact output:
the fp32 rounding of the row mean (each lane adds cols/32 values in sequence, then 5 butterfly
levels: at most (cols/32 + 8) * 2^-24 * mean|x|), of rstd (2^-17 relative) and of the affine
step (2^-22 of |t gamma| + |beta|). At least 99 % of codes and scales must equal those
of the exact values."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import check_mx_band, element_codes, plain_scales, to_dev
from workloads import bf16_bits_to_f32, f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def _bsq():
    import block_scaled_precision_bsq_gb300 as bsq

    return bsq


def _inputs(rows, cols, seed, f32=False):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)) * 3 + 1
    x[:, rng.choice(cols, max(1, cols // 200), replace=False)] *= 20  # outlier channels
    x = x.astype(np.float32)
    if not f32:
        x = f32_to_bf16_bits(x)
    g = f32_to_bf16_bits((1 + 0.1 * rng.standard_normal(cols)).astype(np.float32))
    b = f32_to_bf16_bits((0.1 * rng.standard_normal(cols)).astype(np.float32))
    return x, g, b


def _band(x, g, b, eps, exact):
    xv = (bf16_bits_to_f32(x) if x.dtype == np.uint16 else x).astype(np.float64)
    gv, bv = bf16_bits_to_f32(g).astype(np.float64), bf16_bits_to_f32(b).astype(np.float64)
    mean = xv.mean(axis=1, keepdims=True)
    rstd = 1.0 / np.sqrt(xv.var(axis=1, keepdims=True) + eps)
    t = (xv - mean) * rstd
    err_mean = (xv.shape[1] / 32 + 8) * 2.0 ** -24 * np.abs(xv).mean(axis=1, keepdims=True)
    return np.abs(gv) * (err_mean * rstd + np.abs(t) * 2.0 ** -17) + 2.0 ** -22 * (np.abs(t * gv) + np.abs(bv)) + 1e-30


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("rows,cols", [(300, 768), (128, 1024), (7, 4096), (1, 32), (257, 96)])
def test_layernorm_quantize(fmt, rows, cols):
    bsq = _bsq()
    x, g, b = _inputs(rows, cols, seed=90 + rows)
    eps = 1e-6
    q = bsq.layernorm_quantize(fmt, to_dev(x), to_dev(g), to_dev(b), eps)
    assert bsq.device_status() == 0
    exact = oracle.layernorm(x, g, b, eps)
    tiled = q.scales.cpu().numpy()
    plain = plain_scales(tiled, rows, cols)
    assert np.array_equal(tiled, oracle.tile_scales(fmt, plain, rows, cols))  # layout and zero padding
    check_mx_band(fmt, element_codes(fmt, q.codes.cpu().numpy(), rows, cols), plain, exact,
                  _band(x, g, b, eps, exact))


def test_layernorm_quantize_fp32_source():
    bsq = _bsq()
    x, g, b = _inputs(200, 1024, seed=95, f32=True)
    q = bsq.layernorm_quantize("mxfp8", to_dev(x), to_dev(g), to_dev(b), 1e-5)
    assert bsq.device_status() == 0
    exact = oracle.layernorm(x, g, b, 1e-5)
    plain = plain_scales(q.scales.cpu().numpy(), 200, 1024)
    check_mx_band("mxfp8", element_codes("mxfp8", q.codes.cpu().numpy(), 200, 1024), plain, exact,
                  _band(x, g, b, 1e-5, exact))


@pytest.mark.parametrize("fmt,rows", [("mxfp8", 7168), ("mxfp4", 51200)])
def test_layernorm_quantize_full_size_sampled_rows(fmt, rows):
    """ViT-L LN before fc1 at its full sizes (M = 7168 MXFP8 and M = 51200 MXFP4, 1024 channels:
    the streaming kernel, ten rows per warp at 51200), sampled rows."""
    bsq = _bsq()
    cols = 1024
    x, g, b = _inputs(rows, cols, seed=97)
    q = bsq.layernorm_quantize(fmt, to_dev(x), to_dev(g), to_dev(b), 1e-6)
    assert bsq.device_status() == 0
    idx = np.unique(np.concatenate([np.arange(0, rows, 128), np.arange(127, rows, 128),
                                    np.random.default_rng(1).integers(0, rows, 64)]))
    exact = oracle.layernorm(x[idx], g, b, 1e-6)
    codes = element_codes(fmt, q.codes.cpu().numpy(), rows, cols)[idx]
    plain = plain_scales(q.scales.cpu().numpy(), rows, cols, row_idx=idx)
    check_mx_band(fmt, codes, plain, exact, _band(x[idx], g, b, 1e-6, exact))


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("rows,cols", [(300, 768), (129, 1024), (33, 96)])
def test_streaming_and_shared_memory_kernels_agree(fmt, rows, cols):
    """bf16 rows of at most 1024 elements take the streaming kernel, fp32 rows the shared-memory
    kernel; both run the same row statistics and affine arithmetic, so the same values (a bf16
    matrix and its exact fp32 copy) give the same bytes."""
    bsq = _bsq()
    x, g, b = _inputs(rows, cols, seed=120 + cols)
    xd = to_dev(x)
    q16 = bsq.layernorm_quantize(fmt, xd, to_dev(g), to_dev(b), 1e-6)
    q32 = bsq.layernorm_quantize(fmt, xd.float(), to_dev(g), to_dev(b), 1e-6)
    assert bsq.device_status() == 0
    assert torch.equal(q16.codes, q32.codes)
    assert torch.equal(q16.scales, q32.scales)
