"""GPU parity of the head's kernel-2 stride-2 transposed convolution (a block-scaled GEMM whose
epilogue stores each output column at its output pixel, optionally after GELU) against the
oracle's transposed convolution by definition on the same quantized operands: every output
pixel within |gpu - y| <= 2^-7 |y| + 1e-5 sum |a b| (bf16 output of an fp32-accumulated GEMM),
plus the GELU evaluation error where GELU is fused."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import to_dev
from workloads import f32_to_bf16_bits, random_matrix

pytestmark = pytest.mark.gpu


def _bsq():
    import block_scaled_precision_bsq_gb300 as bsq

    return bsq


def _run(fmt, batch, H, W, C_in, C_out, gelu, seed):
    bsq = _bsq()
    x = random_matrix(batch * H * W, C_in, seed=seed, dist="normal")
    w = random_matrix(4 * C_out, C_in, seed=seed + 1, std=0.05)
    rng = np.random.default_rng(seed + 2)
    bias = f32_to_bf16_bits((rng.standard_normal(C_out) * 0.1).astype(np.float32))
    qx, qw = bsq.quantize(fmt, to_dev(x)), bsq.quantize(fmt, to_dev(w))
    out = bsq.convt2x2(qx, qw, batch, H, W, bias=to_dev(bias), gelu=gelu)
    torch.cuda.synchronize()
    assert bsq.device_status() == 0
    ox, ow = oracle.quantize(fmt, x), oracle.quantize(fmt, w)
    A, B = ox.decode(), ow.decode()
    alpha = ox.g * ow.g if fmt == "nvfp4" else 1.0
    y = oracle.convt2x2(A, B, bias, batch, H, W, alpha=alpha)             # pre-activation
    absum = oracle.convt2x2(np.abs(A), np.abs(B), None, batch, H, W, alpha=abs(alpha))
    got = out.float().cpu().numpy().astype(np.float64)
    assert got.shape == (batch, 2 * H, 2 * W, C_out)
    if gelu:
        G = oracle.convt2x2(A, B, bias, batch, H, W, alpha=alpha, gelu=True)
        tol = 2.0 ** -7 * np.abs(G) + 1.13 * 1e-5 * absum + 4e-7 * np.abs(y) + 1e-30
        want = G
    else:
        tol = 2.0 ** -7 * np.abs(y) + 1e-5 * absum + 1e-30
        want = y
    bad = np.abs(got - want) > tol
    assert not bad.any(), "%d of %d outputs out of tolerance, first at %s" % (
        int(bad.sum()), bad.size, np.unravel_index(int(np.argmax(bad)), bad.shape))


# W divides 32 (whole image rows per 32-token chunk) or 32 divides W (part of one row); ragged
# token counts (batch H W not a multiple of 32 or 128) and C_out not a multiple of the 256-column tile
SHAPES = [(2, 8, 8, 64), (1, 4, 64, 96), (3, 5, 32, 256), (1, 3, 4, 32), (2, 2, 1, 64)]


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("batch,H,W,C_out", SHAPES)
@pytest.mark.parametrize("gelu", [False, True])
def test_convt_matches_oracle(fmt, batch, H, W, C_out, gelu):
    C_in = 128 if fmt == "mxfp8" else 256
    _run(fmt, batch, H, W, C_in, C_out, gelu, seed=batch * 1000 + H * 100 + W + C_out)


def test_convt_head_shapes_vitl():
    """ConvT1 of a ViT-L/16 head on a 512 x 512 frame: the 32 x 32 patch grid, 1024 channels in
    and out, GELU fused; every output pixel checked."""
    _run("mxfp8", 1, 32, 32, 1024, 1024, True, seed=5)
