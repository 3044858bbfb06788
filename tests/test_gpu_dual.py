"""GPU parity of the dual-layout MX quantizer (row-wise operand plus the transposed column-wise
operand from one read, round-to-nearest-even or Philox4x32-10 stochastic rounding) against the
CPU oracle: codes and tiled scales of both layouts bit-identical, padding included."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import to_dev
from workloads import f32_to_bf16_bits, random_matrix

pytestmark = pytest.mark.gpu

# several 128 x 128 tiles, ragged row and column tails (R or C = 32 mod 128), the smallest shape
SHAPES = [(32, 32), (96, 160), (128, 128), (160, 288), (256, 384), (544, 800)]


def _bsq():
    import block_scaled_precision_bsq_gb300 as bsq

    return bsq


def _check(fmt, x_np, stochastic, seed, label, global_scale=None):
    bsq = _bsq()
    qr_o, qc_o = oracle.quantize_dual(fmt, x_np, stochastic=stochastic, seed=seed, global_scale=global_scale)
    gs = None if global_scale is None else torch.tensor([global_scale], dtype=torch.float32, device="cuda")
    qr, qc = bsq.quantize_dual(fmt, to_dev(x_np), stochastic=stochastic, seed=seed, global_scale=gs)
    assert bsq.device_status() == 0
    for name, got, want in (("row", qr, qr_o), ("col", qc, qc_o)):
        codes = got.codes.cpu().numpy()
        assert np.array_equal(codes, want.codes), "%s %s codes: %d of %d bytes differ (first at %d)" % (
            label, name, int((codes != want.codes).sum()), codes.size, int(np.argmax(codes != want.codes)))
        scales = got.scales.cpu().numpy()
        ws = want.tiled_scales()
        assert np.array_equal(scales, ws), "%s %s scales: %d bytes differ (first at %d)" % (
            label, name, int((scales != ws).sum()), int(np.argmax(scales != ws)))
    return qr, qc


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "nvfp4"])
@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("stochastic", [False, True])
def test_dual_bf16_matches_oracle(fmt, rows, cols, stochastic):
    x = random_matrix(rows, cols, seed=rows * 3 + cols, dist="student_t4")
    _check(fmt, x, stochastic, seed=rows * 1000 + cols, label="%s %dx%d sr=%d" % (fmt, rows, cols, stochastic))


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "nvfp4"])
@pytest.mark.parametrize("rows,cols", [(32, 64), (96, 160), (192, 416)])
@pytest.mark.parametrize("stochastic", [False, True])
def test_dual_fp32_matches_oracle(fmt, rows, cols, stochastic):
    x = random_matrix(rows, cols, seed=rows + cols, dist="uniform_exp", src_f32=True)
    _check(fmt, x, stochastic, seed=7, label="%s f32 %dx%d sr=%d" % (fmt, rows, cols, stochastic))


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "nvfp4"])
@pytest.mark.parametrize("src_f32", [False, True])
def test_dual_special_values(fmt, src_f32):
    """Zeros of both signs, all-zero blocks, exact grid points, values at and past saturation,
    subnormal sources and blocks spanning many binades."""
    rng = np.random.default_rng(11)
    R, C = 160, 192
    x = rng.standard_normal((R, C))
    x[:32, :32] = 0.0
    x[32:64, :32] = -0.0
    x[:, 32:64] = np.array([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -6.0])[rng.integers(0, 8, size=(R, 32))]
    x[:, 64:96] *= 2.0 ** rng.integers(-40, 40, size=(R, 32))
    x[64:96, 96:128] = 448.0 * rng.choice([-1.0, 1.0], size=(32, 32))
    x[96:128, :] *= 1e-39 if src_f32 else 1e-40          # subnormal sources
    x[128:160, 128:160] = np.ldexp(1.0, 100) * rng.standard_normal((32, 32))
    x[5, 130] = -0.0
    # one huge element per block, the rest 2^-40 smaller: codes far below the element format's
    # subnormal spacing (stochastic rounding then steps up only when u is 0)
    x[0:64, 160:192] = rng.standard_normal((64, 32)) * 2.0 ** -20
    x[0, 160:192] = 2.0 ** 20
    x[32:64, 160] = -(2.0 ** 20)
    data = x.astype(np.float32) if src_f32 else f32_to_bf16_bits(x.astype(np.float32))
    for sr in (False, True):
        _check(fmt, data, sr, seed=3, label="%s special f32=%d sr=%d" % (fmt, src_f32, sr))


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "nvfp4"])
def test_dual_rne_equals_two_quantizer_calls(fmt):
    """Without stochastic rounding the two layouts are exactly bsq_quantize of X and of X^T
    (NVFP4: both with the tensor's own per-tensor scale, which X and X^T share)."""
    bsq = _bsq()
    x = to_dev(random_matrix(288, 416, seed=1, dist="normal"))
    qr, qc = bsq.quantize_dual(fmt, x)
    a = bsq.quantize(fmt, x)
    b = bsq.quantize(fmt, x.t().contiguous())
    assert torch.equal(qr.codes, a.codes) and torch.equal(qr.scales, a.scales)
    assert torch.equal(qc.codes, b.codes) and torch.equal(qc.scales, b.scales)


@pytest.mark.parametrize("stochastic", [False, True])
@pytest.mark.parametrize("g", [0.00123, 1.0, 0.0])
def test_dual_nvfp4_given_scale(stochastic, g):
    """A given per-tensor scale (the delayed scale of training): both layouts use it, and both
    tails record it with the tensor's own amax; g = 0 gives signed zero codes everywhere."""
    x = random_matrix(160, 288, seed=4, dist="student_t4")
    _check("nvfp4", x, stochastic, seed=9, label="nvfp4 given g=%g sr=%d" % (g, stochastic), global_scale=g)


def test_dual_seed_determines_the_codes():
    """The same seed gives the same bytes on every call; another seed moves some codes but never
    a scale (scales do not depend on the rounding)."""
    bsq = _bsq()
    x = to_dev(random_matrix(256, 256, seed=2, dist="normal"))
    r1, c1 = bsq.quantize_dual("mxfp8", x, stochastic=True, seed=42)
    r2, c2 = bsq.quantize_dual("mxfp8", x, stochastic=True, seed=42)
    r3, c3 = bsq.quantize_dual("mxfp8", x, stochastic=True, seed=43 + (1 << 40))
    assert torch.equal(r1.codes, r2.codes) and torch.equal(c1.codes, c2.codes)
    assert not torch.equal(r1.codes, r3.codes) and not torch.equal(c1.codes, c3.codes)
    assert torch.equal(r1.scales, r3.scales) and torch.equal(c1.scales, c3.scales)


@pytest.mark.parametrize("stochastic", [False, True])
def test_dual_full_size_vitb_fc1_grad(stochastic):
    """The ViT-B/16 fc1 output gradient at training shape (14336 x 3072), in the launch
    configuration the bench times, against the oracle in full."""
    x = random_matrix(14336, 3072, seed=21, std=1e-3)
    _check("mxfp8", x, stochastic, seed=5, label="dY 14336x3072 sr=%d" % stochastic)
