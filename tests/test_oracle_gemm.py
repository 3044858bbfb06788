"""Pins for the oracle's decode + fp64 GEMM: a library matmul on tiny non-square cases,
closed forms (identity and all-ones operands), and the whole path's error band."""
import numpy as np
import pytest

import oracle
from workloads import WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, make_activations, make_bias, \
    make_weights, random_matrix


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("M,N,K", [(32, 48, 64), (7, 40, 96), (64, 32, 128)])
def test_gemm_vs_numpy_matmul(fmt, M, N, K):
    a = random_matrix(M, K, seed=1, dist="student_t4")
    b = random_matrix(N, K, seed=2, std=0.02)
    bias = f32_to_bf16_bits(np.linspace(-1, 1, N).astype(np.float32))
    qa, qb, out, ab = oracle.reference_linear(fmt, a, b, bias)
    A, B = qa.decode(), qb.decode()
    alpha = qa.g * qb.g if fmt == "nvfp4" else 1.0
    want = alpha * (A @ B.T) + bf16_bits_to_f32(bias).astype(np.float64)[None, :]
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())
    np.testing.assert_allclose(ab, np.abs(alpha) * (np.abs(A) @ np.abs(B).T), rtol=1e-12)
    # a row slice equals the same rows of the full product
    part, _ = oracle.gemm(A, B, bias, alpha, rows=(M // 2, M))
    assert np.array_equal(part, out[M // 2:])


def test_decode_values_by_hand():
    # MXFP8: code 0x38 (1.0) with scale byte 130 (2^3) -> 8; code 0xC4 (-3.0, hmm: 0xC4 = -(1.5 * 2^1)) -> -24
    codes = np.array([[0x38, 0xC4] + [0] * 30], dtype=np.uint8)
    scales = np.array([[130]], dtype=np.uint8)
    d = oracle.decode("mxfp8", codes, scales, 1, 32)
    assert d[0, 0] == 8.0 and d[0, 1] == -24.0
    # NVFP4: byte 0x73 = low nibble 3 (1.5), high nibble 7 (6); scale 0x40 (2.0) -> 3.0, 12.0
    codes = np.array([[0x73] + [0] * 7], dtype=np.uint8)
    d = oracle.decode("nvfp4", codes, np.array([[0x40]], np.uint8), 1, 16)
    assert d[0, 0] == 3.0 and d[0, 1] == 12.0


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
def test_identity_and_ones_closed_forms(fmt):
    K = 64
    a = random_matrix(16, K, seed=4)
    qa = oracle.quantize(fmt, a)
    A = qa.decode()
    eye = oracle.quantize(fmt, f32_to_bf16_bits(np.eye(K, dtype=np.float32)))
    # identity weights: out = alpha * A_hat. Each row of I quantizes to a single nonzero code; for
    # NVFP4 it decodes to 6 * 448 * g with g = fp32(1 / 2688), i.e. 1 within one fp32 rounding
    np.testing.assert_allclose(eye.decode() * (eye.g if fmt == "nvfp4" else 1.0), np.eye(K), rtol=2.0 ** -24)
    alpha = qa.g * eye.g if fmt == "nvfp4" else 1.0
    out, _ = oracle.gemm(A, eye.decode(), None, alpha)
    np.testing.assert_allclose(out, A * (qa.g if fmt == "nvfp4" else 1.0) * np.diag(eye.decode() * (eye.g if fmt == "nvfp4" else 1.0))[None, :], rtol=1e-15)
    # all-ones weights: out[m, n] = alpha * row sum of A_hat, for every n
    ones = oracle.quantize(fmt, f32_to_bf16_bits(np.ones((8, K), np.float32)))
    alpha = qa.g * ones.g if fmt == "nvfp4" else 1.0
    out, _ = oracle.gemm(A, ones.decode(), None, alpha)
    Ones = ones.decode()
    assert np.all(Ones == Ones[0, 0])
    unit = Ones[0, 0] * (ones.g if fmt == "nvfp4" else 1.0)    # 1, up to fp32 rounding of g for NVFP4
    assert abs(unit - 1.0) <= 2.0 ** -24
    rs = A.sum(axis=1) * (qa.g if fmt == "nvfp4" else 1.0) * unit
    np.testing.assert_allclose(out, np.repeat(rs[:, None], 8, axis=1), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fmt,lo,hi", [("mxfp8", 0.01, 0.08), ("nvfp4", 0.04, 0.2), ("mxfp4", 0.06, 0.3)])
def test_error_band_plausibility(fmt, lo, hi):
    # the per-GEMM relative L2 errors quoted for real activations are ~0.03 / ~0.11 / ~0.19
    # (lightly-train README, section 5.4); on Gaussian data ours must land in the same decade
    a = random_matrix(64, 512, seed=8)
    b = random_matrix(96, 512, seed=9, std=0.02)
    _, _, out, _ = oracle.reference_linear(fmt, a, b)
    exact = bf16_bits_to_f32(a).astype(np.float64) @ bf16_bits_to_f32(b).astype(np.float64).T
    rel = np.linalg.norm(out - exact) / np.linalg.norm(exact)
    assert lo < rel < hi, rel


def test_tiny_workload_end_to_end():
    g = WORKLOADS["tiny_mxfp8"].gemms[0]
    a, b = make_activations(g), make_weights(g)
    assert a.dtype == np.float32 and a.shape == (128, 256) and b.shape == (256, 256)
    assert make_bias(g) is None
    # 1% of A entries are outliers x50
    # (an outlier whose N(0,1) draw was below 0.16 in magnitude stays under 8)
    assert 250 <= (np.abs(a) > 8).sum() <= 328
    qa, qb, out, ab = oracle.reference_linear("mxfp8", a, b)
    assert out.shape == (128, 256) and np.all(np.isfinite(out))
    exact = a.astype(np.float64) @ b.astype(np.float64).T
    assert np.linalg.norm(out - exact) / np.linalg.norm(exact) < 0.08
