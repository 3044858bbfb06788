"""Pins of the oracle's LayerNorm (reading R9): numpy's mean and variance as the library route,
closed-form row statistics, and invariance of LayerNorm under x -> a x + b (a > 0) with eps 0."""
import numpy as np
import pytest

import oracle
from workloads import bf16_bits_to_f32, f32_to_bf16_bits


def _gb(cols, seed, unit=False):
    rng = np.random.default_rng(seed)
    if unit:
        return f32_to_bf16_bits(np.ones(cols, np.float32)), f32_to_bf16_bits(np.zeros(cols, np.float32))
    return (f32_to_bf16_bits((1 + 0.1 * rng.standard_normal(cols)).astype(np.float32)),
            f32_to_bf16_bits((0.1 * rng.standard_normal(cols)).astype(np.float32)))


def test_layernorm_matches_numpy():
    rng = np.random.default_rng(1)
    x = f32_to_bf16_bits((rng.standard_normal((50, 768)) * 3 + 1).astype(np.float32))
    g, b = _gb(768, 2)
    xv = bf16_bits_to_f32(x).astype(np.float64)
    mu, var = xv.mean(axis=1, keepdims=True), xv.var(axis=1, keepdims=True)
    want = (xv - mu) / np.sqrt(var + 1e-6) * bf16_bits_to_f32(g) + bf16_bits_to_f32(b)
    assert np.allclose(oracle.layernorm(x, g, b, 1e-6), want, rtol=1e-12, atol=1e-12)


def test_layernorm_unit_affine_row_statistics():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((20, 1024)) * 5).astype(np.float32)
    g, b = _gb(1024, 0, unit=True)
    y = oracle.layernorm(x, g, b, 0.0)
    assert np.allclose(y.mean(axis=1), 0.0, atol=1e-12)
    assert np.allclose((y * y).mean(axis=1), 1.0, atol=1e-12)


def test_layernorm_shift_scale_invariance():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((8, 256)).astype(np.float32)
    g, b = _gb(256, 5)
    a = oracle.layernorm(x, g, b, 0.0)
    z = oracle.layernorm((x * np.float32(4.0) + np.float32(0.5)).astype(np.float32), g, b, 0.0)
    assert np.allclose(a, z, rtol=0, atol=1e-5)  # 4x + 0.5 is exact in fp32 up to one rounding of the shift


def test_layernorm_constant_row_is_beta():
    x = np.full((3, 64), 2.5, np.float32)
    g, b = _gb(64, 6)
    assert np.array_equal(oracle.layernorm(x, g, b, 1e-5), np.broadcast_to(bf16_bits_to_f32(b).astype(np.float64), (3, 64)))
