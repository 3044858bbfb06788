"""Pins of the oracle's producer-fused quantization step (reading R8): exact-erf GELU and the
MX rule on fp64 values. Each is tied to something other than the code under test: closed
forms of GELU, an independent statistics library, and the already pinned bf16/fp32 MX
quantizer on values both can represent."""
import math

import numpy as np
import pytest

import oracle
from workloads import f32_to_bf16_bits


def test_gelu_closed_forms():
    # GELU(0) = 0; GELU(x) - GELU(-x) = x (erf is odd); GELU(x) -> x and GELU(-x) -> 0 for large x
    x = np.array([0.0, 0.5, 1.0, 2.0, 3.0, 7.5, 30.0])
    g, gm = oracle.gelu_erf(x), oracle.gelu_erf(-x)
    assert g[0] == 0.0
    assert np.allclose(g - gm, x, rtol=0, atol=1e-15 * np.maximum(1, x))
    assert g[-1] == 30.0 and -1e-190 < gm[-1] <= 0.0
    # no cancellation: deep in the negative tail GELU is x * Phi(x), tiny but not zero
    assert oracle.gelu_erf(np.array([-10.0]))[0] == pytest.approx(-10.0 * 7.619853024160527e-24, rel=1e-12)


def test_gelu_is_x_times_normal_cdf():
    # GELU(x) = x * Phi(x), Phi from the statistics library (a different route to erf)
    stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(4000) * 3, np.linspace(-8, 8, 257)])
    want = x * stats.norm.cdf(x)
    assert np.allclose(oracle.gelu_erf(x), want, rtol=1e-12, atol=1e-300)
    # and against the stdlib, value by value (erf form where it does not cancel, erfc elsewhere)
    got = oracle.gelu_erf(x[:400])
    for xi, gi in zip(x[:400], got):
        want_i = 0.5 * xi * (1 + math.erf(xi / math.sqrt(2))) if xi > 0 else 0.5 * xi * math.erfc(-xi / math.sqrt(2))
        assert gi == pytest.approx(want_i, rel=1e-14, abs=1e-300)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_mx_f64_equals_pinned_quantizer_on_bf16_values(fmt):
    # on values exactly representable in bf16 the fp64 path must give the pinned path's bytes
    rng = np.random.default_rng(6)
    x = rng.standard_t(4, size=(37, 256)) * np.exp2(rng.integers(-20, 20, size=(37, 1)))
    bits = f32_to_bf16_bits(x.astype(np.float32))
    exact = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    a = oracle.quantize_mx_f64(fmt, exact)
    b = oracle.quantize(fmt, bits)
    assert np.array_equal(a.codes, b.codes) and np.array_equal(a.scales, b.scales)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_mx_f64_shift_invariance_and_zero_block(fmt):
    rng = np.random.default_rng(7)
    y = rng.standard_normal((8, 64))
    y[3, :32] = 0.0
    a, b = oracle.quantize_mx_f64(fmt, y), oracle.quantize_mx_f64(fmt, y * 2.0 ** 9)
    assert np.array_equal(a.codes, b.codes)
    sa, sb = a.scales.astype(int), b.scales.astype(int)
    assert np.array_equal(sb[sa != 0], sa[sa != 0] + 9)
    assert a.scales[3, 0] == 0  # amax 0 -> e = -127 -> byte 0


def test_encode_array_equals_scalar_encoders():
    rng = np.random.default_rng(8)
    v = np.concatenate([rng.standard_normal(2000) * 100, rng.standard_normal(2000) * 3,
                        [0.0, -0.0, 448.0, 464.0, 6.0, 5.0, -7.0]])
    e4 = oracle.encode_array("e4m3", v)
    e2 = oracle.encode_array("e2m1", v)
    assert all(int(c) == oracle.encode_e4m3(float(x)) for c, x in zip(e4, v))
    assert all(int(c) == oracle.encode_e2m1(float(x)) for c, x in zip(e2, v))
