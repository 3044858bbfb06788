"""Pins of the oracle's dual-layout quantizer and stochastic rounding (reading R10): Philox's
published known-answer vectors, stochastic rounding against brute-force neighbours and exact
unbiasedness, and the round-to-nearest dual quantizer against the pinned quantizer applied to
the matrix and to its transpose."""
import os

import numpy as np
import pytest

import oracle
from tests.bruteforce import value_table
from workloads import f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def test_philox_known_answers():
    n = 0
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(t, 16) for t in line.split()]
        assert oracle.philox4x32_10(w[0:4], w[4:6]) == tuple(w[6:10])
        n += 1
    assert n == 3


def _neighbours(v, mags):
    """Largest representable magnitude <= |v| and smallest >= |v| (brute force over the table)."""
    a = abs(v)
    lo = mags[mags <= a].max()
    hi = mags[mags >= a].min() if a <= mags.max() else mags.max()
    return lo, hi


@pytest.mark.parametrize("elem", ["e4m3", "e2m1"])
def test_sr_extremes_are_round_up_and_truncation(elem):
    # the value tables come from the decoders, which are pinned to two float8/float4 libraries
    if elem == "e4m3":
        _, mags = value_table(oracle.decode_e4m3, 256, 0x80)
    else:
        _, mags = value_table(oracle.decode_e2m1, 16, 0x8)
    rng = np.random.default_rng(11)
    vmax = 448.0 if elem == "e4m3" else 6.0
    v = np.concatenate([rng.uniform(-vmax, vmax, 3000), rng.uniform(-1, 1, 1000) * 2.0 ** -6])
    v = f32_to_bf16_bits(v.astype(np.float32)).astype(np.uint32) << 16
    v = v.view(np.float32).astype(np.float64)
    dec = oracle.decode_e4m3 if elem == "e4m3" else oracle.decode_e2m1
    up = oracle.encode_sr_array(elem, v, np.zeros_like(v))
    down = oracle.encode_sr_array(elem, v, np.full_like(v, 1.0 - 2.0 ** -24))
    for x, cu, cd in zip(v, up, down):
        lo, hi = _neighbours(x, mags)
        assert abs(dec(int(cu))) == hi and abs(dec(int(cd))) == lo
        assert (x < 0) == (dec(int(cu)) < 0 or (dec(int(cu)) == 0 and np.signbit(dec(int(cu)))))


def test_sr_is_exactly_unbiased_on_dyadic_values():
    # v with few fractional bits relative to its spacing: the mean over a full grid of u is v
    rng = np.random.default_rng(12)
    v = (rng.integers(-400 * 8, 400 * 8, 200) / 8.0).astype(np.float64)  # multiples of 1/8 in (-400, 400)
    k = 12
    u = np.arange(2 ** k) / 2.0 ** k
    for x in v:
        codes = oracle.encode_sr_array("e4m3", np.full(u.shape, x), u)
        mean = np.mean([oracle.decode_e4m3(int(c)) for c in codes])
        assert mean == x


@pytest.mark.parametrize("elem", ["e4m3", "e2m1"])
def test_sr_mean_over_all_16_bit_u_is_exact_or_within_bound(elem):
    """Reading R10 draws u on the grid h 2^-16: the mean code over all 2^16 values of h equals v
    exactly when frac(|v| / spacing) has at most 16 bits (normal and subnormal targets), and
    exceeds |v| by less than 2^-16 spacing when the fraction is longer (P(up) =
    ceil(frac 2^16) / 2^16)."""
    rng = np.random.default_rng(19)
    dec = oracle.decode_e4m3 if elem == "e4m3" else oracle.decode_e2m1
    # (start, end, spacing) of the subnormal range and of normal binades
    ranges = ([(0.0, 2.0 ** -6, 2.0 ** -9), (2.0 ** -6, 2.0 ** -5, 2.0 ** -9), (1.0, 2.0, 2.0 ** -3),
               (256.0, 448.0, 32.0)] if elem == "e4m3" else
              [(0.0, 1.0, 0.5), (1.0, 2.0, 0.5), (2.0, 4.0, 1.0), (4.0, 6.0, 2.0)])
    u = np.arange(2 ** 16) / 2.0 ** 16
    for start, end, spacing in ranges:
        steps = int(round((end - start) / spacing))
        for _ in range(6):
            q16 = int(rng.integers(0, steps * 2 ** 16))            # 16 fractional bits: exact
            v = start + q16 * spacing * 2.0 ** -16
            sgn = -1.0 if rng.integers(2) else 1.0
            codes = oracle.encode_sr_array(elem, np.full(u.shape, sgn * v), u)
            assert np.mean([dec(int(c)) for c in codes]) == sgn * v, (elem, v)
            q20 = int(rng.integers(0, steps * 2 ** 20)) | 1        # 20 fractional bits
            w = start + q20 * spacing * 2.0 ** -20
            codes = oracle.encode_sr_array(elem, np.full(u.shape, w), u)
            m = np.mean([dec(int(c)) for c in codes])
            assert 0.0 < m - w < spacing * 2.0 ** -16, (elem, w, m)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_dual_rne_equals_pinned_quantizer(fmt):
    rng = np.random.default_rng(13)
    x = f32_to_bf16_bits((rng.standard_t(4, size=(96, 160)) * 2.0).astype(np.float32))
    row, col = oracle.quantize_dual(fmt, x)
    a = oracle.quantize(fmt, x)
    t = oracle.quantize(fmt, np.ascontiguousarray(x.T))
    assert np.array_equal(row.codes, a.codes) and np.array_equal(row.scales, a.scales)
    assert np.array_equal(col.codes, t.codes) and np.array_equal(col.scales, t.scales)


def test_dual_sr_steps_at_most_one_code_and_depends_on_seed():
    rng = np.random.default_rng(14)
    x = f32_to_bf16_bits(rng.standard_normal((64, 128)).astype(np.float32))
    rne_row, rne_col = oracle.quantize_dual("mxfp8", x)
    s1_row, s1_col = oracle.quantize_dual("mxfp8", x, stochastic=True, seed=7)
    s2_row, _ = oracle.quantize_dual("mxfp8", x, stochastic=True, seed=8)
    assert np.array_equal(s1_row.scales, rne_row.scales) and np.array_equal(s1_col.scales, rne_col.scales)
    # same sign, magnitude codes within one step of the RNE code
    for a, b in ((s1_row, rne_row), (s1_col, rne_col)):
        d = (a.codes & 0x7F).astype(int) - (b.codes & 0x7F).astype(int)
        assert np.abs(d).max() <= 1
    assert not np.array_equal(s1_row.codes, s2_row.codes)
    s1_again, _ = oracle.quantize_dual("mxfp8", x, stochastic=True, seed=7)
    assert np.array_equal(s1_again.codes, s1_row.codes)


def test_sr_e2m1_is_exactly_unbiased_on_dyadic_values():
    rng = np.random.default_rng(15)
    v = (rng.integers(-6 * 8, 6 * 8, 120) / 8.0).astype(np.float64)  # multiples of 1/8 in (-6, 6)
    u = np.arange(2 ** 12) / 2.0 ** 12
    for x in v:
        codes = oracle.encode_sr_array("e2m1", np.full(u.shape, x), u)
        assert np.mean([oracle.decode_e2m1(int(c)) for c in codes]) == x


@pytest.mark.parametrize("given", [None, 0.0021])
def test_dual_nvfp4_rne_equals_pinned_quantizer(given):
    """Round to nearest: the two layouts are the pinned NVFP4 quantizer applied to X and to X^T
    with the same per-tensor scale (the tensor's amax, or the given scale)."""
    rng = np.random.default_rng(16)
    x = f32_to_bf16_bits((rng.standard_t(4, size=(96, 160)) * 3.0).astype(np.float32))
    row, col = oracle.quantize_dual("nvfp4", x, global_scale=given)
    a = oracle.quantize("nvfp4", x, global_scale=given)
    t = oracle.quantize("nvfp4", np.ascontiguousarray(x.T), global_scale=given)
    for got, want in ((row, a), (col, t)):
        assert np.array_equal(got.codes, want.codes) and np.array_equal(got.scales, want.scales)
        assert got.g == want.g and got.amax == want.amax
        assert np.array_equal(got.tiled_scales(), want.tiled_scales())


def _nibble(codes, i):
    return (int(codes[i // 2]) >> (4 * (i % 2))) & 0xF


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "nvfp4"])
def test_dual_sr_takes_each_elements_own_word(fmt):
    """Stochastic codes equal the pinned encoder applied to the element's scaled value v with
    u from the 16 Philox bits the reading assigns to the element (counter floor(i/8) and
    layout, key = seed, half i mod 2 of word (i mod 8) / 2; i = r C + c in the row layout,
    c R + r in the column layout),
    and v taken from the round-to-nearest dual quantizer's scales (which rounding leaves
    alone)."""
    rng = np.random.default_rng(17)
    R, C, seed = 64, 96, 0x1234_5678_9ABC_DEF0
    x = f32_to_bf16_bits((rng.standard_normal((R, C)) * 3.0).astype(np.float32))
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    rne = oracle.quantize_dual(fmt, x)
    sr = oracle.quantize_dual(fmt, x, stochastic=True, seed=seed)
    elem = "e4m3" if fmt == "mxfp8" else "e2m1"
    bs = 16 if fmt == "nvfp4" else 32
    for layout, (q_rne, q_sr) in enumerate(zip(rne, sr)):
        rows, cols = q_sr.rows, q_sr.cols
        for _ in range(300):
            r, c = int(rng.integers(rows)), int(rng.integers(cols))
            src = xf[r, c] if layout == 0 else xf[c, r]
            sb = int(q_rne.scales[r, c // bs])
            if fmt == "nvfp4":
                sg = np.float32(oracle.decode_e4m3(sb)) * np.float32(q_rne.g)
                if sg == 0:
                    continue
                v = float(np.float32(src) / sg)
            else:
                v = float(src) * 2.0 ** (127 - sb)
            i = r * cols + c
            words = oracle.philox4x32_10([(i // 8) & 0xFFFFFFFF, (i // 8) >> 32, layout, 0],
                                         [seed & 0xFFFFFFFF, seed >> 32])
            u = ((words[(i % 8) // 2] >> (16 * (i % 2))) & 0xFFFF) * 2.0 ** -16
            want = int(oracle.encode_sr_array(elem, np.array([v]), np.array([u]))[0])
            got = int(q_sr.codes[i]) if fmt == "mxfp8" else _nibble(q_sr.codes, i)
            assert got == want, (fmt, layout, r, c, v, u, got, want)


def test_dual_nvfp4_sr_steps_at_most_one_code():
    rng = np.random.default_rng(18)
    x = f32_to_bf16_bits(rng.standard_t(4, size=(64, 128)).astype(np.float32))
    rne = oracle.quantize_dual("nvfp4", x)
    s1 = oracle.quantize_dual("nvfp4", x, stochastic=True, seed=3)
    s2 = oracle.quantize_dual("nvfp4", x, stochastic=True, seed=4)
    for a, b in zip(s1, rne):
        assert np.array_equal(a.scales, b.scales) and a.g == b.g
        lo_a, hi_a = a.codes & 0xF, a.codes >> 4
        lo_b, hi_b = b.codes & 0xF, b.codes >> 4
        for p, q in ((lo_a, lo_b), (hi_a, hi_b)):
            assert np.array_equal(p & 0x8, q & 0x8)  # the sign of x in both
            assert np.abs((p & 0x7).astype(int) - (q & 0x7).astype(int)).max() <= 1
    assert not np.array_equal(s1[0].codes, s2[0].codes)


def test_delayed_scale_with_unit_headroom_is_the_computed_scale():
    """H = 1: the delayed scale from a tensor's recorded amax equals the scale the NVFP4
    quantizer computes from that tensor (reading R3)."""
    rng = np.random.default_rng(19)
    for k in range(20):
        x = f32_to_bf16_bits((rng.standard_t(3, size=(32, 64)) * 10.0 ** rng.uniform(-6, 6)).astype(np.float32))
        q = oracle.quantize("nvfp4", x)
        assert oracle.delayed_global_scale(q.amax, 1.0) == q.g


def test_delayed_scale_power_of_two_headroom_scales_exactly():
    """For H = 2^j the two rounded fp32 steps commute with the exact scaling: g(H) = 2^j g(1)."""
    rng = np.random.default_rng(20)
    for amax in np.float32(10.0) ** rng.uniform(-20, 20, 200).astype(np.float32):
        g1 = oracle.delayed_global_scale(amax, 1.0)
        for j in (1, 3, 5):
            assert oracle.delayed_global_scale(amax, 2.0 ** j) == g1 * 2.0 ** j
    # and a non-power-of-two headroom differs from scaling the computed g in some cases, i.e.
    # the product is taken before the division
    amax = np.float32(1.1)
    assert oracle.delayed_global_scale(amax, 3.0) == np.float32(np.float32(amax * np.float32(3.0)) / np.float32(2688.0))
