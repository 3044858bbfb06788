"""Pins for the oracle's element codecs (E4M3, e2m1, UE8M0): exhaustive tables against two
independent float8/float4 implementations, encoders against brute-force nearest search."""
import numpy as np
import pytest
import torch

import oracle
from tests.bruteforce import all_bf16_values, nearest_even, value_table

ml_dtypes = pytest.importorskip("ml_dtypes")


def test_e4m3_decode_matches_torch_and_ml_dtypes():
    codes = np.arange(256, dtype=np.uint8)
    ours = np.array([oracle.decode_e4m3(c) for c in codes])
    ref_torch = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    ref_ml = codes.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    nan = np.isnan(ref_torch)
    assert np.array_equal(np.isnan(ours), nan)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(ours[~nan], ref_torch[~nan])
    assert np.array_equal(ours[~nan], ref_ml[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref_ml[~nan]))


def test_e4m3_landmarks():
    # largest finite E4M3 is 448 (BF16 ledger blog, section 5.4)
    assert oracle.decode_e4m3(0x7E) == 448.0
    assert oracle.decode_e4m3(0x01) == 2.0 ** -9      # smallest subnormal
    assert oracle.decode_e4m3(0x08) == 2.0 ** -6      # smallest normal
    assert oracle.decode_e4m3(0x38) == 1.0
    assert oracle.decode_e4m3(0xBE) == -1.75


def test_e2m1_decode_matches_ml_dtypes_and_value_set():
    codes = np.arange(16, dtype=np.uint8)
    ours = np.array([oracle.decode_e2m1(c) for c in codes])
    ref = codes.view(ml_dtypes.float4_e2m1fn).astype(np.float64)
    assert np.array_equal(ours, ref)
    assert np.array_equal(np.signbit(ours), np.signbit(ref))
    assert sorted(set(np.abs(ours))) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_ue8m0_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = np.array([oracle.decode_ue8m0(c) for c in codes])
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).double().numpy()
    assert np.isnan(ours[255]) and np.isnan(ref[255])
    # torch widens 2^-127 exactly; compare all finite entries
    assert np.array_equal(ours[:255], ref[:255])
    assert all(ours[c] == 2.0 ** (c - 127) for c in range(255))


E4M3_TABLE = value_table(oracle.decode_e4m3, 256, 0x80)
E2M1_TABLE = value_table(oracle.decode_e2m1, 16, 0x8)


def _enc_all(enc, v):
    f = np.vectorize(enc, otypes=[np.int64])
    return f(v)


def test_e4m3_encode_exhaustive_bf16_vs_bruteforce():
    v = all_bf16_values()
    ours = _enc_all(oracle.encode_e4m3, v)
    ref = nearest_even(v, *E4M3_TABLE, sign_bit=0x80)
    assert np.array_equal(ours, ref)


def test_e4m3_encode_vs_torch_in_range():
    v = all_bf16_values()
    v = v[np.abs(v) <= 464.0]   # beyond the 448/480 midpoint torch returns NaN, we saturate
    ours = _enc_all(oracle.encode_e4m3, v)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref.astype(np.int64))


def test_e2m1_encode_exhaustive_bf16_vs_bruteforce_and_ml_dtypes():
    v = all_bf16_values()
    ours = _enc_all(oracle.encode_e2m1, v)
    ref = nearest_even(v, *E2M1_TABLE, sign_bit=0x8)
    assert np.array_equal(ours, ref)
    inr = np.abs(v) <= 6.0
    ml = v[inr].astype(np.float32).astype(ml_dtypes.float4_e2m1fn).view(np.uint8) & 0xF
    assert np.array_equal(ours[inr], ml.astype(np.int64))


def test_encoders_random_fp32_vs_bruteforce():
    rng = np.random.default_rng(1234)
    n = 200_000
    mag = np.exp2(rng.uniform(-14, 10, n)).astype(np.float32).astype(np.float64)
    v = mag * rng.choice([-1.0, 1.0], n)
    assert np.array_equal(_enc_all(oracle.encode_e4m3, v), nearest_even(v, *E4M3_TABLE, sign_bit=0x80))
    v2 = np.exp2(rng.uniform(-4, 3.5, n)).astype(np.float32).astype(np.float64) * rng.choice([-1.0, 1.0], n)
    assert np.array_equal(_enc_all(oracle.encode_e2m1, v2), nearest_even(v2, *E2M1_TABLE, sign_bit=0x8))


@pytest.mark.parametrize("dec,enc,n,sign", [(oracle.decode_e4m3, oracle.encode_e4m3, 256, 0x80),
                                            (oracle.decode_e2m1, oracle.encode_e2m1, 16, 0x8)])
def test_roundtrip_every_finite_code(dec, enc, n, sign):
    for c in range(n):
        v = dec(c)
        if np.isfinite(v):
            assert enc(v) == c, (c, v)


@pytest.mark.parametrize("dec,enc,n,sign", [(oracle.decode_e4m3, oracle.encode_e4m3, 256, 0x80),
                                            (oracle.decode_e2m1, oracle.encode_e2m1, 16, 0x8)])
def test_midpoints_tie_to_even_code(dec, enc, n, sign):
    codes, vals = value_table(dec, n, sign)
    for i in range(len(vals) - 1):
        mid = 0.5 * (vals[i] + vals[i + 1])
        want = codes[i] if codes[i] % 2 == 0 else codes[i + 1]
        assert enc(mid) == want, (vals[i], vals[i + 1])
        assert enc(-mid) == want | sign
        # just off the midpoint goes to the nearer value
        assert enc(np.nextafter(mid, -np.inf)) == codes[i]
        assert enc(np.nextafter(mid, np.inf)) == codes[i + 1]


def test_saturation():
    for v in [448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 3e38]:
        assert oracle.encode_e4m3(v) == 0x7E
        assert oracle.encode_e4m3(-v) == 0xFE
    for v in [6.0, 6.5, 7.0, 100.0]:
        assert oracle.encode_e2m1(v) == 0x7
        assert oracle.encode_e2m1(-v) == 0xF


def test_signed_zero():
    assert oracle.encode_e4m3(-0.0) == 0x80
    assert oracle.encode_e4m3(-1e-9) == 0x80
    assert oracle.encode_e4m3(0.0) == 0x00
    assert oracle.encode_e2m1(-0.1) == 0x8
    assert oracle.encode_e2m1(0.25) == 0x0   # tie between 0 and 0.5 goes to the even code 0
