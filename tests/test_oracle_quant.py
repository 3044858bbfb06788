"""Pins for the oracle's block quantizers: hand-derived fixtures, invariants of the UE8M0
shared-exponent rule, NVFP4 two-level scaling properties, and brute-force element checks."""
import numpy as np
import pytest

import oracle
from tests import golden_io
from tests.bruteforce import nearest_even, value_table
from workloads import bf16_bits_to_f32, f32_to_bf16_bits, random_matrix

E4M3_TABLE = value_table(oracle.decode_e4m3, 256, 0x80)
E2M1_TABLE = value_table(oracle.decode_e2m1, 16, 0x8)


def unpack_fp4(codes, n):
    lo = codes & 0xF
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(-1)[:n]


def codes_of(q):
    if q.fmt == oracle.MXFP8:
        return q.codes.astype(np.int64).reshape(q.rows, q.cols)
    return unpack_fp4(q.codes, q.rows * q.cols).astype(np.int64).reshape(q.rows, q.cols)


def bf16(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


@pytest.mark.parametrize("fmt,name", [("mxfp8", "mxfp8_block.txt"), ("mxfp4", "mxfp4_block.txt")])
def test_mx_golden_blocks(fmt, name):
    xs, cs, ss = golden_io.block_rows(golden_io.load(name), 32)
    x = np.concatenate(xs)[None, :]
    src = bf16(x)
    assert np.array_equal(bf16_bits_to_f32(src).astype(np.float64), x), "fixture values must be exact in bf16"
    for src_in in (src, x.astype(np.float32)):           # bf16 and fp32 sources agree
        q = oracle.quantize(fmt, src_in)
        assert np.array_equal(codes_of(q)[0], np.concatenate(cs))
        assert list(q.scales[0]) == ss


def test_nvfp4_golden_blocks():
    fix = golden_io.load("nvfp4_block.txt")
    xs, cs, ss = golden_io.block_rows(fix, 16)
    x = np.stack(xs)
    q = oracle.quantize("nvfp4", bf16(x))
    assert q.g == float(fix["g"][0]) and q.amax == float(fix["amax"][0])
    assert np.array_equal(codes_of(q), np.stack(cs))
    assert list(q.scales[:, 0]) == ss
    # the same tensor with the per-tensor scale given explicitly
    q2 = oracle.quantize("nvfp4", bf16(x), global_scale=1.0)
    assert np.array_equal(q2.codes, q.codes) and np.array_equal(q2.scales, q.scales)


@pytest.mark.parametrize("fmt,emax,maxval", [("mxfp8", 8, 448.0), ("mxfp4", 2, 6.0)])
@pytest.mark.parametrize("dist", ["normal", "student_t4", "uniform_exp"])
def test_mx_scale_invariants(fmt, emax, maxval, dist):
    x = random_matrix(64, 512, seed=7, dist=dist)
    q = oracle.quantize(fmt, x)
    xf = bf16_bits_to_f32(x).astype(np.float64).reshape(64, 16, 32)
    e = q.scales.astype(np.int64) - 127
    amax = np.abs(xf).max(axis=2)
    unclamped = (e > -127) & (amax > 0)
    # the largest element, divided by the power-of-two scale, lands in the top binade [2^emax, 2^(emax+1))
    lead = amax[unclamped] * np.exp2(-e[unclamped].astype(np.float64))
    assert np.all(lead >= 2.0 ** emax) and np.all(lead < 2.0 ** (emax + 1))
    # the largest code magnitude sits in the top binade [2^emax, maxval]
    dec = np.vectorize(oracle.decode_e4m3 if fmt == "mxfp8" else oracle.decode_e2m1)(codes_of(q))
    top = np.abs(dec).reshape(64, 16, 32).max(axis=2)[unclamped]
    assert np.all(top >= 2.0 ** emax) and np.all(top <= maxval)
    # every element is the brute-force nearest value of x / 2^e
    v = (xf * np.exp2(-e.astype(np.float64))[:, :, None]).reshape(-1)
    table, sign = (E4M3_TABLE, 0x80) if fmt == "mxfp8" else (E2M1_TABLE, 0x8)
    assert np.array_equal(codes_of(q).reshape(-1), nearest_even(v, *table, sign_bit=sign))


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_mx_power_of_two_shift(fmt):
    # scaling a tensor by 2^k moves every scale byte by k and leaves every code unchanged
    x = bf16_bits_to_f32(random_matrix(32, 256, seed=3))
    q0 = oracle.quantize(fmt, f32_to_bf16_bits(x))
    for k in (-5, 1, 9):
        qk = oracle.quantize(fmt, f32_to_bf16_bits(x * np.float32(2.0 ** k)))
        assert np.array_equal(qk.codes, q0.codes)
        assert np.array_equal(qk.scales.astype(int), q0.scales.astype(int) + k)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_mx_zero_block_and_tiny_block(fmt):
    x = np.zeros((2, 64), np.float32)
    x[0, 32:] = -0.0
    x[1, :32] = 1e-40            # subnormal fp32: floor(log2) far below -127, e clamps to -127
    q = oracle.quantize(fmt, x)
    assert list(q.scales[0]) == [0, 0] and list(q.scales[1]) == [0, 0]
    c = codes_of(q)
    neg0 = 0x80 if fmt == "mxfp8" else 0x8
    assert np.all(c[0, :32] == 0) and np.all(c[0, 32:] == neg0)
    # 1e-40 * 2^127 ~ 1.7e-2 is above half the smallest E4M3 subnormal (2^-10): a nonzero code
    want = oracle.encode_e4m3(float(np.float32(1e-40)) * 2.0 ** 127) if fmt == "mxfp8" else \
        oracle.encode_e2m1(float(np.float32(1e-40)) * 2.0 ** 127)
    assert np.all(c[1, :32] == want)


@pytest.mark.parametrize("dist", ["normal", "student_t4", "uniform_exp"])
def test_nvfp4_properties(dist):
    x = random_matrix(48, 256, seed=11, dist=dist)
    q = oracle.quantize("nvfp4", x)
    xf = bf16_bits_to_f32(x)
    amax = np.abs(xf).max()
    assert q.amax == amax
    assert q.g == np.float32(amax) / np.float32(2688.0)
    assert q.scales.max() <= 0x7E                     # E4M3 block scales are positive and finite
    # block scale = brute-force nearest E4M3 of fp32(bamax / fp32(6 g))
    bamax = np.abs(xf).reshape(48, 16, 16).max(axis=2)
    qv = (bamax / (np.float32(6.0) * np.float32(q.g))).astype(np.float32)
    assert np.array_equal(q.scales.astype(np.int64).reshape(-1),
                          nearest_even(qv.astype(np.float64).reshape(-1), *E4M3_TABLE, sign_bit=0x80))
    # element = brute-force nearest e2m1 of fp32(x / fp32(s g)), and within half an e2m1 step of it
    s = np.vectorize(oracle.decode_e4m3)(q.scales).astype(np.float32)
    sg = (s * np.float32(q.g)).astype(np.float32)
    zero_blk = np.broadcast_to((sg == 0)[:, :, None], (48, 16, 16)).reshape(-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = (xf.reshape(48, 16, 16) / sg[:, :, None]).astype(np.float32).reshape(-1)
    codes = codes_of(q).reshape(-1)
    # blocks whose scale rounds to 0 hold zeros that keep the sign of their input
    assert np.array_equal(codes[zero_blk], np.where(np.signbit(xf.reshape(-1)[zero_blk]), 0x8, 0x0))
    codes, y = codes[~zero_blk], y[~zero_blk]
    assert np.array_equal(codes, nearest_even(y.astype(np.float64), *E2M1_TABLE, sign_bit=0x8))
    dec = np.vectorize(oracle.decode_e2m1)(codes)
    ycl = np.clip(y, -6, 6)
    step = np.where(np.abs(ycl) < 2, 0.5, np.where(np.abs(ycl) < 4, 1.0, 2.0))
    assert np.all(np.abs(dec - ycl) <= step / 2 + 1e-12)


def test_nvfp4_sign_symmetry():
    x = random_matrix(16, 128, seed=5, dist="student_t4")
    xn = x ^ np.uint16(0x8000)                           # flip the bf16 sign bits
    q, qn = oracle.quantize("nvfp4", x), oracle.quantize("nvfp4", xn)
    assert np.array_equal(q.scales, qn.scales) and q.g == qn.g
    assert np.array_equal(codes_of(qn), codes_of(q) ^ 0x8)


def test_nvfp4_zero_tensor_and_zero_block():
    x = np.zeros((4, 32), np.float32)
    x[1, 3] = -0.0
    q = oracle.quantize("nvfp4", f32_to_bf16_bits(x))
    assert q.g == 0.0 and q.amax == 0.0
    assert np.all(q.scales == 0)
    c = codes_of(q)
    assert c[1, 3] == 0x8 and c.sum() == 0x8
    # a block far below the tensor maximum gets s = 0 and signed-zero codes
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 1000.0
    x[0, 16:] = [-1e-4, 1e-4] * 8
    q = oracle.quantize("nvfp4", f32_to_bf16_bits(x))
    assert q.scales[0, 1] == 0
    assert list(codes_of(q)[0, 16:]) == [0x8, 0x0] * 8


def test_nvfp4_given_scale_saturates():
    # with a small given g the block scale saturates at 448 and the elements at 6
    x = np.full((1, 16), 1000.0, np.float32)
    q = oracle.quantize("nvfp4", f32_to_bf16_bits(x), global_scale=0.125)
    assert q.g == 0.125 and q.scales[0, 0] == 0x7E and np.all(codes_of(q) == 0x7)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
def test_tiled_scale_layout_is_a_bijection_with_zero_pads(fmt):
    for rows, cols in [(128, 128), (200, 96), (1, 32), (257, 512)]:
        bs = oracle.block_size(fmt)
        nsc = cols // bs
        offs = np.array([[oracle.scale_tiled_offset(r, c, nsc) for c in range(nsc)] for r in range(rows)])
        nbytes = oracle.scales_tiled_bytes(fmt, rows, cols)
        body = nbytes - (16 if fmt == "nvfp4" else 0)
        assert body == -(-rows // 128) * 128 * (-(-nsc // 4) * 4)
        assert len(set(offs.reshape(-1))) == offs.size and offs.min() >= 0 and offs.max() < body
        plain = (np.arange(rows * nsc) % 251 + 1).astype(np.uint8).reshape(rows, nsc)
        t = oracle.tile_scales(fmt, plain, rows, cols, g=0.5, amax=3.0)
        assert np.array_equal(t[offs.reshape(-1)], plain.reshape(-1))
        mask = np.ones(body, bool)
        mask[offs.reshape(-1)] = False
        assert np.all(t[:body][mask] == 0)
        if fmt == "nvfp4":
            assert list(t[body:].view(np.float32)) == [0.5, 3.0, 0.0, 0.0]
        # one 128-row tile holds the 4 scale columns of 128 rows in 512 contiguous bytes, 32-row
        # groups interleaved inside each 16-byte line (the tcgen05 scale-factor atom)
        if rows >= 128 and nsc >= 4:
            assert sorted(offs[:128, :4].reshape(-1)) == list(range(512))
            assert offs[0, 1] - offs[0, 0] == 1 and offs[32, 0] - offs[0, 0] == 4 and offs[1, 0] - offs[0, 0] == 16
