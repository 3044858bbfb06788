"""NVFP4 element codes where the quotient x / fp32(s g) sits on, or within a few fp32 ulps of,
an e2m1 decision point (the midpoints 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5 and the codes
themselves), plus zeros of both signs and tiny values: the round-to-nearest ties and near-ties
of the element rounding, where a quotient one ulp off changes the code. Every block holds an
element 6 s g, which fixes its E4M3 scale at s for the given per-tensor scale g. The (s, g)
pairs give d = s g exactly 1, an irregular d, a very small and a very large d. Codes and scales
are compared bit for bit with the oracle, for the single quantizer and both layouts of the dual
one (round-to-nearest and stochastic)."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu

POINTS = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
# (s, g): d = 1; irregular d; d = 448 * 2^-60; d = 2^-74; d = 448 * 2^62
CASES = [(1.0, 1.0), (0.8125, 1.0 / 3.0), (448.0, 2.0 ** -60), (2.0 ** -9, 2.0 ** -65), (448.0, 2.0 ** 62)]


def _bsq():
    import block_scaled_precision_bsq_gb300 as bsq

    return bsq


def _targets():
    """Quotient targets: each decision point and its 3 fp32 neighbours on each side, both
    signs, zeros and tiny values."""
    v = []
    for m in POINTS:
        b = np.float32(m).view(np.uint32)
        for k in range(-3, 4):
            v.append(np.uint32(int(b) + k).view(np.float32))
    v = np.array(v, dtype=np.float32)
    v = np.concatenate([v, -v, np.array([0.0, -0.0, 1e-30, -1e-30, 2 ** -140, 5.999, -0.124], np.float32)])
    return v


def _matrix(s, g, rows=32, cols=64, seed=0):
    """rows x cols fp32: in every 16-element row block, element 0 is fp32(6 s g) (so the block's
    E4M3 scale is s) and the other 15 are fp32(target * fp32(s g)), targets dealt in order."""
    d = np.float32(np.float32(s) * np.float32(g))
    bamax = np.float32(np.float32(6.0) * d)
    t = _targets()
    rng = np.random.default_rng(seed)
    x = np.empty((rows, cols), np.float32)
    k = 0
    for r in range(rows):
        for c0 in range(0, cols, 16):
            x[r, c0] = bamax
            for c in range(c0 + 1, c0 + 16):
                x[r, c] = np.float32(t[k % len(t)] * d)
                k += 1
        rng.shuffle(x[r, 1:16])  # vary which lanes meet the fallback
    return x


@pytest.mark.parametrize("s,g", CASES)
def test_quantize_codes_near_decision_points(s, g):
    bsq = _bsq()
    x = _matrix(s, g)
    want = oracle.quantize("nvfp4", x, global_scale=g)
    got = bsq.quantize("nvfp4", to_dev(x), global_scale=torch.tensor([g], dtype=torch.float32, device="cuda"))
    assert bsq.device_status() == 0
    codes = got.codes.cpu().numpy()
    assert np.array_equal(codes, want.codes), "%d of %d code bytes differ (first at %d)" % (
        int((codes != want.codes).sum()), codes.size, int(np.argmax(codes != want.codes)))
    assert np.array_equal(got.scales.cpu().numpy(), want.tiled_scales())


@pytest.mark.parametrize("s,g", CASES)
@pytest.mark.parametrize("stochastic", [False, True])
def test_dual_codes_near_decision_points(s, g, stochastic):
    bsq = _bsq()
    x = _matrix(s, g, rows=64, cols=96, seed=1)
    want = oracle.quantize_dual("nvfp4", x, stochastic=stochastic, seed=9, global_scale=g)
    got = bsq.quantize_dual("nvfp4", to_dev(x), stochastic=stochastic, seed=9,
                            global_scale=torch.tensor([g], dtype=torch.float32, device="cuda"))
    assert bsq.device_status() == 0
    for name, q, w in (("row", got[0], want[0]), ("col", got[1], want[1])):
        codes = q.codes.cpu().numpy()
        assert np.array_equal(codes, w.codes), "%s: %d of %d code bytes differ (first at %d)" % (
            name, int((codes != w.codes).sum()), codes.size, int(np.argmax(codes != w.codes)))
        assert np.array_equal(q.scales.cpu().numpy(), w.tiled_scales()), name


def _all_scales_matrix(g, seed):
    """fp32 blocks for every nonzero E4M3 scale code s: element 0 of each 16-element block is
    fp32(6 fp32(s g)) (the block's scale is then s), the other 15 carry the quotient targets of
    _targets() times fp32(s g), all targets dealt over the blocks of each s. Rows of 64."""
    t = _targets()
    per = -(-len(t) // 15)  # blocks per scale code
    blocks = []
    rng = np.random.default_rng(seed)
    for code in range(1, 127):
        s = oracle.decode_e4m3(code)
        d = np.float32(np.float32(s) * np.float32(g))
        tt = np.resize(t, per * 15).reshape(per, 15)
        b = np.empty((per, 16), np.float32)
        b[:, 0] = np.float32(np.float32(6.0) * d)
        b[:, 1:] = (tt * d).astype(np.float32)
        for row in b:
            rng.shuffle(row[1:])
        blocks.append(b)
    x = np.concatenate(blocks)
    pad = (-len(x)) % 4
    if pad:
        x = np.concatenate([x, np.zeros((pad, 16), np.float32)])
    return x.reshape(-1, 64)


@pytest.mark.parametrize("seed", range(4))
def test_quantize_every_scale_code_near_decision_points(seed):
    """For ten per-tensor scales g spread log-uniformly over 2^-40 .. 2^40 (so that d = fp32(s g)
    takes 1260 different significands), every one of the 126 nonzero block scales s with element
    quotients on and within three ulps of each e2m1 decision point: codes and scales bit-exact
    against the oracle's IEEE division."""
    bsq = _bsq()
    rng = np.random.default_rng(100 + seed)
    for g in np.exp2(rng.uniform(-40, 40, size=10)).astype(np.float32):
        g = float(g)
        x = _all_scales_matrix(g, seed)
        want = oracle.quantize("nvfp4", x, global_scale=g)
        got = bsq.quantize("nvfp4", to_dev(x), global_scale=torch.tensor([g], dtype=torch.float32, device="cuda"))
        assert bsq.device_status() == 0
        codes = got.codes.cpu().numpy()
        assert np.array_equal(codes, want.codes), "g=%r: %d of %d code bytes differ (first at %d)" % (
            g, int((codes != want.codes).sum()), codes.size, int(np.argmax(codes != want.codes)))
        assert np.array_equal(got.scales.cpu().numpy(), want.tiled_scales()), "g=%r scales" % g


@pytest.mark.parametrize("seed", range(2))
def test_quantize_bf16_every_value_every_scale_code(seed):
    """bf16 sources: for three per-tensor scales and every nonzero block scale s, blocks holding
    every bf16 value whose quotient x / fp32(s g) lies in [1/8, 8) (both signs), with an element
    6 s g fixing the scale: the whole range where e2m1 codes are decided, bit-exact."""
    from workloads import f32_to_bf16_bits

    bsq = _bsq()
    rng = np.random.default_rng(200 + seed)
    allbf = (np.arange(0x8000, dtype=np.uint32) << 16).view(np.float32)  # every non-negative bf16
    allbf = allbf[np.isfinite(allbf)]
    for g in np.exp2(rng.uniform(-20, 20, size=3)).astype(np.float32):
        g = float(g)
        blocks = []
        for code in range(1, 127):
            s = oracle.decode_e4m3(code)
            d = np.float32(np.float32(s) * np.float32(g))
            amax_bf = f32_to_bf16_bits(np.array([np.float32(6.0) * d], np.float32))
            amax = (amax_bf.astype(np.uint32) << 16).view(np.float32)[0]
            q = allbf / d
            v = allbf[(q >= 0.125) & (q < 8.0) & (allbf <= amax)]
            v = np.concatenate([v, -v])
            rng.shuffle(v)
            n = -(-len(v) // 15) * 15
            v = np.resize(v, n).reshape(-1, 15)
            b = np.empty((len(v), 16), np.float32)
            b[:, 0] = amax
            b[:, 1:] = v
            blocks.append(b)
        x = np.concatenate(blocks)
        pad = (-len(x)) % 4
        if pad:
            x = np.concatenate([x, np.zeros((pad, 16), np.float32)])
        xb = f32_to_bf16_bits(x.reshape(-1, 64))  # exact: every value is a bf16 value
        want = oracle.quantize("nvfp4", xb, global_scale=g)
        got = bsq.quantize("nvfp4", to_dev(xb), global_scale=torch.tensor([g], dtype=torch.float32, device="cuda"))
        assert bsq.device_status() == 0
        codes = got.codes.cpu().numpy()
        assert np.array_equal(codes, want.codes), "g=%r: %d of %d code bytes differ" % (
            g, int((codes != want.codes).sum()), codes.size)
        assert np.array_equal(got.scales.cpu().numpy(), want.tiled_scales()), "g=%r scales" % g
