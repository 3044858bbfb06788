"""GPU parity of the quantizer kernels against the CPU oracle: codes, tiled scales (with
padding) and the NVFP4 tail must be bit-identical."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import to_dev
from workloads import WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, make_activations, make_weights, random_matrix

pytestmark = pytest.mark.gpu

SHAPES = [(1, 32), (7, 96), (128, 256), (130, 512), (200, 768), (257, 1056), (64, 4096)]
DISTS = ["normal", "student_t4", "uniform_exp"]


def _bsq():
    import block_scaled_precision_bsq_gb300 as bsq

    return bsq


def _compare(fmt, x_np, global_scale=None, label=""):
    bsq = _bsq()
    q = oracle.quantize(fmt, x_np, global_scale=global_scale)
    x = to_dev(x_np)
    gs = None if global_scale is None else torch.tensor([global_scale], dtype=torch.float32, device="cuda")
    gq = bsq.quantize(fmt, x, global_scale=gs)
    assert bsq.device_status() == 0
    codes = gq.codes.cpu().numpy()
    assert np.array_equal(codes, q.codes), "%s codes: %d bytes differ (first at %d)" % (
        label, int((codes != q.codes).sum()), int(np.argmax(codes != q.codes)))
    scales = gq.scales.cpu().numpy()
    want = q.tiled_scales()
    assert np.array_equal(scales, want), "%s scales: %d bytes differ (first at %d)" % (
        label, int((scales != want).sum()), int(np.argmax(scales != want)))
    if q.fmt == oracle.NVFP4 and global_scale is None:
        assert gq.global_scale.item() == q.g
    return gq, q


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("dist", DISTS)
def test_quantize_bf16_matches_oracle(fmt, rows, cols, dist):
    x = random_matrix(rows, cols, seed=rows * 7 + cols, dist=dist)
    _compare(fmt, x, label="%s %dx%d %s" % (fmt, rows, cols, dist))


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("rows,cols", [(2053, 1024), (1029, 4096)])
def test_quantize_massive_activations(fmt, rows, cols):
    """ViT-L block 0's massive activations (the README's section 5.5: maximum 1992, rms 9) on the
    class and register tokens of each 1024-token image. The block holding 1992 saturates MXFP8
    (shared exponent 2^2, 498 -> 448) and MXFP4 (2^8, 7.8 -> 6), and under NVFP4 it takes the
    largest E4M3 block scale, 448, since g = 1992 / 2688. Ragged rows; bit-exact."""
    x = random_matrix(rows, cols, seed=rows + cols, dist="massive")
    _compare(fmt, x, label="%s massive %dx%d" % (fmt, rows, cols))


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
def test_quantize_past_2_31_elements(fmt):
    """524544 x 4096 bf16, 2^31 + 2^20 elements (4.3 GB): element, code and scale offsets past 2^31.
    The rows repeat a seeded 4095-row base, so a row written at a wrapped offset would land on a
    row of other content. Sampled rows on both sides of element 2^31 against the oracle; NVFP4's
    per-tensor scale against the base's exact maximum."""
    bsq = _bsq()
    rows, cols, nb = 524544, 4096, 4095
    base = random_matrix(nb, cols, seed=31, dist="student_t4")
    x = to_dev(base).repeat((rows + nb - 1) // nb, 1)[:rows]
    q = bsq.quantize(fmt, x)
    assert bsq.device_status() == 0
    del x
    torch.cuda.empty_cache()
    edge = (1 << 31) // cols  # the row holding element 2^31
    idx = np.array(sorted({0, 1, 127, 128, edge - 1, edge, edge + 1, rows - 1} |
                          set(np.random.default_rng(3).integers(0, rows, 24).tolist())), dtype=np.int64)
    g = None
    if fmt == "nvfp4":
        g = float(np.float32(np.abs(bf16_bits_to_f32(base)).max()) / np.float32(2688.0))
        assert q.global_scale.item() == g
    ref = oracle.quantize(fmt, base[idx % nb], global_scale=g)
    rb = cols if fmt == "mxfp8" else cols // 2
    flat = q.codes.view(-1)
    got = torch.stack([flat[int(r) * rb:(int(r) + 1) * rb] for r in idx]).cpu().numpy()
    assert np.array_equal(got, ref.codes.reshape(len(idx), rb))
    nsc = cols // (16 if fmt == "nvfp4" else 32)
    off = np.array([[oracle.scale_tiled_offset(int(r), c, nsc) for c in range(nsc)] for r in idx], dtype=np.int64)
    sc = q.scales.view(-1)[torch.from_numpy(off.ravel()).cuda()].cpu().numpy().reshape(len(idx), nsc)
    assert np.array_equal(sc, ref.scales.reshape(len(idx), nsc))


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("rows,cols", [(3, 32), (128, 256), (131, 1024)])
def test_quantize_fp32_matches_oracle(fmt, rows, cols):
    x = random_matrix(rows, cols, seed=5, dist="uniform_exp", src_f32=True)
    _compare(fmt, x, label="%s f32" % fmt)


@pytest.mark.parametrize("rows,cols", [(3, 48), (130, 272), (64, 1024)])
@pytest.mark.parametrize("g", [1.0, 0.0123, 1e-6])
def test_nvfp4_given_scale(rows, cols, g):
    x = random_matrix(rows, cols, seed=9, dist="student_t4")
    gq, q = _compare("nvfp4", x, global_scale=g, label="nvfp4 given g=%g" % g)
    assert gq.global_scale.item() == np.float32(g)


def test_nvfp4_cols_multiple_of_16_only():
    # 48 and 272 columns: scale columns not a multiple of 4 -> zero padding inside the tile
    for cols in (16, 48, 272):
        _compare("nvfp4", random_matrix(5, cols, seed=cols), label="nvfp4 cols=%d" % cols)


@pytest.mark.parametrize("rows,cols", [(1025, 48), (300, 272), (77, 1040), (3, 16)])
@pytest.mark.parametrize("f32", [False, True])
def test_nvfp4_blocks_across_rows_many_steps(rows, cols, f32):
    """cols % 32 == 16: a lane's two NVFP4 blocks may lie in two rows, and the last piece of the
    matrix may hold a single block; with many warp steps, both per-tensor scale modes."""
    x = random_matrix(rows, cols, seed=rows + cols, dist="student_t4", src_f32=f32)
    _compare("nvfp4", x, label="nvfp4 %dx%d" % (rows, cols))
    _compare("nvfp4", x, global_scale=0.02, label="nvfp4 given %dx%d" % (rows, cols))


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
def test_special_values(fmt):
    # zeros, negative zeros, exact ties, saturating blocks, subnormal bf16, a zero block
    vals = np.array([0.0, -0.0, 448.0, -500.0, 304.0, 2.5, -3.5, 0.25, 6.0, 7.0, 1e-38, -1e-39, 1.0625,
                     3e38, -3e38, 5.0], dtype=np.float32)
    x = np.zeros((4, 64), np.float32)
    x[0, :16] = vals
    x[1, :16] = vals[::-1]
    x[2, 32:48] = vals * np.float32(1e-30)
    x[3, :] = -0.0
    _compare(fmt, f32_to_bf16_bits(x), label="%s specials" % fmt)
    _compare(fmt, x, label="%s specials f32" % fmt)


def test_nvfp4_all_zero_tensor():
    x = np.zeros((2, 32), np.float32)
    x[1, 5] = -0.0
    gq, q = _compare("nvfp4", f32_to_bf16_bits(x), label="nvfp4 zero tensor")
    assert gq.global_scale.item() == 0.0


@pytest.mark.parametrize("name", ["tiny_mxfp8", "vitb_fc1_mxfp8", "vitl_mxfp8", "vitl_nvfp4", "vitl_mlp_large"])
def test_full_size_workload_quantize(name):
    """Every activation and weight tensor of the workload, at full size, bit-exact: codes,
    tiled scales with their padding and (NVFP4) the tail. The tiny case quantizes its fp32
    sources (A 128 x 256 with 1 % of the entries x50, B 256 x 256) along K."""
    seen = set()
    for g in WORKLOADS[name].gemms:
        for kind, make in (("A", make_activations), ("B", make_weights)):
            key = (kind, g.fmt, g.M if kind == "A" else g.N, g.K, g.a_dist if kind == "A" else "w")
            if key in seen:
                continue
            seen.add(key)
            _compare(g.fmt, make(g), label="%s %s %s" % (name, g.name, kind))
            torch.cuda.empty_cache()


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("f32", [False, True])
def test_batch_equals_single_calls_and_oracle(fmt, f32):
    """bsq_quantize_batch over matrices of different shapes (ragged rows, a row longer than a
    chunk) gives the bytes of one bsq_quantize call per matrix, and those of the oracle."""
    bsq = _bsq()
    shapes = [(300, 768), (7, 96), (129, 8192), (1, 32), (1000, 1024)]
    xs_np = [random_matrix(r, c, seed=40 + i, dist="student_t4", src_f32=f32) for i, (r, c) in enumerate(shapes)]
    xs = [to_dev(x) for x in xs_np]
    many = bsq.quantize_many(fmt, xs)
    assert bsq.device_status() == 0
    for x, x_np, qm in zip(xs, xs_np, many):
        q1 = bsq.quantize(fmt, x)
        assert torch.equal(qm.codes, q1.codes) and torch.equal(qm.scales, q1.scales)
        o = oracle.quantize(fmt, x_np)
        assert np.array_equal(qm.codes.cpu().numpy(), o.codes)
        assert np.array_equal(qm.scales.cpu().numpy(), o.tiled_scales())
        if fmt == "nvfp4":
            assert qm.global_scale.item() == o.g


def test_batch_nvfp4_mixed_magnitudes_and_narrow_rows():
    """One batch of NVFP4 matrices whose magnitudes differ by 10^8 (and one all-zero matrix):
    the single amax launch must give every matrix its own per-tensor scale. The shapes put many
    rows into one 1024-element warp step (cols 64, 128, 192: the word-wide scale stores of lane
    pairs) and a width that is not a multiple of 64 (1088: byte stores)."""
    bsq = _bsq()
    shapes = [(33, 64), (9, 192), (130, 128), (5, 1088)]
    mags = [1e-4, 1.0, 1e4, 0.0]
    from workloads import bf16_bits_to_f32, f32_to_bf16_bits

    xs_np = [f32_to_bf16_bits((bf16_bits_to_f32(random_matrix(r, c, seed=60 + i, dist="student_t4")) *
                               np.float32(m)).astype(np.float32))
             for i, ((r, c), m) in enumerate(zip(shapes, mags))]
    xs = [to_dev(x) for x in xs_np]
    many = bsq.quantize_many("nvfp4", xs)
    assert bsq.device_status() == 0
    for x_np, qm, m in zip(xs_np, many, mags):
        o = oracle.quantize("nvfp4", x_np)
        assert np.array_equal(qm.codes.cpu().numpy(), o.codes), "magnitude %g" % m
        assert np.array_equal(qm.scales.cpu().numpy(), o.tiled_scales()), "magnitude %g" % m
        assert qm.global_scale.item() == o.g
        assert (o.g == 0.0) == (m == 0.0)


def test_batch_nvfp4_given_scales():
    bsq = _bsq()
    xs_np = [random_matrix(64, 256, seed=50, dist="normal"), random_matrix(200, 512, seed=51, dist="student_t4")]
    gs = [0.01, 0.003]
    xs = [to_dev(x) for x in xs_np]
    outs = [bsq.empty_qtensor("nvfp4", x.shape[0], x.shape[1]) for x in xs]
    for q, g in zip(outs, gs):
        q.global_scale.fill_(g)
    items = [(x, x.shape[0], x.shape[1], q.codes, q.scales, q.global_scale) for x, q in zip(xs, outs)]
    assert bsq.bsq_quantize_batch(bsq.NVFP4 | bsq.FLAG_GLOBAL_GIVEN, items) == bsq.OK
    assert bsq.device_status() == 0
    for x_np, q, g in zip(xs_np, outs, gs):
        o = oracle.quantize("nvfp4", x_np, global_scale=g)
        assert np.array_equal(q.codes.cpu().numpy(), o.codes)
        assert np.array_equal(q.scales.cpu().numpy(), o.tiled_scales())


def _nudge(v, k):
    """The float32 k ulps above (k > 0) or below v."""
    v = np.float32(v)
    for _ in range(abs(k)):
        v = np.nextafter(v, np.float32(np.inf if k > 0 else -np.inf))
    return v


def _boundary_blocks(g32, seed):
    """16 x 64 fp32: every 16-element block starts with its maximum amax = 6 s g (fixing the
    block scale s), the other 15 elements have quotients x / (s g) on or within 3 ulps of the
    e2m1 rounding boundaries."""
    rng = np.random.default_rng(seed)
    pairs = [(m, k) for m in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0) for k in range(-3, 4)]
    rows = []
    for r in range(16):
        row = []
        for b in range(4):
            s_target = float(rng.choice([0.875, 1.125, 1.375, 3.25, 13.0, 0.3125]))
            amax = np.float32(6.0 * s_target * g32)
            sc = np.float32(oracle.decode_e4m3(oracle.encode_e4m3(float(amax / np.float32(np.float32(6.0) * np.float32(g32))))))
            sg = np.float32(sc * np.float32(g32))
            block = [amax]
            for j in range(15):
                m, k = pairs[(r * 60 + b * 15 + j) % len(pairs)]
                block.append(_nudge(np.float32(np.float32(m) * sg), k))
            signs = rng.choice([-1.0, 1.0], size=16).astype(np.float32)
            signs[0] = 1.0
            row.extend(np.array(block, dtype=np.float32) * signs)
        rows.append(row)
    return np.array(rows, dtype=np.float32)


@pytest.mark.parametrize("g", [1.0 / 3.0, 0.0123, 7.77])
def test_nvfp4_quotients_at_rounding_boundaries(g):
    """Element quotients x / (s g) exactly on, and within three ulps of, every e2m1 rounding
    boundary (0.25 ... 5): the codes must follow the IEEE quotient, which a reciprocal-multiply
    alone would not get right there. The quantizer and the dual-layout quantizer (row layout)
    against the oracle, with the per-tensor scale given."""
    bsq = _bsq()
    g32 = float(np.float32(g))
    x = _boundary_blocks(g32, seed=int(g * 1000))
    _compare("nvfp4", x, global_scale=g32, label="boundaries g=%g" % g)
    xd = np.concatenate([x, x], axis=0)  # 32 rows for the dual kernel
    qr, _ = oracle.quantize_dual("nvfp4", xd, global_scale=g32)
    gr, _ = bsq.quantize_dual("nvfp4", to_dev(xd), global_scale=torch.tensor([g32], device="cuda"))
    assert np.array_equal(gr.codes.cpu().numpy(), qr.codes)
