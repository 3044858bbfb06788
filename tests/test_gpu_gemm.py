"""GPU parity of the block-scaled GEMM against the oracle's fp64 GEMM, with the tolerance
|gpu - y| <= 2^-7 |y| + 1e-5 sum_k |a_ik b_kj| on every (or every sampled) output."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import bf16_to_f64, check_gemm_rows, sample_rows, to_dev
from workloads import WORKLOADS, f32_to_bf16_bits, make_activations, make_bias, make_weights, random_matrix

pytestmark = pytest.mark.gpu


def _bsq():
    import block_scaled_precision_bsq_gb300 as bsq

    return bsq


def _qtensor_from_oracle(q: "oracle.Quantized"):
    """Device copies of oracle-made codes and scales: isolates the GEMM from the quantizer."""
    bsq = _bsq()
    t = bsq.QTensor(q.fmt, q.rows, q.cols, to_dev(q.codes), to_dev(q.tiled_scales()))
    return t


def _run_linear(fmt, a, b, bias):
    bsq = _bsq()
    qa, qb = bsq.quantize(fmt, to_dev(a)), bsq.quantize(fmt, to_dev(b))
    out = bsq.gemm(qa, qb, None if bias is None else to_dev(bias))
    assert bsq.device_status() == 0
    return out


# (M, N, K): one tile, several tiles with ragged M, several N tiles, long K
SMALL = [(128, 256, 256), (200, 512, 512), (300, 768, 1024), (1, 256, 512), (129, 256, 2048), (384, 1024, 256)]


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("M,N,K", SMALL)
def test_gemm_oracle_operands(fmt, M, N, K):
    """The GEMM alone, fed the oracle's own codes and scales."""
    bsq = _bsq()
    a = random_matrix(M, K, seed=M + K, dist="student_t4")
    b = random_matrix(N, K, seed=N + K + 1, std=0.02)
    bias = f32_to_bf16_bits(np.random.default_rng(3).standard_normal(N).astype(np.float32) * 0.1)
    qa, qb = oracle.quantize(fmt, a), oracle.quantize(fmt, b)
    ta, tb = _qtensor_from_oracle(qa), _qtensor_from_oracle(qb)
    out = bsq.gemm(ta, tb, to_dev(bias))
    assert bsq.device_status() == 0
    check_gemm_rows(bf16_to_f64(out), qa, qb, bias, np.arange(M), "%s %dx%dx%d" % (fmt, M, N, K))


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("M,N,K", SMALL[:4])
def test_linear_end_to_end(fmt, M, N, K):
    """Quantizer + GEMM on the device against the oracle's whole path."""
    a = random_matrix(M, K, seed=2 * M + K, dist="normal")
    b = random_matrix(N, K, seed=N + 3 * K, std=0.02)
    bias = f32_to_bf16_bits(np.linspace(-0.05, 0.05, N).astype(np.float32))
    out = _run_linear(fmt, a, b, bias)
    qa, qb = oracle.quantize(fmt, a), oracle.quantize(fmt, b)
    check_gemm_rows(bf16_to_f64(out), qa, qb, bias, np.arange(M), "%s linear" % fmt)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
def test_gemm_output_past_2_31_elements(fmt):
    """M = 524544, N = 4096, K = 256: a bf16 output of 2^31 + 2^20 elements (4.3 GB), stored by the
    epilogue's tensor map past element 2^31. A's rows repeat a seeded 4095-row base, so an output
    row stored at a wrapped offset would hold another row's values; sampled rows on both sides of
    element 2^31 against the oracle."""
    bsq = _bsq()
    M, N, K, nb = 524544, 4096, 256, 4095
    base = random_matrix(nb, K, seed=41, dist="student_t4")
    b = random_matrix(N, K, seed=42, std=0.02)
    bias = f32_to_bf16_bits(np.random.default_rng(43).standard_normal(N).astype(np.float32) * 0.01)
    qa = bsq.quantize(fmt, to_dev(base).repeat((M + nb - 1) // nb, 1)[:M])
    qb = bsq.quantize(fmt, to_dev(b))
    out = bsq.gemm(qa, qb, to_dev(bias))
    assert bsq.device_status() == 0
    edge = (1 << 31) // N  # the output row holding element 2^31
    idx = np.array(sorted({0, 1, 127, 128, edge - 1, edge, edge + 1, M - 1} |
                          set(np.random.default_rng(4).integers(0, M, 24).tolist())), dtype=np.int64)
    got = bf16_to_f64(out[torch.from_numpy(idx).cuda()])
    del out
    torch.cuda.empty_cache()
    ra = oracle.quantize(fmt, base[idx % nb], global_scale=qa.global_scale.item() if fmt == "nvfp4" else None)
    rb = oracle.quantize(fmt, b, global_scale=qb.global_scale.item() if fmt == "nvfp4" else None)
    check_gemm_rows(got, ra, rb, bias, np.arange(len(idx)), "%s M = %d" % (fmt, M))


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
def test_linear_massive_activations(fmt):
    """Quantizer + GEMM on ViT-L block 0's massive activations (maximum 1992 on the class and
    register tokens, rms 9; the README's section 5.5) against the oracle, every output of a
    ragged 1029-token, two-image batch."""
    M, N, K = 1029, 1024, 1024
    a = random_matrix(M, K, seed=77, dist="massive")
    b = random_matrix(N, K, seed=78, std=0.02)
    bias = f32_to_bf16_bits(np.random.default_rng(79).standard_normal(N).astype(np.float32) * 0.01)
    out = _run_linear(fmt, a, b, bias)
    qa, qb = oracle.quantize(fmt, a), oracle.quantize(fmt, b)
    check_gemm_rows(bf16_to_f64(out), qa, qb, bias, np.arange(M), "%s massive" % fmt)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
def test_gemm_no_bias_and_structured_scales(fmt):
    """Rows, columns and K blocks with very different scales: a wrong scale-factor mapping
    (row of A, row of B, or K block) shows up as large errors."""
    bsq = _bsq()
    M, N, K = 256, 512, 512
    rng = np.random.default_rng(42)
    a = rng.standard_normal((M, K)) * np.exp2(rng.integers(-6, 7, size=(M, 1))) \
        * np.exp2(np.repeat(rng.integers(-4, 5, size=(1, K // 32)), 32, axis=1))
    b = rng.standard_normal((N, K)) * np.exp2(rng.integers(-6, 7, size=(N, 1))) \
        * np.exp2(np.repeat(rng.integers(-4, 5, size=(1, K // 16)), 16, axis=1))
    a, b = f32_to_bf16_bits(a.astype(np.float32)), f32_to_bf16_bits(b.astype(np.float32))
    out = _run_linear(fmt, a, b, None)
    qa, qb = oracle.quantize(fmt, a), oracle.quantize(fmt, b)
    check_gemm_rows(bf16_to_f64(out), qa, qb, None, np.arange(M), "%s structured" % fmt)
    del bsq


def test_tiny_workload():
    """The 128x256x256 fp32 MXFP8 case, every output."""
    g = WORKLOADS["tiny_mxfp8"].gemms[0]
    a, b = make_activations(g), make_weights(g)
    out = _run_linear("mxfp8", a, b, None)
    qa, qb = oracle.quantize("mxfp8", a), oracle.quantize("mxfp8", b)
    check_gemm_rows(bf16_to_f64(out), qa, qb, None, np.arange(g.M), "tiny_mxfp8")


def test_ragged_m_7203_tokens():
    """7 * 1029 tokens (cls + 4 registers + 32 x 32 patches per image): M not a multiple of 128."""
    M, N, K = 7203, 1024, 1024
    a = random_matrix(M, K, seed=77)
    b = random_matrix(N, K, seed=78, std=0.02)
    bias = f32_to_bf16_bits(np.full(N, 0.01, np.float32))
    for fmt in ("mxfp8", "nvfp4"):
        out = _run_linear(fmt, a, b, bias)
        qa, qb = oracle.quantize(fmt, a), oracle.quantize(fmt, b)
        check_gemm_rows(bf16_to_f64(out[sample_rows(M)]), qa, qb, bias, sample_rows(M), "%s M=7203" % fmt)
        assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("name", ["vitb_fc1_mxfp8", "vitl_mxfp8", "vitl_nvfp4", "vitl_mlp_large"])
def test_full_size_workload_gemm(name):
    """Full-size shapes, as launched by the benchmark; outputs checked on sampled rows (first,
    last and two random rows of every 128-row tile)."""
    for g in WORKLOADS[name].gemms:
        a, b, bias = make_activations(g), make_weights(g), make_bias(g)
        out = _run_linear(g.fmt, a, b, bias)
        idx = sample_rows(g.M, seed=g.K + g.N)
        got = bf16_to_f64(out[torch.from_numpy(idx).cuda()])
        del out
        qa, qb = oracle.quantize(g.fmt, a), oracle.quantize(g.fmt, b)
        check_gemm_rows(got, qa, qb, bias, idx, "%s %s" % (name, g.name))
        torch.cuda.empty_cache()


def test_bounded_wait_reports_timeout_and_context_survives():
    bsq = _bsq()
    assert bsq.bsq_selftest_timeout(20_000_000) == 0          # 20 ms
    assert bsq.device_status() == bsq.ERR_TIMEOUT
    assert bsq.device_status() == 0                           # read-and-clear
    # the context is still usable
    test_gemm_oracle_operands("mxfp8", 128, 256, 256)


@pytest.mark.parametrize("fmt,K", [("mxfp8", 384), ("mxfp8", 640), ("mxfp4", 256), ("mxfp4", 768), ("nvfp4", 768)])
def test_gemm_partial_last_stage(fmt, K):
    """K that leaves the last pipeline stage with a single 128-byte K chunk."""
    bsq = _bsq()
    M, N = 300, 512
    a = random_matrix(M, K, seed=K, dist="student_t4")
    b = random_matrix(N, K, seed=K + 1, std=0.02)
    qa, qb = oracle.quantize(fmt, a), oracle.quantize(fmt, b)
    out = bsq.gemm(_qtensor_from_oracle(qa), _qtensor_from_oracle(qb), None)
    assert bsq.device_status() == 0
    check_gemm_rows(bf16_to_f64(out), qa, qb, None, np.arange(M), "%s K=%d" % (fmt, K))


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("M,N", [(1, 8), (33, 24), (130, 136), (257, 8)])
def test_gemm_narrow_n_and_single_stage_k(fmt, M, N):
    """The smallest legal shapes: N of 8 (one 16-byte bf16 row piece; the tile's store boxes
    clip at N), ragged M across the pair's two CTAs, and K of one pipeline stage (128 for MXFP8,
    256 for the FP4 formats); the output buffer is pre-filled so that a store past N or M shows."""
    bsq = _bsq()
    K = 128 if fmt == "mxfp8" else 256
    a = random_matrix(M, K, seed=M * 7 + N, dist="student_t4")
    b = random_matrix(N, K, seed=N * 5 + M, std=0.02)
    bias = f32_to_bf16_bits(np.random.default_rng(M + N).standard_normal(N).astype(np.float32) * 0.1)
    qa, qb = oracle.quantize(fmt, a), oracle.quantize(fmt, b)
    # a guard region after the M x N output must stay untouched
    buf = torch.full((M * N + 4096,), 12345, dtype=torch.int16, device="cuda")
    out = buf[: M * N].view(torch.bfloat16).view(M, N)
    bsq.gemm(_qtensor_from_oracle(qa), _qtensor_from_oracle(qb), to_dev(bias), out=out)
    assert bsq.device_status() == 0
    assert bool((buf[M * N:] == 12345).all())
    check_gemm_rows(bf16_to_f64(out), qa, qb, bias, np.arange(M), "%s %dx%dx%d" % (fmt, M, N, K))
