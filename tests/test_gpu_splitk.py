"""GPU parity of the split-K GEMM (bsq_gemm_splitk): K cut into ranges whose fp32 partial sums
land in a workspace and are added in order by a second kernel. Against the oracle's fp64 GEMM with
the GEMM tolerance |gpu - y| <= 2^-7 |y| + 1e-5 sum_k |a_ik b_kj|; against bsq_gemm where the
result must match exactly (one range) or run to run (determinism)."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import bf16_to_f64, check_gemm_rows, to_dev
from workloads import f32_to_bf16_bits, random_matrix

pytestmark = pytest.mark.gpu


def _bsq():
    import block_scaled_precision_bsq_gb300 as bsq

    return bsq


def _operands(fmt, M, N, K, seed):
    bsq = _bsq()
    a = random_matrix(M, K, seed=seed, dist="student_t4")
    b = random_matrix(N, K, seed=seed + 1, std=0.02)
    bias = f32_to_bf16_bits(np.random.default_rng(seed + 2).standard_normal(N).astype(np.float32) * 0.1)
    qa, qb = oracle.quantize(fmt, a), oracle.quantize(fmt, b)
    ta = bsq.QTensor(qa.fmt, M, K, to_dev(qa.codes), to_dev(qa.tiled_scales()))
    tb = bsq.QTensor(qb.fmt, N, K, to_dev(qb.codes), to_dev(qb.tiled_scales()))
    return qa, qb, ta, tb, bias


# (M, N, K, splits): uneven ranges (16 stages in 3), ragged M and N, one-row M, 8 ranges, a
# partial N tile, a wgrad-like shape (few tiles, long K)
CASES = [(300, 264, 2048, 3), (1, 256, 1024, 2), (200, 512, 2048, 8), (129, 776, 1024, 4), (512, 256, 4096, 2)]


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("M,N,K,splits", CASES)
def test_splitk_against_oracle(fmt, M, N, K, splits):
    bsq = _bsq()
    stages = K // (128 if fmt == "mxfp8" else 256)
    splits = min(splits, stages)
    qa, qb, ta, tb, bias = _operands(fmt, M, N, K, seed=M + N + K)
    out = bsq.gemm_splitk(ta, tb, to_dev(bias), splits=splits)
    assert bsq.device_status() == 0
    check_gemm_rows(bf16_to_f64(out), qa, qb, bias, np.arange(M), "splitk %s %dx%dx%d / %d" % (fmt, M, N, K, splits))


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_one_range_is_bsq_gemm_and_splits_are_deterministic(fmt):
    bsq = _bsq()
    qa, qb, ta, tb, bias = _operands(fmt, 300, 512, 2048, seed=41)
    ref = bsq.gemm(ta, tb, to_dev(bias))
    one = bsq.gemm_splitk(ta, tb, to_dev(bias), splits=1)
    assert torch.equal(one.view(torch.int16), ref.view(torch.int16))
    ws = torch.empty(4 * 300 * 512, dtype=torch.float32, device="cuda")
    r1 = bsq.gemm_splitk(ta, tb, to_dev(bias), splits=4, workspace=ws)
    ws.fill_(float("nan"))  # no dependence on what the workspace held
    r2 = bsq.gemm_splitk(ta, tb, to_dev(bias), splits=4, workspace=ws)
    assert torch.equal(r1.view(torch.int16), r2.view(torch.int16))
    # a different summation order only: nearly every bf16 output equals the single-range one
    same = (r1.view(torch.int16) == ref.view(torch.int16)).float().mean().item()
    assert same > 0.97, same
    assert bsq.device_status() == 0


def test_splitk_argument_errors():
    bsq = _bsq()
    qa, qb, ta, tb, bias = _operands("mxfp8", 128, 256, 1024, seed=7)
    out = torch.empty(128, 256, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(2 * 128 * 256 + 4, dtype=torch.float32, device="cuda")
    args = (bsq.MXFP8, ta.codes, ta.scales, tb.codes, tb.scales, None, out, 128, 256, 1024)
    nbytes = ws.numel() * 4
    assert bsq.bsq_gemm_splitk(*args, 0, ws, nbytes) == bsq.ERR_ARG
    assert bsq.bsq_gemm_splitk(*args, 9, ws, nbytes) == bsq.ERR_ARG
    assert bsq.bsq_gemm_splitk(*args, 3, ws, nbytes) == bsq.ERR_ARG          # 3 x M x N does not fit
    assert bsq.bsq_gemm_splitk(*args, 2, None, nbytes) == bsq.ERR_ARG
    assert bsq.bsq_gemm_splitk(*args, 2, ws[1:], nbytes - 4) == bsq.ERR_ALIGN
    qa2, qb2, ta2, tb2, _ = _operands("mxfp8", 128, 256, 256, seed=8)        # 2 stages: at most 2 ranges
    args2 = (bsq.MXFP8, ta2.codes, ta2.scales, tb2.codes, tb2.scales, None, out, 128, 256, 256)
    assert bsq.bsq_gemm_splitk(*args2, 3, ws, nbytes) == bsq.ERR_ARG
    assert bsq.bsq_gemm_splitk(*args, 2, ws, nbytes) == bsq.OK
    assert bsq.device_status() == 0


def test_library_split_choice():
    """Two ranges for ViT-B/16 fc1's weight gradient (36 output tiles on 76 SM pairs), one for
    the forward GEMMs, never more ranges than K stages / 8."""
    bsq = _bsq()
    sm_pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    assert bsq.bsq_gemm_splitk_splits("mxfp8", 3072, 768, 14336) == min(8, sm_pairs // 36, 112 // 8)
    assert bsq.bsq_gemm_splitk_splits("mxfp8", 14336, 3072, 768) == 1
    assert bsq.bsq_gemm_splitk_splits("nvfp4", 7168, 1024, 4096) == 1
    assert bsq.bsq_gemm_splitk_splits("mxfp8", 128, 256, 1024) == 1  # 8 stages: one range of 8
    assert bsq.bsq_gemm_splitk_splits("mxfp8", 0, 256, 1024) == bsq.ERR_ARG
