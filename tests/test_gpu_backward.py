"""GPU parity of the backward GEMMs of a block-scaled linear layer against the CPU oracle:
dgrad dX = dY . W (dY quantized along N, W along N: its column-wise layout) and wgrad
dW = dY^T . X (dY and X quantized along M: their column-wise layouts), every operand from the
dual-layout quantizer, the output gradient with stochastic rounding. Operands bit-identical to
the oracle's; outputs within |gpu - y| <= 2^-7 |y| + 1e-5 sum_k |a b| of the oracle's fp64
GEMM on them."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import check_gemm_rows, sample_rows, to_dev
from workloads import Gemm, MXFP8, NVFP4, make_activations, make_output_grad, make_weights, random_matrix

pytestmark = pytest.mark.gpu


def _bsq():
    import block_scaled_precision_bsq_gb300 as bsq

    return bsq


def _same(got, want, what):
    codes = got.codes.cpu().numpy()
    assert np.array_equal(codes, want.codes), "%s codes differ in %d bytes" % (what, int((codes != want.codes).sum()))
    assert np.array_equal(got.scales.cpu().numpy(), want.tiled_scales()), "%s scales differ" % what


def _run(fmt, M, K, N, sr, seed, full_rows=False):
    bsq = _bsq()
    g = Gemm("layer", fmt, M, K, N, seed=seed)
    x, w, dy = make_activations(g), make_weights(g), make_output_grad(g)
    xr, xc = bsq.quantize_dual(fmt, to_dev(x))
    wr, wc = bsq.quantize_dual(fmt, to_dev(w))
    dx, dw = bsq.linear_backward(to_dev(dy), xc, wc, stochastic=sr, seed=seed + 99)
    if fmt == NVFP4:  # the GEMM's alpha is g_A * g_B, read from the operands' tails
        assert xc.global_scale is not None and wc.global_scale is not None
    torch.cuda.synchronize()
    assert bsq.device_status() == 0
    ox = oracle.quantize_dual(fmt, x)
    ow = oracle.quantize_dual(fmt, w)
    ody = oracle.quantize_dual(fmt, dy, stochastic=sr, seed=seed + 99)
    _same(xc, ox[1], "X column-wise")
    _same(wc, ow[1], "W column-wise")
    dyr, dyc = bsq.quantize_dual(fmt, to_dev(dy), stochastic=sr, seed=seed + 99)
    _same(dyr, ody[0], "dY row-wise")
    _same(dyc, ody[1], "dY column-wise")
    rows_dx = np.arange(M) if full_rows else sample_rows(M, seed=1)
    rows_dw = np.arange(N) if full_rows else sample_rows(N, seed=2)
    dx_np = dx.float().cpu().numpy().astype(np.float64)[rows_dx]
    dw_np = dw.float().cpu().numpy().astype(np.float64)[rows_dw]
    check_gemm_rows(dx_np, ody[0], ow[1], None, rows_dx, "dgrad")
    check_gemm_rows(dw_np, ody[1], ox[1], None, rows_dw, "wgrad")


# dgrad contracts over N and wgrad over M, so both are multiples of 128 (the MXFP8 GEMM's K
# step); output tiles of 256 x 256 are ragged in every case
@pytest.mark.parametrize("M,K,N", [(128, 128, 128), (384, 256, 640), (640, 416, 384)])
@pytest.mark.parametrize("sr", [False, True])
def test_backward_mxfp8_matches_oracle(M, K, N, sr):
    _run(MXFP8, M, K, N, sr, seed=M + K + N, full_rows=True)


# NVFP4 contracts in steps of 256
@pytest.mark.parametrize("M,K,N", [(256, 256, 256), (512, 416, 768)])
@pytest.mark.parametrize("sr", [False, True])
def test_backward_nvfp4_matches_oracle(M, K, N, sr):
    _run(NVFP4, M, K, N, sr, seed=M + K + N, full_rows=True)


def test_delayed_scale_feeds_the_next_quantization():
    """Step 1 quantizes dY with its own amax; the delayed scale (headroom 32) from step 1's tail
    quantizes step 2's dY (stochastic): scale value and both layouts bit-exact against the
    oracle, and step 2's tails record g and step 2's own amax."""
    bsq = _bsq()
    d1 = random_matrix(256, 384, seed=31, std=1e-3)
    d2 = random_matrix(256, 384, seed=32, std=3e-3)
    q1 = bsq.quantize_dual("nvfp4", to_dev(d1))
    g2 = bsq.delayed_global_scale(q1[1], headroom=32.0)
    o1 = oracle.quantize_dual("nvfp4", d1)
    g2_want = oracle.delayed_global_scale(o1[0].amax, 32.0)
    assert g2.item() == g2_want
    q2 = bsq.quantize_dual("nvfp4", to_dev(d2), stochastic=True, seed=77, global_scale=g2)
    assert bsq.device_status() == 0
    o2 = oracle.quantize_dual("nvfp4", d2, stochastic=True, seed=77, global_scale=g2_want)
    _same(q2[0], o2[0], "dY step 2 row-wise")
    _same(q2[1], o2[1], "dY step 2 column-wise")


def test_backward_full_size_vitb_fc1():
    """ViT-B/16 fc1 at training shape (M = 14336 tokens, K = 768, N = 3072): dgrad is
    14336 x 768 over N = 3072, wgrad 3072 x 768 over M = 14336; sampled rows."""
    _run(MXFP8, 14336, 768, 3072, True, seed=0)
