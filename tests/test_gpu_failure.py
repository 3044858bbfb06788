"""The failure path of every kernel that waits on barriers, driven without any GPU fault.

bsq_test_inject_stall arms a one-shot stall for the calling thread's next launch of one kernel
class: its TMA producers stop issuing loads after a given number of pipeline stages (announcing no
bytes for the rest), so a consumer waits for a stage that never arrives. The launch's bounded waits
use a short limit (a few milliseconds). The starved wait must give up and record BSQ_ERR_TIMEOUT in
the device status word, every role must leave its loop, the producer must wait for the loads it
did issue (nothing left in flight), TMEM must be released -- and the context must stay usable: the
next launch of the same kernel produces exactly the bytes it produces without any stall, which
the other tests pin to the oracle. Stalls are placed before the first stage, inside the first tile
and inside a later tile."""
import time

import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import bf16_to_f64, check_gemm_rows, to_dev
from workloads import random_matrix

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000  # 2 ms per bounded wait in the stalled launch


def _bsq():
    import block_scaled_precision_bsq_gb300 as bsq

    return bsq


def _stalled(bsq, kernel, after, launch):
    """Arm the stall, launch, and return the device status (and the time it took to get it)."""
    assert bsq.bsq_test_inject_stall(kernel, after, LIMIT_NS) == bsq.OK
    t0 = time.perf_counter()
    launch()
    st = bsq.device_status()
    return st, time.perf_counter() - t0


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("after", [0, 3, 11])
def test_gemm_stall_times_out_and_next_gemm_is_unchanged(fmt, after):
    """M = 10240, N = 512: 80 tiles of 256 x 256, so the first SM pairs take two; K = 2048: 16
    (MXFP8) or 8 (FP4) stages per tile. `after` = 0 stalls before the first load, 3 inside the
    first tile, 11 inside the first tile (MXFP8) or the second (FP4: only the pairs with two tiles
    stall, the others finish normally)."""
    bsq = _bsq()
    M, N, K = 10240, 512, 2048
    a_np = random_matrix(M, K, seed=1, dist="student_t4")
    b_np = random_matrix(N, K, seed=2, std=0.02)
    qa, qb = bsq.quantize(fmt, to_dev(a_np)), bsq.quantize(fmt, to_dev(b_np))
    bias = (torch.randn(N, device="cuda") * 0.1).to(torch.bfloat16)
    want = bsq.gemm(qa, qb, bias)
    assert bsq.device_status() == bsq.OK
    out = torch.zeros_like(want)
    st, secs = _stalled(bsq, bsq.KERNEL_GEMM, after, lambda: bsq.gemm(qa, qb, bias, out=out))
    assert st == bsq.ERR_TIMEOUT
    assert secs < 1.0  # the short limit, not the 2 s default
    got = bsq.gemm(qa, qb, bias)
    assert bsq.device_status() == bsq.OK
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    # and that result is the oracle's, within the tolerance (rows of both pairs' tiles)
    oa, ob = oracle.quantize(fmt, a_np), oracle.quantize(fmt, b_np)
    rows = np.array([0, 127, 128, 255, 256, 383, 5000, 10239])
    bias_np = bias.view(torch.int16).cpu().numpy().view(np.uint16)
    check_gemm_rows(bf16_to_f64(got[rows]), oa, ob, bias_np, rows, "after stall")


def test_gemm_splitk_stall_times_out_then_recovers():
    bsq = _bsq()
    M, N, K = 256, 512, 4096
    qa = bsq.quantize("mxfp8", to_dev(random_matrix(M, K, seed=3)))
    qb = bsq.quantize("mxfp8", to_dev(random_matrix(N, K, seed=4, std=0.02)))
    want = bsq.gemm_splitk(qa, qb, None, splits=4)
    assert bsq.device_status() == bsq.OK
    st, _ = _stalled(bsq, bsq.KERNEL_GEMM, 5, lambda: bsq.gemm_splitk(qa, qb, None, splits=4))
    assert st == bsq.ERR_TIMEOUT
    got = bsq.gemm_splitk(qa, qb, None, splits=4)
    assert bsq.device_status() == bsq.OK
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("fmt,stochastic", [("mxfp8", False), ("nvfp4", True), ("mxfp4", False)])
@pytest.mark.parametrize("after", [0, 1, 3])
def test_dual_stall_times_out_and_next_dual_is_bit_exact(fmt, stochastic, after):
    """4096 x 4096 bf16: 1024 tiles of 128 x 128 over at most 304 CTAs, three or four each; the
    producers stop after `after` tiles (3: only the CTAs with four)."""
    bsq = _bsq()
    x_np = random_matrix(4096, 4096, seed=5, dist="student_t4")
    x = to_dev(x_np)
    st, secs = _stalled(bsq, bsq.KERNEL_DUAL, after, lambda: bsq.quantize_dual(fmt, x, stochastic=stochastic, seed=3))
    assert st == bsq.ERR_TIMEOUT
    assert secs < 1.0
    r, c = bsq.quantize_dual(fmt, x, stochastic=stochastic, seed=3)
    assert bsq.device_status() == bsq.OK
    wr, wc = oracle.quantize_dual(fmt, x_np, stochastic=stochastic, seed=3)
    for q, w in ((r, wr), (c, wc)):
        assert np.array_equal(q.codes.cpu().numpy(), w.codes)
        assert np.array_equal(q.scales.cpu().numpy(), w.tiled_scales())


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("after", [0, 2])
def test_layernorm_stall_times_out_and_next_call_is_unchanged(fmt, after):
    """Rows of 2048 bf16 take the shared-memory LayerNorm kernel (4096 one-row chunks over at most
    608 CTAs), whose producer the stall stops."""
    bsq = _bsq()
    rows, cols = 4096, 2048
    x = (torch.randn(rows, cols, device="cuda") * 3 + 1).to(torch.bfloat16)
    g = (1 + 0.1 * torch.randn(cols, device="cuda")).to(torch.bfloat16)
    b = (0.1 * torch.randn(cols, device="cuda")).to(torch.bfloat16)
    want = bsq.layernorm_quantize(fmt, x, g, b, 1e-6)
    assert bsq.device_status() == bsq.OK
    st, secs = _stalled(bsq, bsq.KERNEL_LAYERNORM, after, lambda: bsq.layernorm_quantize(fmt, x, g, b, 1e-6))
    assert st == bsq.ERR_TIMEOUT
    assert secs < 1.0
    got = bsq.layernorm_quantize(fmt, x, g, b, 1e-6)
    assert bsq.device_status() == bsq.OK
    assert torch.equal(got.codes, want.codes) and torch.equal(got.scales, want.scales)


def test_injection_is_one_shot_and_only_for_the_named_kernel():
    bsq = _bsq()
    qa = bsq.quantize("mxfp8", to_dev(random_matrix(256, 512, seed=6)))
    qb = bsq.quantize("mxfp8", to_dev(random_matrix(256, 512, seed=7, std=0.02)))
    x = to_dev(random_matrix(256, 256, seed=8))
    assert bsq.bsq_test_inject_stall(bsq.KERNEL_GEMM, 0, LIMIT_NS) == bsq.OK
    bsq.quantize_dual("mxfp8", x)  # another kernel class: unaffected, and does not consume it
    assert bsq.device_status() == bsq.OK
    bsq.gemm(qa, qb)                # consumes the stall
    assert bsq.device_status() == bsq.ERR_TIMEOUT
    bsq.gemm(qa, qb)                # one shot: runs normally
    assert bsq.device_status() == bsq.OK


def test_layernorm_stall_waits_for_the_shared_memory_kernel():
    """bf16 rows of at most 1024 elements take the streaming LayerNorm kernel, which waits on no
    barrier: an armed LayerNorm stall does not act there and stays armed for the next launch of
    the shared-memory kernel."""
    bsq = _bsq()
    g1 = (1 + 0.1 * torch.randn(1024, device="cuda")).to(torch.bfloat16)
    b1 = (0.1 * torch.randn(1024, device="cuda")).to(torch.bfloat16)
    g2 = (1 + 0.1 * torch.randn(2048, device="cuda")).to(torch.bfloat16)
    b2 = (0.1 * torch.randn(2048, device="cuda")).to(torch.bfloat16)
    x1 = torch.randn(512, 1024, device="cuda").to(torch.bfloat16)
    x2 = torch.randn(2048, 2048, device="cuda").to(torch.bfloat16)
    assert bsq.bsq_test_inject_stall(bsq.KERNEL_LAYERNORM, 0, LIMIT_NS) == bsq.OK
    bsq.layernorm_quantize("mxfp8", x1, g1, b1, 1e-6)
    assert bsq.device_status() == bsq.OK
    bsq.layernorm_quantize("mxfp8", x2, g2, b2, 1e-6)
    assert bsq.device_status() == bsq.ERR_TIMEOUT
    bsq.layernorm_quantize("mxfp8", x2, g2, b2, 1e-6)
    assert bsq.device_status() == bsq.OK
