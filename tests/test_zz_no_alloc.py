"""The split-K GEMM whose workspace is the library's fixed device array (bsq_gemm_splitk_scratch)
against bsq_gemm_splitk with a caller workspace: the same kernels on the same operands, so the
outputs must be identical -- on two calls in a row with different operands (nothing carried over
from the first), with one range (no workspace), and with requests over the array's 64 MiB
refused."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _bsq():
    import block_scaled_precision_bsq_gb300 as bsq

    return bsq


def _operands(fmt, M, N, K, seed):
    bsq = _bsq()
    g = torch.Generator(device="cuda").manual_seed(seed)
    qa = bsq.quantize(fmt, torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16))
    qb = bsq.quantize(fmt, (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16))
    bias = (torch.randn(N, device="cuda", generator=g) * 0.1).to(torch.bfloat16)
    return qa, qb, bias


def _scratch(qa, qb, bias, out, splits):
    bsq = _bsq()
    M, K, N = qa.rows, qa.cols, qb.rows
    return bsq.bsq_gemm_splitk_scratch(qa.fmt, qa.codes, qa.scales, qb.codes, qb.scales, bias, out, M, N, K, splits)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_scratch_matches_caller_workspace_on_two_calls_in_a_row(fmt):
    bsq = _bsq()
    # ViT-B/16 fc1's weight gradient shape (2 ranges), then a smaller one with 3 ranges
    for (M, N, K, splits), seed in (((3072, 768, 14336, 2), 1), ((640, 520, 4096, 3), 2)):
        qa, qb, bias = _operands(fmt, M, N, K, seed)
        want = bsq.gemm_splitk(qa, qb, bias, splits=splits)
        got = torch.empty_like(want)
        assert _scratch(qa, qb, bias, got, splits) == bsq.OK
        assert bsq.device_status() == 0
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), (M, N, K, splits)


def test_scratch_one_range_and_size_limit():
    bsq = _bsq()
    qa, qb, bias = _operands("mxfp8", 4096, 4096, 256, 3)
    out = torch.empty(4096, 4096, dtype=torch.bfloat16, device="cuda")
    # 2 x 4096 x 4096 fp32 = 128 MiB: over the array
    assert _scratch(qa, qb, bias, out, 2) == bsq.ERR_ARG
    # one range needs no workspace: bsq_gemm's result
    assert _scratch(qa, qb, bias, out, 1) == bsq.OK
    want = bsq.gemm(qa, qb, bias)
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))
    assert bsq.device_status() == 0


def test_scratch_request_that_fills_the_array_exactly():
    """2 x 4096 x 2048 fp32 partial sums are exactly the array's 64 MiB: the last slice's top edge
    is the array's last byte. The result must equal the caller-workspace split-K bit for bit; a
    request 8 columns wider no longer fits and is refused before anything is enqueued."""
    bsq = _bsq()
    M, N, K, splits = 4096, 2048, 256, 2
    assert splits * M * N * 4 == 64 << 20
    qa, qb, bias = _operands("mxfp8", M, N, K, 4)
    want = bsq.gemm_splitk(qa, qb, bias, splits=splits)
    got = torch.empty_like(want)
    assert _scratch(qa, qb, bias, got, splits) == bsq.OK
    assert bsq.device_status() == 0
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    qa2, qb2, bias2 = _operands("mxfp8", M, N + 8, K, 5)
    out2 = torch.empty(M, N + 8, dtype=torch.bfloat16, device="cuda")
    assert _scratch(qa2, qb2, bias2, out2, splits) == bsq.ERR_ARG
    assert bsq.device_status() == 0
