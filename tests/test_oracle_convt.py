"""Pins of the oracle's kernel-2 stride-2 transposed convolution (reading R13): a library
transposed convolution (torch, fp64, CPU) on random operands, and a hand-derived case."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("batch,H,W,Cin,Cout", [(1, 1, 1, 3, 2), (2, 3, 5, 8, 4), (1, 4, 2, 16, 8)])
@pytest.mark.parametrize("gelu", [False, True])
def test_convt_matches_library_transposed_convolution(batch, H, W, Cin, Cout, gelu):
    rng = np.random.default_rng(batch * 100 + H * 10 + W)
    x = rng.standard_normal((batch, H, W, Cin))                       # NHWC input
    wt = rng.standard_normal((Cin, Cout, 2, 2))                       # ConvTranspose2d weight layout
    bias_f = (rng.standard_normal(Cout) * 0.1).astype(np.float32)
    bias_bits = (bias_f.view(np.uint32) >> 16).astype(np.uint16)      # exact bf16 (truncated values)
    bias_v = (bias_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    A = x.reshape(batch * H * W, Cin)
    B = np.ascontiguousarray(wt.transpose(2, 3, 1, 0).reshape(4 * Cout, Cin))  # row (2 dy + dx) Cout + co
    got = oracle.convt2x2(A, B, bias_bits, batch, H, W, alpha=1.0, gelu=gelu)
    ref = torch.nn.functional.conv_transpose2d(torch.from_numpy(x.transpose(0, 3, 1, 2).copy()),
                                               torch.from_numpy(wt), torch.from_numpy(bias_v), stride=2)
    if gelu:
        ref = torch.nn.functional.gelu(ref)
    ref = ref.numpy().transpose(0, 2, 3, 1)
    assert got.shape == ref.shape
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_convt_single_pixel_by_hand():
    # one input pixel with channels (1, 2); output channel co at tap (dy, dx) weighs
    # w[(2 dy + dx) * Cout + co] = (dy + 1) * (dx + 2) * (co + 1) on both input channels
    Cout = 2
    A = np.array([[1.0, 2.0]])
    B = np.array([[(dy + 1) * (dx + 2) * (co + 1)] * 2 for dy in (0, 1) for dx in (0, 1) for co in range(Cout)],
                 dtype=np.float64)
    out = oracle.convt2x2(A, B, None, 1, 1, 1, alpha=0.5)
    for dy in (0, 1):
        for dx in (0, 1):
            for co in range(Cout):
                assert out[0, dy, dx, co] == 0.5 * 3.0 * (dy + 1) * (dx + 2) * (co + 1)
