"""No kernel writes outside its output buffers. Every output is a slice of a larger buffer filled
with a sentinel byte; after the call the bytes before and after each slice are unchanged, and the
results equal those of the same call into freshly allocated buffers (the kernels are
deterministic). Ragged shapes put the last row tiles, scale padding and store boxes at the edges
of their buffers."""
import pytest
import torch

pytestmark = pytest.mark.gpu

G = 4096         # guard bytes on each side (keeps the slice 16-byte aligned)
SENTINEL = 0xA5


def _bsq():
    import block_scaled_precision_bsq_gb300 as bsq

    return bsq


class Guarded:
    """A uint8 slice of `nbytes` inside a sentinel-filled buffer with G guard bytes on each side."""

    def __init__(self, nbytes: int):
        self.buf = torch.full((nbytes + 2 * G,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.n = nbytes
        self.t = self.buf[G:G + nbytes]

    def intact(self) -> bool:
        return bool((self.buf[:G] == SENTINEL).all()) and bool((self.buf[G + self.n:] == SENTINEL).all())


def _guarded_qtensor(fmt, rows, cols):
    bsq = _bsq()
    f = bsq._fmt(fmt)
    codes = Guarded(bsq.bsq_codes_bytes(f, rows, cols))
    scales = Guarded(bsq.bsq_scales_bytes(f, rows, cols))
    g = Guarded(4) if f == bsq.NVFP4 else None
    q = bsq.QTensor(f, rows, cols, codes.t, scales.t, None if g is None else g.t.view(torch.float32))
    return q, [codes, scales] + ([g] if g is not None else [])


def _same(a, b):
    return torch.equal(a.contiguous().reshape(-1).view(torch.uint8), b.contiguous().reshape(-1).view(torch.uint8))


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,cols", [(1, 32), (130, 96), (257, 160), (33, 2080)])
def test_quantize_stays_inside_codes_and_scales(fmt, dtype, rows, cols):
    bsq = _bsq()
    x = torch.randn(rows, cols, device="cuda", generator=torch.Generator(device="cuda").manual_seed(rows + cols))
    x = (x * 3).to(dtype)
    q, guards = _guarded_qtensor(fmt, rows, cols)
    bsq.quantize(fmt, x, out=q)
    ref = bsq.quantize(fmt, x)
    assert bsq.device_status() == 0
    assert all(g.intact() for g in guards)
    assert _same(q.codes, ref.codes) and _same(q.scales, ref.scales)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("stochastic", [False, True])
@pytest.mark.parametrize("rows,cols", [(32, 32), (96, 160), (160, 96), (288, 64)])
def test_dual_stays_inside_both_layouts(fmt, stochastic, rows, cols):
    bsq = _bsq()
    x = (torch.randn(rows, cols, device="cuda", generator=torch.Generator(device="cuda").manual_seed(rows * cols))
         * 2).to(torch.bfloat16)
    qr, gr = _guarded_qtensor(fmt, rows, cols)
    qc, gc = _guarded_qtensor(fmt, cols, rows)
    bsq.quantize_dual(fmt, x, stochastic=stochastic, seed=5, out=(qr, qc))
    rr, rc = bsq.quantize_dual(fmt, x, stochastic=stochastic, seed=5)
    assert bsq.device_status() == 0
    assert all(g.intact() for g in gr + gc)
    assert _same(qr.codes, rr.codes) and _same(qr.scales, rr.scales)
    assert _same(qc.codes, rc.codes) and _same(qc.scales, rc.scales)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("rows,cols", [(7, 1024), (130, 768), (3, 2048)])
def test_layernorm_quantize_stays_inside(fmt, rows, cols):
    bsq = _bsq()
    gen = torch.Generator(device="cuda").manual_seed(rows + 3 * cols)
    x = torch.randn(rows, cols, device="cuda", generator=gen).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(cols, device="cuda", generator=gen)).to(torch.bfloat16)
    beta = (0.1 * torch.randn(cols, device="cuda", generator=gen)).to(torch.bfloat16)
    q, guards = _guarded_qtensor(fmt, rows, cols)
    bsq.layernorm_quantize(fmt, x, gamma, beta, out=q)
    ref = bsq.layernorm_quantize(fmt, x, gamma, beta)
    assert bsq.device_status() == 0
    assert all(g.intact() for g in guards)
    assert _same(q.codes, ref.codes) and _same(q.scales, ref.scales)


def _operands(fmt, M, N, K, seed):
    bsq = _bsq()
    gen = torch.Generator(device="cuda").manual_seed(seed)
    qa = bsq.quantize(fmt, torch.randn(M, K, device="cuda", generator=gen).to(torch.bfloat16))
    qb = bsq.quantize(fmt, (0.05 * torch.randn(N, K, device="cuda", generator=gen)).to(torch.bfloat16))
    bias = (0.1 * torch.randn(N, device="cuda", generator=gen)).to(torch.bfloat16)
    return qa, qb, bias


@pytest.mark.parametrize("fmt,out_fmt", [("mxfp8", "mxfp8"), ("mxfp8", "mxfp4"), ("nvfp4", "mxfp8"), ("mxfp4", "mxfp4")])
def test_gemm_gelu_quantize_stays_inside(fmt, out_fmt):
    bsq = _bsq()
    M, N, K = 300, 288, 512
    qa, qb, bias = _operands(fmt, M, N, K, 11)
    q, guards = _guarded_qtensor(out_fmt, M, N)
    bsq.gemm_gelu_quantize(qa, qb, bias, out_fmt=out_fmt, out=q)
    ref = bsq.gemm_gelu_quantize(qa, qb, bias, out_fmt=out_fmt)
    assert bsq.device_status() == 0
    assert all(g.intact() for g in guards[:2])
    assert _same(q.codes, ref.codes) and _same(q.scales, ref.scales)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_gemm_and_splitk_stay_inside_output_and_workspace(fmt):
    bsq = _bsq()
    M, N, K = 300, 264, 2048
    qa, qb, bias = _operands(fmt, M, N, K, 12)
    out = Guarded(M * N * 2)
    bsq.gemm(qa, qb, bias, out=out.t.view(torch.bfloat16).view(M, N))
    ref = bsq.gemm(qa, qb, bias)
    assert out.intact() and _same(out.t, ref)
    ws = Guarded(3 * M * N * 4)
    out2 = Guarded(M * N * 2)
    bsq.gemm_splitk(qa, qb, bias, splits=3, workspace=ws.t.view(torch.float32),
                    out=out2.t.view(torch.bfloat16).view(M, N))
    ref2 = bsq.gemm_splitk(qa, qb, bias, splits=3)
    assert bsq.device_status() == 0
    assert ws.intact() and out2.intact() and _same(out2.t, ref2)


def test_convt_stays_inside_output():
    bsq = _bsq()
    B, H, W, Ci, Co = 2, 3, 4, 256, 64
    qx, qw, _ = _operands("mxfp8", B * H * W, 4 * Co, Ci, 13)
    bias = (0.1 * torch.randn(Co, device="cuda")).to(torch.bfloat16)
    out = Guarded(B * 2 * H * 2 * W * Co * 2)
    bsq.convt2x2(qx, qw, B, H, W, bias, gelu=True, out=out.t.view(torch.bfloat16).view(B, 2 * H, 2 * W, Co))
    ref = bsq.convt2x2(qx, qw, B, H, W, bias, gelu=True)
    assert bsq.device_status() == 0
    assert out.intact() and _same(out.t, ref)


def _offset_copy(x: torch.Tensor, offset_bytes: int) -> torch.Tensor:
    """x's values in a tensor whose data starts `offset_bytes` past a 256-byte boundary (16-byte
    aligned, not 32): the kernels' 16-byte load path."""
    n = x.numel() * x.element_size()
    buf = torch.empty(n + 256, dtype=torch.uint8, device=x.device)
    y = buf[offset_bytes:offset_bytes + n].view(x.dtype).view(x.shape)
    y.copy_(x)
    assert y.data_ptr() % 32 == offset_bytes % 32
    return y


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_source_aligned_to_16_bytes_only(fmt, dtype):
    """A source 16-byte aligned but not 32 takes the 16-byte loads: the same bytes as from an
    aligned copy (ragged rows, NVFP4 both per-tensor scale modes)."""
    bsq = _bsq()
    x = (torch.randn(257, 160, device="cuda", generator=torch.Generator(device="cuda").manual_seed(3)) * 3).to(dtype)
    y = _offset_copy(x, 16)
    a, b = bsq.quantize(fmt, x), bsq.quantize(fmt, y)
    assert bsq.device_status() == 0
    assert _same(a.codes, b.codes) and _same(a.scales, b.scales)
    if fmt == "nvfp4":
        g = torch.tensor([0.01], dtype=torch.float32, device="cuda")
        a, b = bsq.quantize(fmt, x, global_scale=g), bsq.quantize(fmt, y, global_scale=g)
        assert bsq.device_status() == 0
        assert _same(a.codes, b.codes) and _same(a.scales, b.scales)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("cols", [768, 1024, 2048])
def test_layernorm_source_aligned_to_16_bytes_only(fmt, cols):
    """The same for LayerNorm + quantize, on both of its kernels (rows of at most 1024 bf16 run the
    streaming one)."""
    bsq = _bsq()
    gen = torch.Generator(device="cuda").manual_seed(cols)
    x = (torch.randn(131, cols, device="cuda", generator=gen) * 3 + 1).to(torch.bfloat16)
    g = (1 + 0.1 * torch.randn(cols, device="cuda", generator=gen)).to(torch.bfloat16)
    b = (0.1 * torch.randn(cols, device="cuda", generator=gen)).to(torch.bfloat16)
    y = _offset_copy(x, 16)
    p, q = bsq.layernorm_quantize(fmt, x, g, b, 1e-6), bsq.layernorm_quantize(fmt, y, g, b, 1e-6)
    assert bsq.device_status() == 0
    assert _same(p.codes, q.codes) and _same(p.scales, q.scales)
