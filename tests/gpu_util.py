"""Helpers for the GPU parity tests: numpy <-> torch transfer and oracle row sampling."""
import numpy as np
import torch

import oracle


def to_dev(a: np.ndarray) -> torch.Tensor:
    """uint16 arrays become bf16 tensors (same bits); float32 stays float32; uint8 stays uint8."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def sample_rows(M: int, seed: int = 0, per_tile: int = 2) -> np.ndarray:
    """First and last row of every 128-row tile plus `per_tile` random rows of each tile."""
    rng = np.random.default_rng(seed)
    rows = set()
    for t0 in range(0, M, 128):
        t1 = min(M, t0 + 128)
        rows.update([t0, t1 - 1])
        rows.update(int(r) for r in rng.integers(t0, t1, size=per_tile))
    return np.array(sorted(rows), dtype=np.int64)


def decode_rows(q: "oracle.Quantized", idx: np.ndarray) -> np.ndarray:
    """Decode only the rows `idx` of an oracle-quantized matrix (fp64, NVFP4 without g)."""
    per_row = q.codes.size // q.rows
    codes = q.codes.reshape(q.rows, per_row)[idx]
    return oracle.decode(q.fmt, codes, q.scales[idx], len(idx), q.cols)


def check_gemm_rows(got: np.ndarray, qa, qb, bias, idx: np.ndarray, what: str = ""):
    """Compare GPU output rows `idx` against the oracle's fp64 GEMM on those rows, with the
    tolerance |gpu - y| <= 2^-7 |y| + 1e-5 sum_k |a b|."""
    A = decode_rows(qa, idx)
    B = qb.decode()
    alpha = qa.g * qb.g if qa.fmt == oracle.NVFP4 else 1.0
    want, absum = oracle.gemm(A, B, bias, alpha)
    tol = 2.0 ** -7 * np.abs(want) + 1e-5 * absum
    err = np.abs(got - want)
    bad = err > tol
    assert not bad.any(), "%s: %d of %d outputs out of tolerance; worst err/tol %.3g at %s" % (
        what, int(bad.sum()), bad.size, float((err / np.maximum(tol, 1e-300)).max()),
        np.unravel_index(int(np.argmax(err / np.maximum(tol, 1e-300))), err.shape))
    return float((err / np.maximum(tol, 1e-300)).max())


# --------------------------------------------------------------------- MX codes within a band
E4M3 = None
E2M1 = None


def _tables():
    global E4M3, E2M1
    if E4M3 is None:
        E4M3 = np.array([oracle.decode_e4m3(c) for c in range(256)])
        E2M1 = np.array([oracle.decode_e2m1(c) for c in range(16)])
    return E4M3, E2M1


def plain_scales(tiled: np.ndarray, rows: int, cols: int, row_idx=None) -> np.ndarray:
    """Plain (rows x cols/32) scale bytes read out of a tiled MX scale buffer."""
    nsc = cols // 32
    rr = range(rows) if row_idx is None else row_idx
    off = np.array([[oracle.scale_tiled_offset(int(r), c, nsc) for c in range(nsc)] for r in rr])
    return tiled[off]


def element_codes(out_fmt, codes: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """One code per element (e2m1 nibbles unpacked, element 2j in the low nibble)."""
    if out_fmt == "mxfp8":
        return codes.reshape(rows, cols)
    c = codes.reshape(rows, cols // 2)
    out = np.empty((rows, cols), dtype=np.uint8)
    out[:, 0::2] = c & 0xF
    out[:, 1::2] = c >> 4
    return out


def _mx_exponent(amax: np.ndarray, emax: int) -> np.ndarray:
    _, ex = np.frexp(amax)
    return np.clip(np.where(amax > 0, ex - 1 - emax, -127), -127, 127)


def check_mx_band(out_fmt, codes_el: np.ndarray, scales_plain: np.ndarray, exact: np.ndarray, band: np.ndarray,
                  min_match: float = 0.99):
    """MX codes / scales of values the kernel computed in fp32 against the exact values: every
    block scale must be the MX exponent of some block maximum inside exact +- band, every code
    the encoding (at the kernel's scale) of some value inside the band, and at least
    `min_match` of codes and scales must equal those of the exact values."""
    rows, cols = exact.shape
    emax = 8 if out_fmt == "mxfp8" else 2
    e4, e2 = _tables()
    tbl = e4 if out_fmt == "mxfp8" else e2
    Gb, Bb = np.abs(exact).reshape(rows, -1, 32), band.reshape(rows, -1, 32)
    e_lo = _mx_exponent(np.maximum(Gb - Bb, 0).max(-1), emax)
    e_hi = _mx_exponent((Gb + Bb).max(-1), emax)
    e_gpu = scales_plain.astype(np.int64) - 127
    assert ((e_lo <= e_gpu) & (e_gpu <= e_hi)).all(), "block scales outside the band"
    scale = np.repeat(np.exp2(e_gpu.astype(np.float64)), 32, axis=1)
    elem = "e4m3" if out_fmt == "mxfp8" else "e2m1"
    d_lo = tbl[oracle.encode_array(elem, (exact - band) / scale)]
    d_hi = tbl[oracle.encode_array(elem, (exact + band) / scale)]
    d = tbl[codes_el]
    bad = ~((d_lo <= d) & (d <= d_hi))
    assert not bad.any(), "%d of %d codes outside the band (first at %s)" % (
        int(bad.sum()), bad.size, np.unravel_index(int(np.argmax(bad)), bad.shape))
    ref = oracle.quantize_mx_f64(out_fmt, exact)
    ref_codes = element_codes(out_fmt, ref.codes, rows, cols)
    code_match = float((ref_codes == codes_el).mean())
    scale_match = float((ref.scales == scales_plain).mean())
    assert code_match >= min_match and scale_match >= min_match, (code_match, scale_match)
    return code_match, scale_match
