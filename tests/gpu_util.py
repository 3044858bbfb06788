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
