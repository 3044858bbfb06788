"""Brute-force references used only by the tests to pin the oracle.

Nearest-value search over an explicit table of a format's values: no exponent
arithmetic, so it shares no reasoning with the oracle's encoder.
"""
import numpy as np


def value_table(decode, n_codes, sign_bit):
    """(codes, values) of every finite non-negative code, values ascending."""
    codes, vals = [], []
    for c in range(n_codes):
        if c & sign_bit:
            continue
        v = decode(c)
        if np.isfinite(v):
            codes.append(c)
            vals.append(v)
    order = np.argsort(vals, kind="stable")
    return np.array(codes)[order], np.array(vals, dtype=np.float64)[order]


def nearest_even(v, codes, vals, sign_bit, chunk=65536):
    """Round each v to the nearest table value; exact ties go to the even code; beyond
    the largest value, saturate; the sign is copied from v (also for zero results)."""
    v = np.asarray(v, dtype=np.float64).reshape(-1)
    out = np.empty(v.shape, dtype=np.int64)
    vmax = vals[-1]
    for s in range(0, v.size, chunk):
        a = np.abs(v[s:s + chunk])
        d = np.abs(a[:, None] - vals[None, :])          # distance to every value
        dmin = d.min(axis=1, keepdims=True)
        cand = d == dmin                                  # one or two nearest values
        odd = (codes[None, :] & 1).astype(bool)
        # among the nearest, prefer even codes
        pick_even = cand & ~odd
        has_even = pick_even.any(axis=1)
        idx = np.where(has_even, pick_even.argmax(axis=1), cand.argmax(axis=1))
        mag = codes[idx]
        mag = np.where(a >= vmax, codes[-1], mag)
        sign = np.signbit(v[s:s + chunk])
        out[s:s + chunk] = np.where(sign, mag | sign_bit, mag)
    return out


def all_bf16_values():
    """Every finite bf16 value as float64 (65536 patterns minus inf/nan)."""
    bits = np.arange(65536, dtype=np.uint32)
    f32 = (bits << 16).view(np.float32)
    return f32[np.isfinite(f32)].astype(np.float64)
