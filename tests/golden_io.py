"""Reader for the hand-derived fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, vals = line.split(":", 1)
            out[key.strip()] = vals.split()
    return out


def floats(tokens):
    return np.array([float(t) for t in tokens], dtype=np.float64)


def ints(tokens):
    return np.array([int(t, 0) for t in tokens], dtype=np.int64)


def block_rows(fix, block):
    """Blocks x0, x1, ... (each padded with zeros to `block` elements), their codes c_i and
    scales s_i, in order."""
    i = 0
    xs, cs, ss = [], [], []
    while "x%d" % i in fix:
        x = np.zeros(block)
        c = np.zeros(block, dtype=np.int64)
        xv, cv = floats(fix["x%d" % i]), ints(fix["c%d" % i])
        x[: len(xv)] = xv
        c[: len(cv)] = cv
        # a padded zero keeps +0 -> code 0; listed -0.0 entries carry their sign
        xs.append(x)
        cs.append(c)
        ss.append(ints(fix["s%d" % i])[0])
        i += 1
    return xs, cs, ss
