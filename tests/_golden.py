"""Reader for the hand-derived text fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    """Parse ``key = v v v; v v v`` lines; '#' starts a comment. Returns str -> ndarray."""
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, _, val = line.partition("=")
            rows = [r.split() for r in val.split(";")]
            if len(rows) == 1:
                out[key.strip()] = np.array([float(x) for x in rows[0]], dtype=np.float64)
            else:
                out[key.strip()] = np.array([[float(x) for x in r] for r in rows], dtype=np.float64)
    return out


def ints(a) -> list:
    return [int(x) for x in np.atleast_1d(a)]


def num(a) -> float:
    """The single value of a one-number entry."""
    a = np.asarray(a).reshape(-1)
    assert a.size == 1
    return float(a[0])


def i(a) -> int:
    return int(num(a))
