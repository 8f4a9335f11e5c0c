"""Shared test helpers (no method arithmetic)."""
import numpy as np


def max_rel(x, y):
    """max |x - y| / max |y| over a tensor, in FP64 (the tolerance measure used
    throughout the parity tests)."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    denom = np.max(np.abs(y)) if y.size else 0.0
    if y.size == 0:
        return 0.0
    if denom == 0.0:
        return float(np.max(np.abs(x - y)))
    return float(np.max(np.abs(x - y)) / denom)
