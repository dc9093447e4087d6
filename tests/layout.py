"""Storage helpers for tests: place a logical matrix into a padded, optionally
transposed row-major buffer (data movement only, no arithmetic)."""

import numpy as np


def store(logical, trans, ld, pad=np.nan):
    """Return a flat float32 buffer holding ``logical`` (rows x cols) row-major
    with leading dimension ``ld``; when ``trans`` is 1 the buffer holds the
    transpose (cols x rows).  Padding columns are filled with ``pad`` so a
    kernel or oracle that ignores ``ld`` reads garbage and fails."""
    m = np.asarray(logical, dtype=np.float32)
    if trans:
        m = m.T
    r, c = m.shape
    assert ld >= max(1, c)
    buf = np.full((max(r, 1), ld), pad, dtype=np.float32)
    buf[:r, :c] = m
    return np.ascontiguousarray(buf[:r].reshape(-1) if r else np.zeros(0, np.float32))


def stored_ld(rows, cols, trans, extra=0):
    """Smallest legal leading dimension for a rows x cols logical operand, plus ``extra``."""
    return max(1, (rows if trans else cols)) + extra


def unstore(buf, rows, cols, ld):
    """Read a rows x cols row-major matrix back out of a flat buffer with leading dimension ld."""
    flat = np.asarray(buf).reshape(-1)
    out = np.empty((rows, cols), dtype=flat.dtype)
    for r in range(rows):
        out[r] = flat[r * ld: r * ld + cols]
    return out
