"""Per-block compression ratio ([CAS] section 3.1, Eq. 1; Algorithm 1 step 1).

r_i = |compress(x[i*b:(i+1)*b])| / b

[CAS] uses gzip at level 1 and b = 128; the workloads here use zlib framing at level
6 and b in {32, 64, 128}. gzip and zlib wrap the same deflate stream; they differ only
by a constant number of header/trailer bytes (pinned in the tests), so the ordering of
ratios and the mean-threshold decision are the same under either framing.

The ratio is returned as float32: the compressed length is an integer below 2^24 and b
is a power of two, so the quotient is exact in float32 (a dyadic rational).

Reading: [CAS] states r_i is in (0, 1]; for small blocks of random bytes the deflate
output is longer than the input, so r_i > 1 occurs and is permitted here.
"""
from __future__ import annotations

import zlib

import numpy as np


def zlib_version() -> str:
    return zlib.ZLIB_RUNTIME_VERSION


def block_ratios(data: np.ndarray, block: int, level: int = 6) -> np.ndarray:
    """Ratios ``float32[batch, nb]`` of a ``uint8[batch, N]`` byte array (or 1-D)."""
    arr = np.asarray(data, dtype=np.uint8)
    squeeze = arr.ndim == 1
    if squeeze:
        arr = arr[None, :]
    bt, n = arr.shape
    if n % block != 0:
        raise ValueError("sequence length must be a multiple of the block size")
    nb = n // block
    out = np.empty((bt, nb), dtype=np.float32)
    for s in range(bt):
        for i in range(nb):
            chunk = arr[s, i * block:(i + 1) * block].tobytes()
            out[s, i] = np.float32(len(zlib.compress(chunk, level)) / block)
    return out[0] if squeeze else out
