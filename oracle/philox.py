"""Philox4x64-10 counter-based generator (Salmon, Moraes, Dror, Shaw, "Parallel random
numbers: as easy as 1, 2, 3", SC'11), used for the BigBird random blocks.

The BigBird page (section 2, "Random attention G_R") draws r keys per query uniformly;
its sketch (section 3) uses torch.randperm. To make the draw reproducible on two
independent implementations, the random stream is fixed as follows (a reading of the
page, which names no generator):

  word(p) = Philox4x64_10(counter = (p // 4 + 1, 0, 0, 0), key = (seed, 0))[p % 4]

i.e. the raw 64-bit output stream of numpy's ``Philox(key=seed)`` bit generator. Draw
t of query block I uses word(I * r_b + t). The tests pin this function against
numpy's implementation.
"""
from __future__ import annotations

MASK64 = (1 << 64) - 1
_M0 = 0xD2E7470EE14C6C93   # Philox4x64 round multipliers (SC'11, Table 2)
_M1 = 0xCA5A826395121157
_W0 = 0x9E3779B97F4A7C15   # Weyl key increments (golden ratio, sqrt(3)-1)
_W1 = 0xBB67AE8584CAA73B


def _mulhilo(a: int, b: int) -> tuple[int, int]:
    prod = a * b
    return (prod >> 64) & MASK64, prod & MASK64


def philox4x64_10(counter: tuple[int, int, int, int], key: tuple[int, int]) -> list[int]:
    """One Philox4x64 block with 10 rounds; returns four 64-bit words."""
    c0, c1, c2, c3 = (int(x) & MASK64 for x in counter)
    k0, k1 = (int(x) & MASK64 for x in key)
    for _ in range(10):
        hi0, lo0 = _mulhilo(_M0, c0)
        hi1, lo1 = _mulhilo(_M1, c2)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + _W0) & MASK64
        k1 = (k1 + _W1) & MASK64
    return [c0, c1, c2, c3]


def philox_word(seed: int, p: int) -> int:
    """Word ``p`` of the raw 64-bit stream for ``seed``."""
    block = philox4x64_10((p // 4 + 1, 0, 0, 0), (seed & MASK64, 0))
    return block[p % 4]
