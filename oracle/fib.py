"""Fibonacci offsets with a per-layer scale ([FIB] section 2 "Method").

* Rungs: f = 1, 2, 3, 5, 8, ..., 987 (K = 15) in [FIB]; the workload statement instead
  allows every f_k <= N. Both are available (``fib_rungs(K)`` / ``fib_rungs_upto(N)``).
* Linear stagger: alpha_l = alpha_lo + (alpha_hi - alpha_lo) * l / (L - 1), held as an
  exact fraction ([FIB]: 0.5 -> 1.5; the workload statement: 0.5 -> 2.0).
* Offsets d_k = round(alpha * f_k). Reading: [FIB] only says the fixed and staggered
  variants have integer offsets; "round" is taken as round-half-to-even (Python and
  torch ``round``). Ties occur (alpha = 1/2 with odd f).
* Key set of query i: { i - delta : delta in {0, ..., W} u D, i - delta >= 0 } as a set
  (the union is deduplicated; offsets inside the window add nothing).
* Coprime stagger ([FIB] section 2 "The per-layer scalar"): the linear ramp's values
  reassigned to layers by l -> (S l mod L), S = 7. Reading: layer l takes the ramp
  value at index (S l) mod L. For L = 16, S = 7 is its own inverse (7 * 7 = 49 = 1 mod
  16), so the other reading (ramp index l goes to layer S l mod L) is the same map.
* Power-of-2 control base ([FIB] section 2 "Control base"): rungs 1, 2, 4, ..., "reach
  matched" to the Fibonacci base. Reading: 11 rungs up to 1024, the power of two the
  page itself equates with f_15 = 987 ("987 ~ 1024"); ``pow2_rungs_upto(N)`` is the
  every-rung-up-to-N variant.
"""
from __future__ import annotations

import math
from fractions import Fraction


def fib_rungs(n_rungs: int = 15) -> list[int]:
    out = []
    a, b = 1, 2
    for _ in range(n_rungs):
        out.append(a)
        a, b = b, a + b
    return out


def fib_rungs_upto(n: int) -> list[int]:
    out = []
    a, b = 1, 2
    while a <= n:
        out.append(a)
        a, b = b, a + b
    return out


def pow2_rungs(n_rungs: int = 11) -> list[int]:
    return [2 ** k for k in range(n_rungs)]


def pow2_rungs_upto(n: int) -> list[int]:
    out = []
    a = 1
    while a <= n:
        out.append(a)
        a *= 2
    return out


def alpha_schedule(layers: int, lo=(1, 2), hi=(3, 2), stride: int = 1) -> list[Fraction]:
    """Per-layer alpha: the linear ramp lo -> hi over ``layers`` layers; with
    ``stride`` S > 1 layer l takes the ramp value at index (S l) mod L (coprime
    stagger; S must be coprime to L)."""
    a_lo = Fraction(*lo)
    a_hi = Fraction(*hi)
    if layers == 1:
        return [a_lo]
    ramp = [a_lo + (a_hi - a_lo) * Fraction(l, layers - 1) for l in range(layers)]
    if stride == 1:
        return ramp
    if math.gcd(stride, layers) != 1:
        raise ValueError("the stagger stride must be coprime to the layer count")
    return [ramp[(stride * l) % layers] for l in range(layers)]


def fib_offsets(alpha: Fraction, rungs: list[int]) -> list[int]:
    """Sorted distinct d_k = round_half_even(alpha * f_k)."""
    return sorted({round(Fraction(alpha) * f) for f in rungs})


def offset_key_set(i: int, window: int, offsets: list[int]) -> list[int]:
    deltas = set(range(window + 1)) | set(offsets)
    return sorted({i - d for d in deltas if i - d >= 0})


def interp_rungs(alpha: float, rungs: list[int], window: int) -> list[tuple[int, float]]:
    """Rungs of the interpolated gather ([FIB] section 2 "Attended set"): the distance
    d_k = alpha * f_k is continuous (the IEEE double product), and the gathered key and
    value are the linear interpolation between rows i - floor(d_k) and i - floor(d_k) - 1
    with weight t_k = d_k - floor(d_k) on the farther row. Returns (floor(d_k), t_k) per
    rung kept. Reading: a rung whose distance is an integer inside the window is the same
    key as a window row and is dropped, so that integer alphas give exactly the
    integer-offset key set (the page states the gather and the boolean-mask paths agree
    for integer offsets, section 2 "Implementation note")."""
    out = []
    for f in rungs:
        d = float(alpha) * float(f)
        lo = math.floor(d)
        t = d - lo
        if t == 0.0 and lo <= window:
            continue
        out.append((int(lo), float(t)))
    return out
