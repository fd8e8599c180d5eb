"""Exact T5 bucket ids from integer E-th roots (threshold form), for tests only.

A distance n >= me lands in bucket me + t, t the largest integer <= E-1 with
n >= me * (md/me)^(t/E), i.e. n^E >= me^(E-t) * md^t. Computed with Python integers.
"""


def iroot_ceil(x: int, e: int) -> int:
    """Smallest integer n with n**e >= x."""
    lo, hi = 0, 1
    while hi ** e < x:
        hi *= 2
    while lo < hi:
        mid = (lo + hi) // 2
        if mid ** e >= x:
            hi = mid
        else:
            lo = mid + 1
    return lo


def exact_thresholds(nbh: int, md: int):
    me = nbh // 2
    E = nbh - me
    return [iroot_ceil(me ** (E - t) * md ** t, E) for t in range(1, E)]


_cache = {}


def exact_bucket(delta: int, nb: int, md: int, bidir: bool) -> int:
    nbh = nb // 2 if bidir else nb
    off = nbh if (bidir and delta > 0) else 0
    n = abs(delta) if bidir else max(-delta, 0)
    me = nbh // 2
    if n < me:
        return off + n
    key = (nbh, md)
    if key not in _cache:
        _cache[key] = exact_thresholds(nbh, md)
    t = sum(1 for th in _cache[key] if n >= th)
    return off + me + t
