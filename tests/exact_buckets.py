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


def exact_bucket_array(deltas, nb: int, md: int, bidir: bool):
    """exact_bucket over a numpy array of deltas: the thresholds come from the integer roots
    above, the count of thresholds <= n from a sorted search."""
    import numpy as np
    deltas = np.asarray(deltas, dtype=np.int64)
    nbh = nb // 2 if bidir else nb
    me = nbh // 2
    thr = np.asarray(exact_thresholds(nbh, md), dtype=np.int64)
    if bidir:
        off = np.where(deltas > 0, nbh, 0)
        n = np.abs(deltas)
    else:
        off = np.zeros_like(deltas)
        n = np.maximum(-deltas, 0)
    t = np.searchsorted(thr, n, side="right")
    return off + np.where(n < me, n, me + t)
