"""A second, independent restatement of attention in pure Python.

Used only to pin the C++ oracle on tiny inputs: exact softmax(scale q.K^T) V
with ``math.fsum`` sums, on already-contiguous keys and values (the formula in
"Chapter 1: attention backends", section 2.1).  It shares nothing with the
oracle or the CUDA library.
"""

import math


def attend(q, keys, values, scale):
    """q: list[float]; keys, values: list of rows.  Returns (o, lse)."""
    n = len(keys)
    dv = len(values[0]) if n else 0
    if n == 0:
        return [0.0] * dv, -math.inf
    s = [scale * math.fsum(a * b for a, b in zip(q, k)) for k in keys]
    m = max(s)
    w = [math.exp(x - m) for x in s]
    l = math.fsum(w)
    o = [math.fsum(w[p] * values[p][e] for p in range(n)) / l for e in range(dv)]
    return o, m + math.log(l)
