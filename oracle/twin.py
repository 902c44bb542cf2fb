"""Pure-Python brute-force twin of the oracle, for tiny shapes only.

TEST INFRASTRUCTURE ONLY.  A second, independent statement of masked softmax
attention written with Python floats and ``math`` (no numpy, no C), used to
cross-check the C oracle.  Softmax here is computed as explicit normalised
weights w_n = exp(z_n - max) / sum_m exp(z_m - max), a different evaluation
order from the C code's ``exp(z - lse)``, so a slip in either shows up.
"""
from __future__ import annotations

import math


def attend_row(qrow, keys, values, scale):
    """One query row over a list of visible (key, value) vectors.

    Returns (out list, lse float).  No visible key -> zeros and -inf.
    """
    if not keys:
        return [0.0] * len(qrow), float("-inf")
    z = [scale * math.fsum(a * b for a, b in zip(qrow, k)) for k in keys]
    zmax = max(z)
    e = [math.exp(x - zmax) for x in z]
    tot = math.fsum(e)
    w = [x / tot for x in e]
    D = len(values[0])
    out = [math.fsum(w[n] * values[n][d] for n in range(len(values))) for d in range(D)]
    return out, zmax + math.log(tot)


def attention(q, k, v, visible, scale):
    """q [T][Hq][D], k/v [n][Hkv][D] nested lists of floats, visible [T][n] bools.

    Returns out [T][Hq][D], lse [Hq][T] as nested lists.
    """
    T = len(q)
    Hq = len(q[0])
    Hkv = len(k[0]) if k else 1
    g = Hq // Hkv
    out = [[None] * Hq for _ in range(T)]
    lse = [[None] * T for _ in range(Hq)]
    for i in range(T):
        for h in range(Hq):
            kv = h // g
            keys = [k[n][kv] for n in range(len(k)) if visible[i][n]]
            vals = [v[n][kv] for n in range(len(k)) if visible[i][n]]
            out[i][h], lse[h][i] = attend_row(q[i][h], keys, vals, scale)
    return out, lse


def ancestors(parent, i):
    """Set of nodes on the path from i to its root (inclusive)."""
    seen = set()
    while i >= 0:
        seen.add(i)
        i = parent[i]
    return seen
