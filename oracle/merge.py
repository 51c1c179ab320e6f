"""Composition of partial attention results over disjoint key sets (test oracle).

pwwt.cn "SageAttention deployment pitfalls guide" §4.1: the forward can return the
log-sum-exp of each query row ``for Ring Attention and similar`` schemes, which split the
keys into chunks (across devices or steps), attend to each chunk separately and combine
the partial outputs. For a row with partial results (o_i, lse_i) over disjoint key sets:

    lse = ln sum_i exp(lse_i)
    o   = sum_i exp(lse_i - lse) * o_i

which is the softmax over the union of the key sets (each o_i is already normalised by
its own sum exp(lse_i)). Plain float64; a part with lse_i = -inf (no visible key) has
weight 0, and a row no part sees gets o = 0, lse = -inf.
"""

import numpy as np


def merge_partials(outs, lses):
    """outs: sequence of arrays [..., d]; lses: sequence of arrays [...] (natural log).

    Returns (o, lse) as float64 arrays of shapes [..., d] and [...]."""
    if len(outs) == 0 or len(outs) != len(lses):
        raise ValueError("need one lse per partial output, at least one part")
    L = np.stack([np.asarray(x, np.float64) for x in lses])          # [n, ...]
    O = np.stack([np.asarray(x, np.float64) for x in outs])          # [n, ..., d]
    m = L.max(axis=0)
    seen = np.isfinite(m)
    m_safe = np.where(seen, m, 0.0)
    w = np.where(np.isfinite(L), np.exp(L - m_safe), 0.0)            # [n, ...]
    s = w.sum(axis=0)
    lse = np.where(seen, m_safe + np.log(np.where(seen, s, 1.0)), -np.inf)
    o = (w[..., None] * O).sum(axis=0) / np.where(seen, s, 1.0)[..., None]
    o = np.where(seen[..., None], o, 0.0)
    return o, lse
