"""Online-softmax (tiled) attention recurrence in fp64 NumPy.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Restates the running-state recurrence of "RoPE and FlashAttention: relative
positions and online softmax", section 5: for each query row keep the running
maximum m, the exponential denominator l and the unnormalised weighted-value
numerator u.  A tile with scores s and values V updates

    m' = max(m, max_j s_j),   alpha = exp(m - m'),
    l' = alpha * l + sum_j exp(s_j - m'),
    u' = alpha * u + sum_j exp(s_j - m') V_j,

and the output is u / l after the last tile.  Rows for which a tile holds no
admissible key skip that tile (so -inf - -inf never occurs); a row with no
admissible key at all is rejected, as the page does.  Query blocks form the
outer loop and key/value blocks the inner loop, the order that page uses.

The mask is generated per tile from the causal offset (key j admissible for
query i iff j <= kv_offset + i), or taken from an explicit dense boolean
matrix when one is given (the teaching form on that page).
"""
from __future__ import annotations

import numpy as np


def tiled_attention(q, k, v, kv_offset: int = 0, block_q: int = 3, block_k: int | None = None,
                    scale: float | None = None, allowed=None, return_lse: bool = False):
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if q.ndim != 2 or k.ndim != 2 or v.ndim != 2:
        raise ValueError("2-D query, key and value matrices required")
    if q.shape[1] != k.shape[1] or k.shape[0] != v.shape[0]:
        raise ValueError("query/key width or key/value length mismatch")
    block_k = block_q if block_k is None else block_k
    if block_q <= 0 or block_k <= 0:
        raise ValueError("positive block sizes required")
    n_q, n_k = q.shape[0], k.shape[0]
    scale = 1.0 / np.sqrt(q.shape[1]) if scale is None else float(scale)
    if allowed is not None:
        allowed = np.asarray(allowed, dtype=bool)
        if allowed.shape != (n_q, n_k):
            raise ValueError("allowed must be [Sq, Sk]")
        has_key = allowed.any(axis=1)
    else:
        has_key = (kv_offset + np.arange(n_q)) >= 0
    if not np.all(has_key):
        raise ValueError("every query row needs at least one admissible key")

    out = np.empty((n_q, v.shape[1]))
    lse = np.empty(n_q)
    for q0 in range(0, n_q, block_q):
        rows = np.arange(q0, min(q0 + block_q, n_q))
        m = np.full(rows.size, -np.inf)
        l = np.zeros(rows.size)
        u = np.zeros((rows.size, v.shape[1]))
        for k0 in range(0, n_k, block_k):
            cols = np.arange(k0, min(k0 + block_k, n_k))
            if allowed is not None:
                ok = allowed[np.ix_(rows, cols)]
            else:
                ok = cols[None, :] <= (kv_offset + rows)[:, None]
            live = ok.any(axis=1)
            if not live.any():
                continue  # whole tile in the future of every row: skipped
            s = np.where(ok, (q[rows] @ k[cols].T) * scale, -np.inf)[live]
            m_new = np.maximum(m[live], s.max(axis=1))
            alpha = np.exp(m[live] - m_new)
            w = np.exp(s - m_new[:, None])
            l[live] = alpha * l[live] + w.sum(axis=1)
            u[live] = alpha[:, None] * u[live] + w @ v[cols]
            m[live] = m_new
        out[rows] = u / l[:, None]
        lse[rows] = m + np.log(l)
    return (out, lse) if return_lse else out
