"""Backward of causal attention with RoPE, fp64 (TEST INFRASTRUCTURE ONLY:
the test-suite, ``__graft_entry__.smoke()`` and the benchmark's CPU leg may
use it; the CUDA library never does).

The plain definition, one (batch, q-head) at a time, with the probabilities
rebuilt from Q and K ("RoPE and FlashAttention: relative positions and online
softmax", section 5: backward reconstructs P from Q/K and the saved row
normalisation instead of storing it; sections 1-2 for the rotation):

  q~_i = R(kv_offset + i) q_i,   k~_j = R(j) k_j,   V unrotated;
  s_ij = scale <q~_i, k~_j> for j <= kv_offset + i (else excluded);
  P = softmax_j(s),  O = P V;
  given dO:  dV = P^T dO,  dP = dO V^T,
             dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)   (softmax Jacobian),
             dq~ = scale dS k~,  dk~ = scale dS^T q~,
             dq_i = R(kv_offset + i)^T dq~_i,  dk_j = R(j)^T dk~_j,
  where R(p)^T = R(-p) (a rotation's inverse), so the rotation back is the
  oracle's own rotation at the negated positions.  Dims past rot_dim pass
  straight through.  With grouped-query attention the kv-head gradients sum
  over the q-heads of the group.

``attention_bwd_rows`` gives selected rows of the same gradients for
problems too large to differentiate densely (each query row from its own
probabilities, each key row from its column of probabilities over the rows
that see it, with the rows' LSE and O from the forward oracle).

Parity unpinned?  No: ``attention_bwd`` is pinned in
tests/test_oracle_backward.py by central finite differences of the forward
oracle, by torch's automatic differentiation of the definition on the CPU,
and by invariants; ``attention_bwd_rows`` is pinned there against
``attention_bwd`` on every row of small problems.
"""
from __future__ import annotations

import numpy as np

from . import NEOX, rope_rows


def attention_bwd(q, k, v, dout, kv_offset: int = 0, apply_rope: bool = True,
                  rot_dim: int | None = None, base: float = 10000.0, layout: int = NEOX,
                  scale: float | None = None, freq_dim: int = 0):
    """q, dout [B,Hq,Sq,D]; k, v [B,Hkv,Sk,D] (any real dtype, taken through
    float32 like the forward oracle).  Returns fp64 (dq, dk, dv)."""
    f = lambda x: np.asarray(np.asarray(x, dtype=np.float32), dtype=np.float64)
    q, k, v, dout = f(q), f(k), f(v), f(dout)
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    rot_dim = D if rot_dim is None else rot_dim
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    qpos = kv_offset + np.arange(Sq, dtype=np.int64)
    kpos = np.arange(Sk, dtype=np.int64)
    if apply_rope:
        qr = rope_rows(q, qpos, rot_dim, base, layout, freq_dim)
        kr = rope_rows(k, kpos, rot_dim, base, layout, freq_dim)
    else:
        qr, kr = q, k
    allowed = kpos[None, :] <= qpos[:, None]
    if not allowed.any(axis=1).all():
        raise ValueError("every query row needs at least one admissible key")
    dqr = np.zeros_like(q)
    dkr = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            s = scale * (qr[b, h] @ kr[b, hk].T)
            s = np.where(allowed, s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            dv[b, hk] += p.T @ dout[b, h]
            dp = dout[b, h] @ v[b, hk].T
            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dqr[b, h] = scale * (ds @ kr[b, hk])
            dkr[b, hk] += scale * (ds.T @ qr[b, h])
    if apply_rope:
        dq = rope_rows(dqr, -qpos, rot_dim, base, layout, freq_dim)
        dk = rope_rows(dkr, -kpos, rot_dim, base, layout, freq_dim)
    else:
        dq, dk = dqr, dkr
    return dq, dk, dv


def attention_bwd_rows(q, k, v, dout, dq_rows=None, dkv_rows=None, kv_offset: int = 0,
                       apply_rope: bool = True, rot_dim: int | None = None,
                       base: float = 10000.0, layout: int = NEOX, scale: float | None = None,
                       freq_dim: int = 0, nthreads: int | None = None):
    """Selected rows of the same gradients as ``attention_bwd``, for problems
    too large to differentiate densely.  Same arguments and definitions.

    dq_rows: flat query-row indices (b*Hq + h)*Sq + i, or None.  Row i needs
      only its own probabilities and dP over every key it sees:
        s_j = scale <q~_i, k~_j> (j <= kv_offset + i),  P = softmax_j(s),
        dP_j = <dO_i, V_j>,  dS_j = P_j (dP_j - sum_k P_k dP_k),
        dq~_i = scale sum_j dS_j k~_j,  dq_i = R(kv_offset + i)^T dq~_i.
    dkv_rows: flat key-row indices (b*Hkv + hk)*Sk + j, or None.  Key j needs
      column j of P and dS over every query row of its kv group that sees it,
      with each row's normaliser taken from the oracle's own forward
      (``oracle.attention``: LSE_i = m_i + ln l_i and O_i):
        P_ij = exp(s_ij - LSE_i),  dP_ij = <dO_i, V_j>,
        dS_ij = P_ij (dP_ij - <dO_i, O_i>)   (sum_k P_ik dP_ik = <dO_i, O_i>),
        dv_j = sum_i P_ij dO_i,  dk~_j = scale sum_i dS_ij q~_i,
        dk_j = R(j)^T dk~_j,
      the sums running over the q-heads of the group and their rows.
    Returns (dq [n, D] or None, dk [m, D] or None, dv [m, D] or None), fp64.
    """
    from . import attention  # the package's forward oracle (LSE and O)

    f = lambda x: np.asarray(np.asarray(x, dtype=np.float32), dtype=np.float64)
    q32 = np.ascontiguousarray(np.asarray(q, dtype=np.float32))
    k32 = np.ascontiguousarray(np.asarray(k, dtype=np.float32))
    v32 = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    B, Hq, Sq, D = q32.shape
    _, Hkv, Sk, _ = k32.shape
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    rot_dim = D if rot_dim is None else rot_dim
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    do64 = f(dout)
    kpos_all = np.arange(Sk, dtype=np.int64)

    def rot(x, pos):
        return rope_rows(x, pos, rot_dim, base, layout, freq_dim) if apply_rope else x

    def rot_back(x, pos):
        return rope_rows(x, -pos, rot_dim, base, layout, freq_dim) if apply_rope else x

    kr_cache = {}

    def k_rot(b, hk):  # every key row of one kv head, rotated at its position
        if (b, hk) not in kr_cache:
            kr_cache[(b, hk)] = rot(f(k32[b, hk]), kpos_all)
        return kr_cache[(b, hk)]

    dq = dk = dv = None
    if dq_rows is not None:
        rows = np.asarray(dq_rows, dtype=np.int64).reshape(-1)
        dq = np.empty((rows.shape[0], D), dtype=np.float64)
        for n, r in enumerate(rows):
            i, bh = int(r % Sq), int(r // Sq)
            h, b = bh % Hq, bh // Hq
            hk = h // G
            p_i = kv_offset + i
            L = min(Sk, p_i + 1)
            if L < 1:
                raise ValueError("every query row needs at least one admissible key")
            qr = rot(f(q32[b, h, i:i + 1]), np.array([p_i], dtype=np.int64))[0]
            kr = k_rot(b, hk)[:L]
            s = scale * (kr @ qr)
            p = np.exp(s - s.max())
            p /= p.sum()
            dp = f(v32[b, hk, :L]) @ do64[b, h, i]
            ds = p * (dp - (p * dp).sum())
            dq[n] = rot_back((scale * (ds @ kr))[None], np.array([p_i], dtype=np.int64))[0]
    if dkv_rows is not None:
        rows = np.asarray(dkv_rows, dtype=np.int64).reshape(-1)
        dk = np.empty((rows.shape[0], D), dtype=np.float64)
        dv = np.empty((rows.shape[0], D), dtype=np.float64)
        groups = {}
        for n, r in enumerate(rows):
            groups.setdefault(int(r // Sk), []).append((n, int(r % Sk)))
        for bhk, items in groups.items():
            b, hk = bhk // Hkv, bhk % Hkv
            j = np.array([jj for _, jj in items], dtype=np.int64)
            # query rows of the group that see at least one selected key
            i0 = max(0, int(j.min()) - kv_offset)
            if i0 >= Sq:  # no query sees these keys: zero gradients
                for n, _ in items:
                    dk[n] = 0.0
                    dv[n] = 0.0
                continue
            ii = np.arange(i0, Sq, dtype=np.int64)
            heads = np.arange(hk * G, hk * G + G, dtype=np.int64)
            flat = ((b * Hq + heads[:, None]) * Sq + ii[None, :]).reshape(-1)
            o_ref, lse_ref = attention(q32, k32, v32, kv_offset=kv_offset,
                                       apply_rope=apply_rope, rot_dim=rot_dim, base=base,
                                       layout=layout, scale=scale, freq_dim=freq_dim,
                                       rows=flat, nthreads=nthreads)
            qr = rot(f(q32[b, hk * G:hk * G + G, i0:]).reshape(-1, D), np.tile(kv_offset + ii, G))
            dor = do64[b, hk * G:hk * G + G, i0:].reshape(-1, D)
            qpos = np.tile(kv_offset + ii, G)
            kr = k_rot(b, hk)[j]
            vj = f(v32[b, hk, j])
            s = scale * (qr @ kr.T)
            seen = j[None, :] <= qpos[:, None]
            pm = np.where(seen, np.exp(np.where(seen, s, 0.0) - lse_ref[:, None]), 0.0)
            dpm = dor @ vj.T
            drow = (dor * o_ref).sum(axis=1)
            dsm = pm * (dpm - drow[:, None])
            dv_sel = pm.T @ dor
            dk_sel = rot_back(scale * (dsm.T @ qr), j)
            for c, (n, _) in enumerate(items):
                dk[n] = dk_sel[c]
                dv[n] = dv_sel[c]
    return dq, dk, dv
