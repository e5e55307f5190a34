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

Parity unpinned?  No: pinned in tests/test_oracle_backward.py by central
finite differences of the forward oracle, by torch's automatic
differentiation of the definition on the CPU, and by invariants.
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
