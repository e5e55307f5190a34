"""Pins of the backward oracle (``oracle.attention_bwd``).

* Central finite differences of the forward oracle (the pages' own check in
  "RoPE and FlashAttention ...", section 5: an input derivative of a scalar
  loss compared with a difference quotient), on entries of q, k and v.
* torch's automatic differentiation (CPU, fp64) of the definition written
  with torch operations: gradients come from autograd, not from the oracle's
  hand-derived formulas.
* Invariants: sum_j dV_j = sum over the group's rows of dO (rows of P sum to
  one); a grouped kv head's gradients equal the sums over the q-heads of the
  same problem with the kv head replicated.
"""
import numpy as np
import pytest
import torch

NEOX, GPTJ = 0, 1


def inputs(B, Hq, Hkv, Sq, Sk, D, seed):
    rng = np.random.default_rng(seed)
    f = lambda *s: rng.standard_normal(s).astype(np.float32).astype(np.float64)
    return f(B, Hq, Sq, D), f(B, Hkv, Sk, D), f(B, Hkv, Sk, D), f(B, Hq, Sq, D)


@pytest.mark.parametrize("layout,rot_dim,off", [(NEOX, 8, 0), (GPTJ, 8, 3), (NEOX, 4, 2)])
def test_finite_differences_of_the_forward(oracle_mod, layout, rot_dim, off):
    """L = sum(O * G); dL/dx by central differences with a step exact in
    fp32 (the forward oracle takes its inputs through float32)."""
    B, Hq, Hkv, Sq, D = 1, 2, 1, 5, 8
    Sk = Sq + off
    q, k, v, g = inputs(B, Hq, Hkv, Sq, Sk, D, seed=5 + off)
    kw = dict(kv_offset=off, rot_dim=rot_dim, base=100.0, layout=layout)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, g, **kw)

    def loss(q_, k_, v_):
        o, _ = oracle_mod.attention(q_, k_, v_, **kw)
        return float((o * g).sum())

    eps = 2.0 ** -12
    rng = np.random.default_rng(1)
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            argm = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd = (loss(*args) - loss(*argm)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-5 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def torch_rope(x, pos, rot_dim, base, layout):
    """Rotation written with torch operations (for autograd)."""
    half = rot_dim // 2
    theta = base ** (-2.0 * torch.arange(half, dtype=torch.float64) / rot_dim)
    ang = pos.to(torch.float64)[:, None] * theta[None, :]
    c, s = torch.cos(ang), torch.sin(ang)
    if layout == NEOX:
        lo, hi = x[..., :half], x[..., half:rot_dim]
    else:
        lo, hi = x[..., 0:rot_dim:2], x[..., 1:rot_dim:2]
    a, b = lo * c - hi * s, hi * c + lo * s
    rot = torch.cat([a, b], -1) if layout == NEOX else torch.stack([a, b], -1).flatten(-2)
    return torch.cat([rot, x[..., rot_dim:]], -1)


@pytest.mark.parametrize("layout,rot_dim,off,Hq,Hkv", [(NEOX, 16, 0, 4, 2), (GPTJ, 16, 7, 2, 2),
                                                      (NEOX, 8, 3, 6, 3), (GPTJ, 12, 0, 3, 1)])
def test_matches_torch_autograd(oracle_mod, layout, rot_dim, off, Hq, Hkv):
    B, Sq, D = 2, 9, 16
    Sk = Sq + off
    q, k, v, g = inputs(B, Hq, Hkv, Sq, Sk, D, seed=off + Hq)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, g, kv_offset=off, rot_dim=rot_dim, base=50.0,
                                          layout=layout)
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    G = Hq // Hkv
    qr = torch_rope(qt, torch.arange(off, off + Sq), rot_dim, 50.0, layout)
    kr = torch_rope(kt, torch.arange(Sk), rot_dim, 50.0, layout)
    kr, vr = kr.repeat_interleave(G, dim=1), vt.repeat_interleave(G, dim=1)
    mask = torch.arange(Sk)[None, :] <= (off + torch.arange(Sq))[:, None]
    s = (qr @ kr.transpose(-1, -2)) / np.sqrt(D)
    o = torch.softmax(s.masked_fill(~mask, float("-inf")), -1) @ vr
    (o * torch.tensor(g)).sum().backward()
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-12)


def test_no_rope_and_custom_scale_match_autograd(oracle_mod):
    B, Hq, Hkv, Sq, Sk, D, off = 1, 2, 1, 6, 10, 8, 4
    q, k, v, g = inputs(B, Hq, Hkv, Sq, Sk, D, seed=2)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, g, kv_offset=off, apply_rope=False, scale=0.3)
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    mask = torch.arange(Sk)[None, :] <= (off + torch.arange(Sq))[:, None]
    s = 0.3 * (qt @ kt.repeat_interleave(2, 1).transpose(-1, -2))
    o = torch.softmax(s.masked_fill(~mask, float("-inf")), -1) @ vt.repeat_interleave(2, 1)
    (o * torch.tensor(g)).sum().backward()
    for a, t in ((dq, qt), (dk, kt), (dv, vt)):
        np.testing.assert_allclose(a, t.grad.numpy(), atol=1e-12)


def test_invariants(oracle_mod):
    B, Hq, Hkv, Sq, Sk, D, off = 2, 4, 2, 7, 11, 8, 4
    q, k, v, g = inputs(B, Hq, Hkv, Sq, Sk, D, seed=9)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, g, kv_offset=off, rot_dim=8, base=30.0)
    # rows of P sum to one: sum_j dV_j = sum of dO over the group's rows
    for hk in range(Hkv):
        np.testing.assert_allclose(dv[:, hk].sum(axis=1),
                                   g[:, 2 * hk:2 * hk + 2].sum(axis=(1, 2)), atol=1e-12)
    # grouped kv head == replicated kv heads, gradients summed over the group
    rq, rk, rv = oracle_mod.attention_bwd(q, np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1), g,
                                          kv_offset=off, rot_dim=8, base=30.0)
    np.testing.assert_allclose(dq, rq, atol=1e-12)
    np.testing.assert_allclose(dk, rk.reshape(B, Hkv, 2, Sk, D).sum(axis=2), atol=1e-12)
    np.testing.assert_allclose(dv, rv.reshape(B, Hkv, 2, Sk, D).sum(axis=2), atol=1e-12)
    # keys no query can see get zero gradient (Sk > kv_offset + Sq)
    dq2, dk2, dv2 = oracle_mod.attention_bwd(q, np.concatenate([k, k[:, :, :3]], 2),
                                             np.concatenate([v, v[:, :, :3]], 2), g,
                                             kv_offset=off, rot_dim=8, base=30.0)
    assert np.all(dk2[:, :, Sk:] == 0) and np.all(dv2[:, :, Sk:] == 0)
    np.testing.assert_allclose(dq2, dq, atol=1e-12)


@pytest.mark.parametrize("layout,rot_dim,off,Hq,Hkv,Sq,Sk", [
    (NEOX, 16, 0, 4, 2, 9, 9),      # square, full rotation, GQA
    (GPTJ, 8, 5, 2, 1, 7, 15),      # cached prefix, partial rotation, keys no query sees
    (NEOX, 12, 3, 6, 3, 11, 14),    # partial NeoX, odd group count
])
def test_selected_rows_equal_dense_rows(oracle_mod, layout, rot_dim, off, Hq, Hkv, Sq, Sk):
    """attention_bwd_rows, asked for every query row and every key row (in a
    shuffled order), reproduces attention_bwd row by row."""
    B, D = 2, 16
    q, k, v, g = inputs(B, Hq, Hkv, Sq, Sk, D, seed=11 + off + Hq)
    kw = dict(kv_offset=off, rot_dim=rot_dim, base=70.0, layout=layout)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, g, **kw)
    rng = np.random.default_rng(off)
    qr = rng.permutation(B * Hq * Sq)
    kr = rng.permutation(B * Hkv * Sk)
    sq, sk, sv = oracle_mod.attention_bwd_rows(q, k, v, g, dq_rows=qr, dkv_rows=kr, nthreads=2,
                                               **kw)
    np.testing.assert_allclose(sq, dq.reshape(-1, D)[qr], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sk, dk.reshape(-1, D)[kr], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sv, dv.reshape(-1, D)[kr], rtol=0, atol=1e-12)


def test_selected_rows_no_rope_custom_scale(oracle_mod):
    B, Hq, Hkv, Sq, Sk, D, off = 1, 4, 1, 6, 10, 8, 4
    q, k, v, g = inputs(B, Hq, Hkv, Sq, Sk, D, seed=21)
    kw = dict(kv_offset=off, apply_rope=False, scale=0.35)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, g, **kw)
    qr, kr = np.array([0, 5, 23, 12]), np.array([9, 0, 4])
    sq, sk, sv = oracle_mod.attention_bwd_rows(q, k, v, g, dq_rows=qr, dkv_rows=kr, **kw)
    np.testing.assert_allclose(sq, dq.reshape(-1, D)[qr], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sk, dk.reshape(-1, D)[kr], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sv, dv.reshape(-1, D)[kr], rtol=0, atol=1e-12)
    # only one side asked for: the other comes back as None
    oq, ok_, ov = oracle_mod.attention_bwd_rows(q, k, v, g, dq_rows=qr[:1], **kw)
    assert ok_ is None and ov is None and oq.shape == (1, D)
