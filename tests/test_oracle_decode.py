"""Pins of the decoder-step oracle (``oracle.decode_attention``) against the
plain causal attention definition ("RoPE and FlashAttention: relative
positions and online softmax", sections 2 and 5): decoding the last Sq
queries over a cache equals the last Sq rows of full causal attention over
the same sequence, and a cache of rotated keys with rotated queries equals
attention with RoPE applied to the raw tensors (section 2's convention)."""
import numpy as np
import pytest

NEOX, GPTJ = 0, 1


def scatter_cache(rng, seqs, Hkv, D, gap=5):
    """Packs per-sequence [L, Hkv, D] arrays into one cache with gaps between
    sequences; returns (cache, seq_start)."""
    starts, rows = [], 3
    for x in seqs:
        starts.append(rows)
        rows += x.shape[0] + gap
    cache = rng.standard_normal((rows, Hkv, D)) * 100.0  # junk outside the sequences
    for s0, x in zip(starts, seqs):
        cache[s0:s0 + x.shape[0]] = x
    return cache, np.array(starts, dtype=np.int64)


@pytest.mark.parametrize("Hq,Hkv,Sq,D", [(4, 2, 1, 16), (6, 3, 3, 8), (2, 2, 5, 12)])
def test_decode_equals_last_rows_of_full_attention(oracle_mod, Hq, Hkv, Sq, D):
    rng = np.random.default_rng(7)
    lens = [Sq, Sq + 9, Sq + 30]
    ks = [rng.standard_normal((L, Hkv, D)) for L in lens]
    vs = [rng.standard_normal((L, Hkv, D)) for L in lens]
    qs = [rng.standard_normal((1, Hq, L, D)) for L in lens]
    kc, st = scatter_cache(rng, ks, Hkv, D)
    vc, _ = scatter_cache(rng, vs, Hkv, D)
    # entries visit the sequences in a permuted order
    order = [2, 0, 1]
    q = np.stack([qs[s][0, :, -Sq:, :] for s in order])
    o, lse = oracle_mod.decode_attention(q, kc, vc, st, [lens[s] for s in order],
                                         seq_ids=order)
    for b, s in enumerate(order):
        fo, fl = oracle_mod.attention(qs[s], ks[s].transpose(1, 0, 2)[None],
                                      vs[s].transpose(1, 0, 2)[None], apply_rope=False)
        np.testing.assert_allclose(o[b], fo[0, :, -Sq:, :], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b], fl[0, :, -Sq:], rtol=0, atol=1e-12)


def test_decode_first_query_sees_only_key_zero(oracle_mod):
    """Sq = L: query 0 sits at position 0, so its output is v_0 and its LSE
    is its single scaled score."""
    rng = np.random.default_rng(3)
    L, D = 6, 8
    k = rng.standard_normal((L, 1, D))
    v = rng.standard_normal((L, 1, D))
    q = rng.standard_normal((1, 1, L, D))
    o, lse = oracle_mod.decode_attention(q, k, v, [0], [L])
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0], atol=1e-14)
    np.testing.assert_allclose(lse[0, 0, 0], q[0, 0, 0] @ k[0, 0] / np.sqrt(D), atol=1e-13)


@pytest.mark.parametrize("layout,rot_dim", [(NEOX, 16), (GPTJ, 16), (NEOX, 8)])
def test_cached_rotated_keys_equal_fused_rope(oracle_mod, layout, rot_dim):
    """Section 2: rotate new Q/K at their absolute positions, cache rotated K
    and raw V, never rotate cached K again -- the decode result equals
    attention with RoPE applied inside, on the raw tensors."""
    rng = np.random.default_rng(11)
    Hq, Hkv, D, Sq, L = 4, 2, 16, 2, 23
    k = rng.standard_normal((L, Hkv, D))
    v = rng.standard_normal((L, Hkv, D))
    q = rng.standard_normal((1, Hq, Sq, D))
    k, v, q = (x.astype(np.float32).astype(np.float64) for x in (k, v, q))
    pos = np.arange(L)
    k_rot = oracle_mod.rope_tokens(k, pos, rot_dim=rot_dim, base=500.0, layout=layout)
    q_rot = oracle_mod.rope_rows(q, pos[L - Sq:], rot_dim=rot_dim, base=500.0, layout=layout)
    o, lse = oracle_mod.decode_attention(q_rot, k_rot, v, [0], [L])
    fo, fl = oracle_mod.attention(q, k.transpose(1, 0, 2)[None], v.transpose(1, 0, 2)[None],
                                  kv_offset=L - Sq, rot_dim=rot_dim, base=500.0, layout=layout)
    # the attention oracle takes its inputs through fp32, so the pre-rotated
    # side carries one fp32 rounding of q and k that the fused side does not
    np.testing.assert_allclose(o, fo, atol=2e-6)
    np.testing.assert_allclose(lse, fl, atol=2e-6)
    # re-rotating the cached keys (the mistake section 2 warns about) changes the result
    k_twice = oracle_mod.rope_tokens(k_rot, pos, rot_dim=rot_dim, base=500.0, layout=layout)
    o2, _ = oracle_mod.decode_attention(q_rot, k_twice, v, [0], [L])
    assert np.abs(o2 - fo).max() > 1e-3
