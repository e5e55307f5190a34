"""Pins for the oracle's attention: the pages' tiled-softmax test, textbook
softmax attention from library routines, closed forms and invariants."""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

from conftest import golden_kv

NEOX, GPTJ = 0, 1


def _page_setup():
    g = golden_kv("tiled_attention_setup.txt")
    rng = np.random.default_rng(int(g["seed"][0]))
    Q = rng.normal(size=tuple(map(int, g["q_shape"])))
    K = rng.normal(size=tuple(map(int, g["k_shape"])))
    V = rng.normal(size=tuple(map(int, g["v_shape"])))
    return (Q, K, V, int(g["kv_offset"][0]), [int(b) for b in g["blocks"]],
            float(g["tolerance"][0]))


def _dense_reference(Q, K, V, off, scale):
    mask = np.arange(K.shape[0])[None, :] <= (off + np.arange(Q.shape[0]))[:, None]
    s = np.where(mask, Q @ K.T * scale, -np.inf)
    return softmax(s, axis=-1) @ V, logsumexp(s, axis=-1)


def test_tiled_matches_dense_softmax_page_setup(oracle_mod):
    """"RoPE and FlashAttention ...", section 5: the recurrence equals SciPy's
    softmax for tile sizes 1, 2, 3 and 20 on the 7x9 offset-causal setup."""
    Q, K, V, off, blocks, tol = _page_setup()
    ref, ref_lse = _dense_reference(Q, K, V, off, 0.5)
    for b in blocks:
        out, lse = oracle_mod.tiled_attention(Q, K, V, kv_offset=off, block_q=b, return_lse=True)
        np.testing.assert_allclose(out, ref, rtol=tol, atol=tol)
        np.testing.assert_allclose(lse, ref_lse, rtol=tol, atol=tol)
    for bq, bk in [(2, 5), (7, 1), (1, 9), (4, 3)]:
        out = oracle_mod.tiled_attention(Q, K, V, kv_offset=off, block_q=bq, block_k=bk)
        np.testing.assert_allclose(out, ref, rtol=tol, atol=tol)


def test_naive_oracle_matches_page_setup(oracle_mod):
    """The C oracle without rotation on the same setup (one head)."""
    Q, K, V, off, _, tol = _page_setup()
    # V has width 5, the C oracle needs equal q/v width: pad q/k to 5 with zeros
    Qp = np.concatenate([Q, np.zeros((7, 1))], 1)
    Kp = np.concatenate([K, np.zeros((9, 1))], 1)
    o, lse = oracle_mod.attention(Qp[None, None].astype(np.float32),
                                  Kp[None, None].astype(np.float32),
                                  V[None, None].astype(np.float32), kv_offset=off,
                                  apply_rope=False, scale=0.5)
    ref, ref_lse = _dense_reference(Q.astype(np.float32).astype(np.float64),
                                    K.astype(np.float32).astype(np.float64),
                                    V.astype(np.float32).astype(np.float64), off, 0.5)
    np.testing.assert_allclose(o[0, 0], ref, rtol=tol, atol=tol)
    np.testing.assert_allclose(lse[0, 0], ref_lse, rtol=tol, atol=tol)


def test_rising_max_requires_rescale(oracle_mod):
    """Section 5 control: averaging separately normalised tiles is wrong by
    more than 1 on scores (0, 1, 20); the recurrence (tile 2 then 1, so the
    max rises inside the row) gets the softmax-weighted value."""
    g = golden_kv("rising_max_control.txt")
    x = np.array([float(t) for t in g["scores"]])
    vals = np.array([float(t) for t in g["values"]])
    naive = (softmax(x[:2]) @ vals[:2] + vals[2]) / 2
    truth = softmax(x) @ vals
    assert abs(naive - truth) > float(g["min_gap"][0])
    # one query whose scores are exactly x: q = 1, keys = x, scale 1
    out = oracle_mod.tiled_attention(np.ones((1, 1)), x[:, None], vals[:, None],
                                     kv_offset=2, block_q=1, block_k=2, scale=1.0)
    assert out[0, 0] == pytest.approx(truth, abs=1e-12)


def test_empty_rows_rejected(oracle_mod):
    """Section 5: a row with no admissible key is rejected, not turned into NaN."""
    Q, K, V, off, _, _ = _page_setup()
    with pytest.raises(ValueError):
        oracle_mod.tiled_attention(Q, K, V, allowed=np.zeros((7, 9), dtype=bool))
    with pytest.raises(ValueError):
        oracle_mod.tiled_attention(Q, K, V, kv_offset=-1)
    z = np.zeros((1, 1, 4, 8), dtype=np.float32)
    with pytest.raises(ValueError):
        oracle_mod.attention(z, z, z, kv_offset=-1, apply_rope=False)


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,off", [(2, 4, 2, 9, 13, 8, 4), (1, 3, 3, 16, 16, 6, 0),
                                                 (1, 2, 1, 5, 5, 4, 0), (1, 2, 2, 3, 20, 4, 7)])
def test_textbook_attention_without_rope(oracle_mod, B, Hq, Hkv, Sq, Sk, D, off):
    """"RoPE and FlashAttention ...", section 4: S = QK^T / sqrt(d), P = softmax(S),
    O = PV, with the offset-causal mask; LSE from SciPy's logsumexp.  Keys
    past kv_offset + Sq (when Sk is larger) are never admissible."""
    rng = np.random.default_rng(Sq * 31 + D)
    q = rng.standard_normal((B, Hq, Sq, D)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, Sk, D)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, Sk, D)).astype(np.float32)
    o, lse = oracle_mod.attention(q, k, v, kv_offset=off, apply_rope=False)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            ref, ref_lse = _dense_reference(q[b, h].astype(np.float64),
                                            k[b, h // G].astype(np.float64),
                                            v[b, h // G].astype(np.float64), off, 1 / math.sqrt(D))
            np.testing.assert_allclose(o[b, h], ref, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(lse[b, h], ref_lse, rtol=1e-12, atol=1e-12)


def test_matches_torch_sdpa_cpu_fp64(oracle_mod):
    """Second library check: torch's CPU scaled_dot_product_attention in fp64
    with an explicit offset mask (section 6: rectangular queries need the
    explicit offset mask, not is_causal)."""
    rng = np.random.default_rng(17)
    q = rng.standard_normal((1, 2, 6, 8)).astype(np.float32)
    k = rng.standard_normal((1, 2, 10, 8)).astype(np.float32)
    v = rng.standard_normal((1, 2, 10, 8)).astype(np.float32)
    o, _ = oracle_mod.attention(q, k, v, kv_offset=4, apply_rope=False)
    mask = torch.arange(10)[None, :] <= (4 + torch.arange(6))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).double(), torch.from_numpy(k).double(), torch.from_numpy(v).double(),
        attn_mask=mask, dropout_p=0.0)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("off", [0, 5])
def test_rope_positions_closed_form(oracle_mod, off):
    """D = 2, q = k = (1, 0): query row i sits at kv_offset + i, key j at j, and
    the score is scale * cos(kv_offset + i - j) (section 1's identity, theta_0 = 1),
    so O and LSE have a closed form.  Pins the position convention and the mask."""
    Sq, Sk = 4, off + 4
    q = np.zeros((1, 1, Sq, 2), np.float32)
    q[..., 0] = 1
    k = np.zeros((1, 1, Sk, 2), np.float32)
    k[..., 0] = 1
    v = np.random.default_rng(1).standard_normal((1, 1, Sk, 2)).astype(np.float32)
    scale = 0.75
    for layout in (NEOX, GPTJ):
        o, lse = oracle_mod.attention(q, k, v, kv_offset=off, scale=scale, layout=layout)
        for i in range(Sq):
            js = np.arange(0, off + i + 1)
            s = scale * np.cos(off + i - js)
            w = np.exp(s - s.max())
            np.testing.assert_allclose(o[0, 0, i], (w / w.sum()) @ v[0, 0, js].astype(np.float64),
                                       rtol=1e-13, atol=1e-13)
            assert lse[0, 0, i] == pytest.approx(math.log(np.exp(s).sum()), abs=1e-13)


@pytest.mark.parametrize("layout,rot_dim", [(NEOX, None), (GPTJ, None), (NEOX, 4), (GPTJ, 6)])
def test_rope_attention_is_attention_of_rotated(oracle_mod, layout, rot_dim):
    """Attention with RoPE equals textbook attention of Q rotated at
    kv_offset + i and K rotated at j; V is never rotated."""
    rng = np.random.default_rng(21)
    B, Hq, Hkv, Sq, Sk, D, off = 1, 4, 2, 6, 9, 8, 3
    q = rng.standard_normal((B, Hq, Sq, D)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, Sk, D)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, Sk, D)).astype(np.float32)
    o, lse = oracle_mod.attention(q, k, v, kv_offset=off, layout=layout, rot_dim=rot_dim,
                                  base=100.0)
    qr = oracle_mod.rope_rows(q, np.arange(Sq) + off, rot_dim=rot_dim, base=100.0, layout=layout)
    kr = oracle_mod.rope_rows(k, np.arange(Sk), rot_dim=rot_dim, base=100.0, layout=layout)
    for h in range(Hq):
        ref, ref_lse = _dense_reference(qr[0, h], kr[0, h // 2], v[0, h // 2].astype(np.float64),
                                        off, 1 / math.sqrt(D))
        np.testing.assert_allclose(o[0, h], ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[0, h], ref_lse, rtol=1e-12, atol=1e-12)
    # negative control: rotating V as well changes O ("rotate V" is wrong)
    vr = oracle_mod.rope_rows(v, np.arange(Sk), base=100.0, layout=layout).astype(np.float32)
    o_bad, _ = oracle_mod.attention(q, k, vr, kv_offset=off, layout=layout, rot_dim=rot_dim,
                                    base=100.0)
    assert not np.allclose(o, o_bad)


def test_gqa_head_mapping(oracle_mod):
    """q-head h reads kv-head h // (Hq/Hkv): equal to one-head calls on the
    matching kv head, and different from the interleaved mapping h % Hkv."""
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 6, 5, 4)).astype(np.float32)
    k = rng.standard_normal((1, 2, 5, 4)).astype(np.float32)
    v = rng.standard_normal((1, 2, 5, 4)).astype(np.float32)
    o, _ = oracle_mod.attention(q, k, v)
    for h in range(6):
        oh, _ = oracle_mod.attention(q[:, h:h + 1], k[:, h // 3:h // 3 + 1], v[:, h // 3:h // 3 + 1])
        np.testing.assert_array_equal(o[:, h], oh[:, 0])
    o1, _ = oracle_mod.attention(q[:, 1:2], k[:, 1:2], v[:, 1:2])
    assert not np.allclose(o[:, 1], o1[:, 0])


def test_first_row_sees_only_key_zero(oracle_mod):
    """With kv_offset 0 row 0 has one key: O_0 = V_0 and LSE_0 = s_00."""
    rng = np.random.default_rng(8)
    q = rng.standard_normal((1, 1, 3, 4)).astype(np.float32)
    k = rng.standard_normal((1, 1, 3, 4)).astype(np.float32)
    v = rng.standard_normal((1, 1, 3, 4)).astype(np.float32)
    o, lse = oracle_mod.attention(q, k, v, apply_rope=False, scale=0.5)
    np.testing.assert_array_equal(o[0, 0, 0], v[0, 0, 0].astype(np.float64))
    s00 = 0.5 * float(q[0, 0, 0].astype(np.float64) @ k[0, 0, 0].astype(np.float64))
    assert lse[0, 0, 0] == pytest.approx(s00, abs=1e-14)


def test_uniform_scores_average_values(oracle_mod):
    """q = 0 gives equal scores: O_i is the mean of the admissible V rows and
    LSE_i = ln(count)."""
    rng = np.random.default_rng(6)
    q = np.zeros((1, 1, 5, 4), np.float32)
    k = rng.standard_normal((1, 1, 8, 4)).astype(np.float32)
    v = rng.standard_normal((1, 1, 8, 4)).astype(np.float32)
    o, lse = oracle_mod.attention(q, k, v, kv_offset=2)
    for i in range(5):
        n = min(8, 2 + i + 1)
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :n].astype(np.float64).mean(0), atol=1e-14)
        assert lse[0, 0, i] == pytest.approx(math.log(n), abs=1e-14)


def test_row_subset_matches_full(oracle_mod):
    rng = np.random.default_rng(12)
    q = rng.standard_normal((2, 4, 7, 8)).astype(np.float32)
    k = rng.standard_normal((2, 2, 10, 8)).astype(np.float32)
    v = rng.standard_normal((2, 2, 10, 8)).astype(np.float32)
    o, lse = oracle_mod.attention(q, k, v, kv_offset=3, layout=GPTJ)
    rows = np.array([0, 5, 17, 55, 40])
    os_, ls = oracle_mod.attention(q, k, v, kv_offset=3, layout=GPTJ, rows=rows)
    np.testing.assert_array_equal(os_, o.reshape(-1, 8)[rows])
    np.testing.assert_array_equal(ls, lse.reshape(-1)[rows])


@pytest.mark.parametrize("bq,bk,off", [(1, 1, 0), (3, 2, 4), (16, 5, 1), (4, 64, 0)])
def test_tiled_recurrence_equals_naive_with_rope(oracle_mod, bq, bk, off):
    """The online-softmax recurrence over rotated Q/K reaches the naive
    two-pass result for uneven tilings and offsets."""
    rng = np.random.default_rng(bq * 7 + bk)
    Sq, D = 13, 8
    Sk = Sq + off
    q = rng.standard_normal((1, 1, Sq, D)).astype(np.float32)
    k = rng.standard_normal((1, 1, Sk, D)).astype(np.float32)
    v = rng.standard_normal((1, 1, Sk, D)).astype(np.float32)
    o, lse = oracle_mod.attention(q, k, v, kv_offset=off, layout=GPTJ)
    qr = oracle_mod.rope_rows(q[0, 0], np.arange(Sq) + off, layout=GPTJ)
    kr = oracle_mod.rope_rows(k[0, 0], np.arange(Sk), layout=GPTJ)
    ot, lt = oracle_mod.tiled_attention(qr, kr, v[0, 0], kv_offset=off, block_q=bq, block_k=bk,
                                        return_lse=True)
    np.testing.assert_allclose(ot, o[0, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lt, lse[0, 0], rtol=1e-12, atol=1e-12)
