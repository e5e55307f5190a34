"""Pins for the oracle's RoPE: values and properties the pages fix.

Each test names the passage it follows.  None of them retypes the oracle's
formula: they check printed values, closed forms, invariants and
equivalences that a dropped term, a flipped sign, a wrong pairing or a wrong
frequency would break.
"""
import math

import numpy as np
import pytest

from conftest import golden_kv, read_golden

NEOX, GPTJ = 0, 1
LAYOUTS = [NEOX, GPTJ]


def test_worked_example_scores(oracle_mod):
    """"RoPE and FlashAttention ...", section 2 practice solution: q = k = (1, 0),
    theta = 1 (D = 2 so theta_0 = 1 for any base): score(m=2, n=5) = cos 3,
    both moved by 10 -> cos 3, only k moved -> cos 13, m = n -> q.k."""
    for layout in LAYOUTS:
        for qp, kp, want in read_golden("rope_worked_example.txt"):
            q = oracle_mod.rope_rows([[1.0, 0.0]], [int(qp)], base=10000.0, layout=layout)
            k = oracle_mod.rope_rows([[1.0, 0.0]], [int(kp)], base=10000.0, layout=layout)
            assert float(q[0] @ k[0]) == pytest.approx(float(want), abs=1e-14)


def _shift_setup():
    g = golden_kv("rope_shift_setup.txt")
    a, b = map(int, g["q_positions"])
    c, d = map(int, g["k_positions"])
    return (np.arange(a, b + 1), np.arange(c, d + 1), int(g["width"][0]), float(g["base"][0]),
            int(g["shift"][0]), float(g["tolerance"][0]), int(g["seed"][0]))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("rot_dim", [None, 4])
def test_all_pairs_relative_shift(oracle_mod, layout, rot_dim):
    """Section 2 of the same page: all q.k scores at unequal positions are
    unchanged when both position sets move by 23; moving k alone by 1 changes
    them.  Checked for both layouts and for partial rotation."""
    qp, kp, width, base, shift, tol, seed = _shift_setup()
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((2, 3, qp.size, width))
    k = rng.standard_normal((2, 3, kp.size, width))
    rope = lambda x, p: oracle_mod.rope_rows(x, p, rot_dim=rot_dim, base=base, layout=layout)
    a = rope(q, qp) @ np.swapaxes(rope(k, kp), -1, -2)
    b = rope(q, qp + shift) @ np.swapaxes(rope(k, kp + shift), -1, -2)
    np.testing.assert_allclose(a, b, rtol=tol, atol=tol)
    wrong = rope(q, qp) @ np.swapaxes(rope(k, kp + 1), -1, -2)
    assert not np.allclose(a, wrong)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_shift_invariance_random_positions(oracle_mod, layout):
    """The same invariance for scattered positions (continuous batching) and a
    large shift, as the relative-offset identity R(m)^T R(n) = R(n - m) implies."""
    rng = np.random.default_rng(7)
    qp = rng.integers(0, 5000, 11)
    kp = rng.integers(0, 5000, 13)
    q = rng.standard_normal((qp.size, 16))
    k = rng.standard_normal((kp.size, 16))
    rope = lambda x, p: oracle_mod.rope_rows(x, p, base=10000.0, layout=layout)
    a = rope(q, qp) @ rope(k, kp).T
    b = rope(q, qp + 777) @ rope(k, kp + 777).T
    np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-9)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("rot_dim", [8, 6, 2])
def test_norm_per_pair_and_untouched_tail(oracle_mod, layout, rot_dim):
    """Rotations keep every pair's norm (section 2, 1e-12); dims past rot_dim
    come back bit-identical ("Write Triton Rope Kernel", Correctness
    requirements: partial RoPE tail unchanged)."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 12))
    pos = np.array([0, 1, 17, 4095, 131071])
    y = oracle_mod.rope_rows(x, pos, rot_dim=rot_dim, base=10000.0, layout=layout)
    half = rot_dim // 2
    if layout == NEOX:
        lo, hi = np.arange(half), np.arange(half) + half
    else:
        lo, hi = 2 * np.arange(half), 2 * np.arange(half) + 1
    np.testing.assert_allclose(y[:, lo] ** 2 + y[:, hi] ** 2, x[:, lo] ** 2 + x[:, hi] ** 2,
                               rtol=1e-12, atol=1e-12)
    assert np.array_equal(y[:, rot_dim:], x[:, rot_dim:])


@pytest.mark.parametrize("layout", LAYOUTS)
def test_chunked_equals_full(oracle_mod, layout):
    """Section 2: rotating a cached prefix and the new chunk separately equals
    rotating the whole sequence (bitwise); the chunk rotated at positions that
    restart from 0 differs."""
    rng = np.random.default_rng(43)
    k = rng.standard_normal((2, 3, 9, 8))
    kp = np.arange(2, 11)
    full = oracle_mod.rope_rows(k, kp, layout=layout)
    chunked = np.concatenate([oracle_mod.rope_rows(k[..., :4, :], kp[:4], layout=layout),
                              oracle_mod.rope_rows(k[..., 4:, :], kp[4:], layout=layout)], -2)
    assert np.array_equal(full, chunked)
    restarted = oracle_mod.rope_rows(k[..., 4:, :], np.arange(5), layout=layout)
    assert not np.allclose(full[..., 4:, :], restarted)


@pytest.mark.parametrize("rot_dim", [16, 8])
def test_neox_gptj_equivalence_under_permutation(oracle_mod, rot_dim):
    """Section 2 / section 8 item 3: the two layouts are the same function after
    a consistent permutation of the rotated dims (evens first, then odds):
    neox(x[P]) == gptj(x)[P] bitwise, and all q.k scores agree."""
    D = 16
    P = np.concatenate([np.arange(0, rot_dim, 2), np.arange(1, rot_dim, 2),
                        np.arange(rot_dim, D)])
    rng = np.random.default_rng(11)
    x = rng.standard_normal((6, D))
    k = rng.standard_normal((6, D))
    pos = np.array([0, 3, 99, 1000, 65535, 131071])
    gj = oracle_mod.rope_rows(x, pos, rot_dim=rot_dim, layout=GPTJ)
    nx = oracle_mod.rope_rows(x[:, P], pos, rot_dim=rot_dim, layout=NEOX)
    assert np.array_equal(nx, gj[:, P])
    s_gj = gj @ oracle_mod.rope_rows(k, pos[::-1].copy(), rot_dim=rot_dim, layout=GPTJ).T
    s_nx = nx @ oracle_mod.rope_rows(k[:, P], pos[::-1].copy(), rot_dim=rot_dim, layout=NEOX).T
    np.testing.assert_allclose(s_gj, s_nx, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_position_zero_is_identity(oracle_mod, layout):
    x = np.random.default_rng(5).standard_normal((3, 10))
    y = oracle_mod.rope_rows(x, [0, 0, 0], layout=layout)
    assert np.array_equal(x, y)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_quarter_turn_sign(oracle_mod, layout):
    """A rotation by +pi/2 sends (a, b) to (-b, a): this fixes the sign of sin
    ("Write Triton Rope Kernel", step 6: lo*cos - hi*sin, hi*cos + lo*sin;
    Common failure modes: wrong sign of sin).  With rot_dim = F = 4 the second
    frequency is base^(-1/2); base = (2/pi)^2 makes it pi/2, so position 1
    turns pair 1 by a quarter and pair 0 by 1 radian."""
    base = (2.0 / math.pi) ** 2
    x = np.array([[0.3, -1.7, 2.5, 0.9]])
    y = oracle_mod.rope_rows(x, [1], rot_dim=4, base=base, layout=layout)[0]
    if layout == NEOX:  # pairs (0, 2) at theta 1 and (1, 3) at theta pi/2
        a, b = x[0, 1], x[0, 3]
        np.testing.assert_allclose([y[1], y[3]], [-b, a], atol=1e-15)
        np.testing.assert_allclose([y[0], y[2]],
                                   [0.3 * math.cos(1) - 2.5 * math.sin(1),
                                    2.5 * math.cos(1) + 0.3 * math.sin(1)], atol=1e-15)
    else:  # pairs (0, 1) at theta 1 and (2, 3) at theta pi/2
        a, b = x[0, 2], x[0, 3]
        np.testing.assert_allclose([y[2], y[3]], [-b, a], atol=1e-15)
        np.testing.assert_allclose([y[0], y[1]],
                                   [0.3 * math.cos(1) + 1.7 * math.sin(1),
                                    -1.7 * math.cos(1) + 0.3 * math.sin(1)], atol=1e-15)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_composition_adds_angles(oracle_mod, layout):
    """R(a)R(b) = R(a + b): rotating at p1 then at p2 equals rotating at p1 + p2."""
    x = np.random.default_rng(9).standard_normal((4, 8))
    p1 = np.array([3, 100, 7, 30000])
    p2 = np.array([5, 1, 9000, 2])
    two = oracle_mod.rope_rows(oracle_mod.rope_rows(x, p1, layout=layout), p2, layout=layout)
    one = oracle_mod.rope_rows(x, p1 + p2, layout=layout)
    np.testing.assert_allclose(two, one, rtol=1e-10, atol=1e-10)


def test_frequencies_golden(oracle_mod):
    """theta_i = base^(-2i/d): printed-formula values for small d."""
    for row in read_golden("rope_freqs.txt"):
        base, d = float(row[0]), int(row[1])
        want = np.array([float(t) for t in row[2:]])
        np.testing.assert_allclose(oracle_mod.rope_freqs(d, base), want, rtol=1e-15)


def test_frequency_denominator_reading(oracle_mod):
    """Partial RoPE: the denominator defaults to rot_dim; freq_dim = D selects
    base^(-2i/D) for the first rot_dim/2 pairs (both readings exposed)."""
    np.testing.assert_allclose(oracle_mod.rope_freqs(4, 10000.0), [1.0, 0.01], rtol=1e-15)
    np.testing.assert_allclose(oracle_mod.rope_freqs(4, 10000.0, freq_dim=8), [1.0, 0.1],
                               rtol=1e-15)


def test_tables_angle_addition(oracle_mod):
    """Table rows hold cos/sin of p*theta_i: column 0 is cos p / sin p
    (theta_0 = 1), cos^2 + sin^2 = 1, and rows combine by angle addition
    (row p+q from rows p and q), which fails for any other angle rule."""
    c, s = oracle_mod.rope_tables(300, 16, 10000.0)
    p = np.arange(300)
    np.testing.assert_allclose(c[:, 0], np.cos(p), atol=1e-15)
    np.testing.assert_allclose(s[:, 0], np.sin(p), atol=1e-15)
    np.testing.assert_allclose(c ** 2 + s ** 2, 1.0, atol=1e-15)
    for a, b in [(1, 2), (17, 100), (150, 149)]:
        np.testing.assert_allclose(c[a + b], c[a] * c[b] - s[a] * s[b], atol=1e-13)
        np.testing.assert_allclose(s[a + b], s[a] * c[b] + c[a] * s[b], atol=1e-13)


def test_rows_match_tables(oracle_mod):
    """rope_rows at position p uses exactly table row p."""
    c, s = oracle_mod.rope_tables(64, 8, 10000.0)
    x = np.zeros((1, 8))
    x[0, 0] = 1.0  # NeoX pair 0: (x0, x4) -> (cos, sin)
    y = oracle_mod.rope_rows(x, [37], layout=NEOX)
    assert y[0, 0] == c[37, 0] and y[0, 4] == s[37, 0]


@pytest.mark.parametrize("bad", [dict(D=7), dict(rot_dim=10), dict(rot_dim=3), dict(base=0.0),
                                 dict(base=-1.0), dict(rot_dim=0)])
def test_rejects_invalid(oracle_mod, bad):
    """"RoPE and FlashAttention ...", section 2: positive base and even width
    required; "Write Triton Rope Kernel": rot_dim <= D, even."""
    D = bad.get("D", 8)
    with pytest.raises(ValueError):
        oracle_mod.rope_rows(np.zeros((1, D)), [0], rot_dim=bad.get("rot_dim", D),
                             base=bad.get("base", 10000.0))


def test_rope_tokens_uses_token_positions(oracle_mod):
    """Token-major [T, H, D]: every head of token t uses positions[t], never
    the token index ("Write Triton Rope Kernel", step 3)."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 3, 8))
    pos = np.array([9, 0, 131000, 5, 5])
    y = oracle_mod.rope_tokens(x, pos)
    for t in range(5):
        for h in range(3):
            assert np.array_equal(y[t, h], oracle_mod.rope_rows(x[t, h][None], [pos[t]])[0])


def test_interpolated_tables_pins(oracle_mod):
    """Position interpolation ("RoPE and FlashAttention ...", section 3): the
    table at factor s holds the angles of positions p / s.  Factor 1 is the
    plain table bit for bit; row k*s at factor s (s a power of two, so p / s is
    exact) is row k of the plain table bit for bit; column 0 is cos(p / s)
    (theta_0 = 1); scores of rotated pairs still depend only on the (scaled)
    offset."""
    c1, s1 = oracle_mod.rope_tables(64, 8, 10000.0)
    cs, ss = oracle_mod.rope_tables_scaled(64, 8, 10000.0, 1.0)
    assert np.array_equal(c1, cs) and np.array_equal(s1, ss)
    c4, s4 = oracle_mod.rope_tables_scaled(256, 8, 10000.0, 4.0)
    assert np.array_equal(c4[::4], c1) and np.array_equal(s4[::4], s1)
    p = np.arange(256)
    np.testing.assert_allclose(c4[:, 0], np.cos(p / 4.0), atol=1e-15)
    c15, s15 = oracle_mod.rope_tables_scaled(300, 16, 500000.0, 1.5)
    # angle addition across rows: row a+b from rows a and b (angles are linear in p)
    for a, b in [(3, 7), (100, 150), (1, 298)]:
        np.testing.assert_allclose(c15[a + b], c15[a] * c15[b] - s15[a] * s15[b], atol=1e-13)
        np.testing.assert_allclose(s15[a + b], s15[a] * c15[b] + c15[a] * s15[b], atol=1e-13)
    # a larger base is not position division: theta_0 = 1 under any base, so
    # column 0 of a larger-base table is the plain column 0, while the
    # interpolated table's column 0 turns at 1/s the rate
    cb, _ = oracle_mod.rope_tables(64, 8, 40000.0)
    assert np.array_equal(cb[:, 0], c1[:, 0])
    assert not np.allclose(c4[:64, 0], c1[:, 0])
    assert not np.allclose(cb[:, 1], c1[:, 1])
