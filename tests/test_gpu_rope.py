"""GPU parity: rope_tables_build and rope_apply_qk against the fp64 oracle.

Tolerances (stated for the standalone rotation): fp32 outputs within 1e-5
absolute of the fp64 result; bf16/fp16 outputs within 1 ulp of the fp64
result (plus the fp32-table allowance described in check_rotated); the
unrotated tail bit-identical.  Tables
within 2^-24 absolute of the fp64 cos/sin and almost always equal to their
fp32 rounding (the device's fp64 pow/sincos and the host's libm may differ in
the last fp64 bit, which can flip a rounding).
"""
import numpy as np
import pytest
import torch

import workloads as wl
from rope_check import check_rotated, pair_partner, ulp_of  # noqa: F401

pytestmark = pytest.mark.gpu

NEOX, GPTJ = 0, 1


@pytest.fixture(scope="module")
def ra():
    import __graft_entry__
    __graft_entry__.build()
    import rope_causal_attention_gb300 as m
    assert m.ra_get_device_status() == 0
    return m


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.mark.parametrize("rows,rot_dim,base,freq_dim", [(1, 2, 10000.0, 0), (4096, 64, 10000.0, 0),
                                                        (32768, 128, 10000.0, 0),
                                                        (131072, 64, 10000.0, 0),
                                                        (20480, 128, 500000.0, 0),
                                                        (300, 32, 10000.0, 128)])
def test_tables_match_oracle(ra, orc, rows, rot_dim, base, freq_dim):
    c, s = ra.make_tables(rows, rot_dim, base, freq_dim)
    torch.cuda.synchronize()
    wc, ws = orc.rope_tables(rows, rot_dim, base, freq_dim)
    for got, want in ((c, wc), (s, ws)):
        g = got.cpu().double().numpy()
        # values lie in [-1, 1]: rounding to fp32 moves them by at most 2^-25,
        # and a last-bit difference in the fp64 angle adds far less than that
        assert np.abs(g - want).max() <= 2.0 ** -24
        exact = g == want.astype(np.float32).astype(np.float64)
        assert exact.mean() > 0.999  # nearly every entry is the correctly rounded value


CASES = [
    # dtype, T, Hq, Hkv, D, rot_dim, layout
    (torch.bfloat16, 37, 4, 2, 128, 128, NEOX),
    (torch.bfloat16, 37, 4, 2, 128, 128, GPTJ),
    (torch.bfloat16, 19, 8, 1, 128, 64, NEOX),
    (torch.bfloat16, 19, 8, 1, 128, 32, GPTJ),
    (torch.float16, 23, 3, 3, 64, 64, NEOX),
    (torch.float16, 23, 3, 3, 64, 48, GPTJ),
    (torch.float32, 11, 2, 2, 64, 64, NEOX),
    (torch.float32, 11, 2, 2, 64, 36, GPTJ),
    (torch.float32, 11, 5, 1, 96, 16, NEOX),
    # scalar-kernel cases: widths that break 16-byte vectors
    (torch.bfloat16, 9, 3, 1, 10, 6, NEOX),
    (torch.bfloat16, 9, 3, 1, 2, 2, GPTJ),
    (torch.float32, 7, 2, 1, 6, 4, GPTJ),
    (torch.float16, 5, 2, 2, 24, 12, NEOX),
]


@pytest.mark.parametrize("in_place", [True, False])
@pytest.mark.parametrize("pos64", [False, True])
@pytest.mark.parametrize("dt,T,Hq,Hkv,D,rot_dim,layout", CASES)
def test_rope_apply_matches_oracle(ra, orc, dt, T, Hq, Hkv, D, rot_dim, layout, in_place, pos64):
    q, k = wl.rope_qk(T, Hq, Hkv, D, dt, seed=T * 7 + D)
    pos, _, _ = wl.continuous_batch_positions(3, T, T, 5000, seed=D + rot_dim)
    cos, sin = ra.make_tables(5000, rot_dim, 10000.0)
    posg = torch.from_numpy(pos).to(torch.int64 if pos64 else torch.int32).cuda()
    qg, kg = q.cuda(), k.cuda()
    if in_place:
        ra.rope_apply_qk(qg, kg, posg, cos, sin, layout=layout)
        qr, kr = qg, kg
    else:
        qo, ko = torch.full_like(qg, 7.0), torch.full_like(kg, 7.0)
        qr, kr = ra.rope_apply_qk(qg, kg, posg, cos, sin, layout=layout, q_out=qo, k_out=ko)
        assert torch.equal(qg.cpu(), q) and torch.equal(kg.cpu(), k)  # inputs untouched
    assert ra.ra_get_device_status() == 0
    check_rotated(qr, q, pos, orc, rot_dim, 10000.0, layout)
    check_rotated(kr, k, pos, orc, rot_dim, 10000.0, layout)


def test_strided_views_and_packed_qkv(ra, orc):
    """Q and K as views of one packed [T, Hq + 2*Hkv, D] buffer (token stride
    larger than a head row); V, in the same buffer, must stay bit-identical."""
    T, Hq, Hkv, D = 33, 4, 2, 128
    g = torch.Generator().manual_seed(3)
    qkv = torch.randn(T, Hq + 2 * Hkv, D, generator=g).to(torch.bfloat16)
    pos = np.arange(100, 100 + T)
    cos, sin = ra.make_tables(512, D, 10000.0)
    dev = qkv.cuda()
    q, k, v = dev[:, :Hq], dev[:, Hq:Hq + Hkv], dev[:, Hq + Hkv:]
    ra.rope_apply_qk(q, k, torch.from_numpy(pos).cuda(), cos, sin)
    assert ra.ra_get_device_status() == 0
    check_rotated(q, qkv[:, :Hq], pos, orc, D, 10000.0, NEOX)
    check_rotated(k, qkv[:, Hq:Hq + Hkv], pos, orc, D, 10000.0, NEOX)
    assert torch.equal(v.cpu(), qkv[:, Hq + Hkv:])


def test_q_only_and_k_only(ra, orc):
    q, k = wl.rope_qk(8, 2, 2, 64, torch.bfloat16, seed=1)
    pos = np.array([5, 1, 9, 0, 3, 3, 8, 2])
    cos, sin = ra.make_tables(16, 64, 10000.0)
    qg = q.cuda()
    ra.rope_apply_qk(qg, None, torch.from_numpy(pos).cuda(), cos, sin)
    kg = k.cuda()
    ra.rope_apply_qk(None, kg, torch.from_numpy(pos).cuda(), cos, sin, layout=GPTJ)
    assert ra.ra_get_device_status() == 0
    check_rotated(qg, q, pos, orc, 64, 10000.0, NEOX)
    check_rotated(kg, k, pos, orc, 64, 10000.0, GPTJ)


def test_position_out_of_range_flags_and_skips(ra, orc):
    """A position outside the table records RA_ERR_POSITION_RANGE and leaves
    that token untouched; the other tokens are rotated."""
    q, k = wl.rope_qk(6, 2, 1, 64, torch.bfloat16, seed=2)
    pos = torch.tensor([0, 3, 16, -1, 7, 15], dtype=torch.int32)
    cos, sin = ra.make_tables(16, 64, 10000.0)
    qg, kg = q.cuda(), k.cuda()
    ra.rope_apply_qk(qg, kg, pos.cuda(), cos, sin)
    assert ra.ra_get_device_status() == -7
    assert ra.ra_get_device_status() == 0  # read clears it
    bad = [2, 3]
    good = [0, 1, 4, 5]
    assert torch.equal(qg.cpu()[bad], q[bad]) and torch.equal(kg.cpu()[bad], k[bad])
    check_rotated(qg[good], q[good], pos.numpy()[good], orc, 64, 10000.0, NEOX)


def test_overlap_rejected_with_real_buffers(ra):
    """An output that starts inside its input (neither equal nor disjoint) is
    rejected on the host with RA_ERR_OVERLAP; nothing is written."""
    q, k = wl.rope_qk(8, 2, 2, 64, torch.bfloat16, seed=1)
    cos, sin = ra.make_tables(16, 64, 10000.0)
    buf = torch.zeros(8 * 2 * 64 + 64, dtype=torch.bfloat16, device="cuda")
    qg = buf[:8 * 2 * 64].view(8, 2, 64)
    qg.copy_(q.cuda())
    q_out = buf[8:8 + 8 * 2 * 64].view(8, 2, 64)
    kg = k.cuda()
    pos = torch.zeros(8, dtype=torch.int32, device="cuda")
    with pytest.raises(ra.RAError) as e:
        ra.rope_apply_qk(qg, kg, pos, cos, sin, q_out=q_out)
    assert e.value.code == -4
    assert torch.equal(qg.cpu(), q) and torch.equal(kg.cpu(), k)


def test_decode_workload_full(ra, orc):
    """512 decode tokens at positions up to 131071, 64 + 8 heads, D = 128,
    partial rot_dim 64 (NeoX), in place: every token against the oracle, the
    tail bit-identical."""
    W = wl.DECODE_ROPE
    q, k = W.inputs()
    pos = W.positions()
    cos, sin = ra.make_tables(W.table_rows, W.rot_dim, W.base)
    qg, kg = q.cuda(), k.cuda()
    ra.rope_apply_qk(qg, kg, torch.from_numpy(pos).to(torch.int32).cuda(), cos, sin,
                     layout=W.layout)
    assert ra.ra_get_device_status() == 0
    check_rotated(qg, q, pos, orc, W.rot_dim, W.base, W.layout)
    check_rotated(kg, k, pos, orc, W.rot_dim, W.base, W.layout)


def test_continuous_batching_workload_full_size(ra, orc):
    """T = 65536 packed tokens of 256 requests (lengths 1..512, starts inside a
    32768-row table), 32 + 8 heads, D = 128, in place, as timed by the bench;
    checked on 2048 sampled tokens plus the first and last token."""
    W = wl.CB_ROPE
    q, k = W.inputs()
    pos = W.positions()
    assert pos.shape[0] == W.T and pos.max() < W.table_rows and pos.min() >= 0
    cos, sin = ra.make_tables(W.table_rows, W.rot_dim, W.base)
    qg, kg = q.cuda(), k.cuda()
    ra.rope_apply_qk(qg, kg, torch.from_numpy(pos).to(torch.int32).cuda(), cos, sin,
                     layout=W.layout)
    assert ra.ra_get_device_status() == 0
    rng = np.random.default_rng(0)
    sel = np.unique(np.concatenate([[0, W.T - 1], rng.integers(0, W.T, 2048)]))
    idx = torch.from_numpy(sel)
    check_rotated(qg.cpu()[idx], q[idx], pos[sel], orc, W.rot_dim, W.base, W.layout)
    check_rotated(kg.cpu()[idx], k[idx], pos[sel], orc, W.rot_dim, W.base, W.layout)


@pytest.mark.parametrize("scale,rows,rot_dim,base", [(1.0, 4096, 64, 10000.0), (4.0, 8192, 128, 10000.0),
                                                    (1.5, 3000, 64, 500000.0)])
def test_interpolated_tables_match_oracle(ra, orc, scale, rows, rot_dim, base):
    """rope_tables_build_scaled (position interpolation) against the oracle,
    same bound as the plain tables; a rotation through the scaled table equals
    the oracle's rotation at fractional positions p / scale."""
    c, s = ra.make_tables(rows, rot_dim, base, pos_scale=scale)
    torch.cuda.synchronize()
    wc, ws = orc.rope_tables_scaled(rows, rot_dim, base, scale)
    for got, want in ((c, wc), (s, ws)):
        g = got.cpu().double().numpy()
        assert np.abs(g - want).max() <= 2.0 ** -24
        assert (g == want.astype(np.float32).astype(np.float64)).mean() > 0.999
    q, k = wl.rope_qk(16, 2, 1, rot_dim, torch.float32, seed=8)
    pos = np.arange(0, rows, rows // 16)[:16]
    qg, kg = q.cuda(), k.cuda()
    ra.rope_apply_qk(qg, kg, torch.from_numpy(pos).cuda(), c, s)
    xr = q.double().numpy()
    want_q = np.empty_like(xr)
    half = rot_dim // 2
    for t in range(16):
        lo, hi = xr[t, :, :half], xr[t, :, half:]
        want_q[t, :, :half] = lo * wc[pos[t]] - hi * ws[pos[t]]
        want_q[t, :, half:] = hi * wc[pos[t]] + lo * ws[pos[t]]
    assert np.abs(qg.cpu().double().numpy() - want_q).max() <= 1e-5


def test_past_2g_elements_sampled_tokens(ra, orc):
    """Q with more than 2^31 elements (2^21 + 7 tokens x 8 heads x 128, 4.3 GB):
    64-bit token offsets.  A seeded 4096-token block is repeated along T on
    the device and every token takes a random position; tokens at both ends
    and 512 sampled tokens are checked against the oracle."""
    T, Hq, Hkv, D, R = (1 << 21) + 7, 8, 2, 128, 32768
    qb, kb, _ = wl.attn_qkv(1, Hq, Hkv, 4096, 4096, D, torch.bfloat16, 31)
    qb, kb = qb[0].transpose(0, 1).contiguous(), kb[0].transpose(0, 1).contiguous()  # [4096, H, D]
    reps = (T + 4095) // 4096
    qg = qb.cuda().repeat(reps, 1, 1)[:T].contiguous()
    kg = kb.cuda().repeat(reps, 1, 1)[:T].contiguous()
    assert qg.numel() > 2 ** 31
    pos = np.random.default_rng(31).integers(0, R, T).astype(np.int32)
    cos, sin = ra.make_tables(R, D, 10000.0)
    ra.rope_apply_qk(qg, kg, torch.from_numpy(pos).cuda(), cos, sin, layout=NEOX)
    assert ra.ra_get_device_status() == 0
    rng = np.random.default_rng(32)
    sel = np.unique(np.concatenate([np.arange(16), np.arange(T - 16, T), rng.integers(0, T, 512)]))
    idx = torch.from_numpy(sel)
    src = torch.from_numpy(sel % 4096)
    check_rotated(qg[idx.cuda()].cpu(), qb[src], pos[sel], orc, D, 10000.0, NEOX)
    check_rotated(kg[idx.cuda()].cpu(), kb[src], pos[sel], orc, D, 10000.0, NEOX)
    del qg, kg
    torch.cuda.empty_cache()
