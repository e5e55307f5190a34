"""fp16 operand range of the tensor-core attention ("Write Triton Rope
Kernel", Correctness requirements and Common failure modes: the precision of
the rotated values).

The tensor-core paths round the rotated Q and K (and the backward's
dS = P o (dP - D)) to fp16.  A value that does not round to a finite fp16
must not come back as a silent NaN: the call records RA_ERR_RANGE in the
device status word.  Inputs whose magnitude stays within 32752 always fit
(a rotated pair member is at most |lo| + |hi|), so they must not raise it.
"""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

RANGE = -8
NEOX, GPTJ = 0, 1


@pytest.fixture(scope="module")
def ra():
    import __graft_entry__
    __graft_entry__.build()
    import rope_causal_attention_gb300 as m
    assert m.ra_get_device_status() == 0
    return m


def fwd(ra, q, k, v, off=0, layout=NEOX, apply_rope=True, base=10000.0):
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    cos = sin = None
    if apply_rope:
        cos, sin = ra.make_tables(max(k.shape[2], off + q.shape[2]), q.shape[3], base)
    o, lse = ra.attn_fwd_causal_rope(qg, kg, vg, cos, sin, kv_offset=off, layout=layout,
                                     apply_rope=apply_rope)
    return o, lse, ra.ra_get_device_status()


# (B, Hq, Hkv, S, D, layout): a split-block grid (one wave) and a paired grid
GRIDS = [(1, 2, 2, 300, 128, NEOX), (1, 8, 2, 8192, 128, NEOX), (1, 4, 4, 700, 64, GPTJ)]


@pytest.mark.parametrize("B,Hq,Hkv,S,D,layout", GRIDS)
def test_query_overflow_is_reported(ra, B, Hq, Hkv, S, D, layout):
    q, k, v = wl.attn_qkv(B, Hq, Hkv, S, S, D, torch.bfloat16, seed=S)
    q[0, Hq - 1, S // 2 + 3, 5] = 1.0e5
    _, _, st = fwd(ra, q, k, v, layout=layout)
    assert st == RANGE


@pytest.mark.parametrize("B,Hq,Hkv,S,D,layout", GRIDS)
@pytest.mark.parametrize("where", [0.03, 0.61, 0.99])
def test_key_overflow_is_reported(ra, B, Hq, Hkv, S, D, layout, where):
    """A key row anywhere in the sequence: the first query tile's CTAs check
    the prefix, later CTAs the key tiles their predecessors do not reach."""
    q, k, v = wl.attn_qkv(B, Hq, Hkv, S, S, D, torch.bfloat16, seed=S + 1)
    k[0, Hkv - 1, int(where * (S - 1)), 2] = -1.0e5
    _, _, st = fwd(ra, q, k, v, layout=layout)
    assert st == RANGE


def test_key_overflow_in_the_cached_prefix(ra):
    q, k, v = wl.attn_qkv(1, 8, 2, 1024, 1024 + 640, 128, torch.bfloat16, seed=3)
    k[0, 1, 600, 100] = 2.0e5
    _, _, st = fwd(ra, q, k, v, off=640, base=500000.0)
    assert st == RANGE


def test_unrotated_bf16_beyond_fp16_is_reported(ra):
    """Without RoPE the bf16 rows are still rounded to fp16 operands."""
    q, k, v = wl.attn_qkv(1, 2, 1, 256, 256, 64, torch.bfloat16, seed=4)
    k[0, 0, 200, 7] = 7.0e4
    _, _, st = fwd(ra, q, k, v, apply_rope=False)
    assert st == RANGE


@pytest.mark.parametrize("B,Hq,Hkv,S,D,layout", GRIDS)
def test_large_values_that_fit_are_not_reported(ra, B, Hq, Hkv, S, D, layout):
    """One element of +-32000 in every Q row and in every K row: a rotated
    value is at most |lo| + |hi| < 65504, so everything fits and the status
    stays OK.  The large Q and K elements sit in different rotation pairs,
    so the scores stay moderate (|s| ~ 1e5) and O / LSE stay finite."""
    q, k, v = wl.attn_qkv(B, Hq, Hkv, S, S, D, torch.bfloat16, seed=S + 2)
    q[..., 5] = torch.where(q[..., 5] < 0, -32000.0, 32000.0).to(torch.bfloat16)
    k[..., 40] = torch.where(k[..., 40] < 0, -32000.0, 32000.0).to(torch.bfloat16)
    o, lse, st = fwd(ra, q, k, v, layout=layout)
    assert st == 0
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())


def bwd(ra, q, k, v, dout, off=0):
    qg, kg, vg, dg = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    cos, sin = ra.make_tables(max(k.shape[2], off + q.shape[2]), q.shape[3], 10000.0)
    o, lse = ra.attn_fwd_causal_rope(qg, kg, vg, cos, sin, kv_offset=off)
    st_fwd = ra.ra_get_device_status()
    ra.attn_bwd_causal_rope(qg, kg, vg, o, lse, dg, cos, sin, kv_offset=off)
    return st_fwd, ra.ra_get_device_status()


def test_backward_rotation_overflow_is_reported(ra):
    q, k, v = wl.attn_qkv(1, 4, 2, 384, 384, 128, torch.bfloat16, seed=5)
    dout = wl.randn((1, 4, 384, 128), torch.Generator("cpu").manual_seed(6), torch.bfloat16)
    k[0, 1, 77, 9] = 1.0e5
    st_fwd, st_bwd = bwd(ra, q, k, v, dout)
    assert st_fwd == RANGE and st_bwd == RANGE


def test_backward_ds_overflow_is_reported(ra):
    """|dO| and |V| of 1000: dP - D reaches ~1e7, so dS = P o (dP - D)
    leaves the fp16 range; the forward itself is in range."""
    q, k, v = wl.attn_qkv(1, 4, 2, 384, 384, 128, torch.bfloat16, seed=7)
    dout = wl.randn((1, 4, 384, 128), torch.Generator("cpu").manual_seed(8), torch.bfloat16)
    v = (v.float() * 1000.0).to(torch.bfloat16)
    dout = (dout.float() * 1000.0).to(torch.bfloat16)
    st_fwd, st_bwd = bwd(ra, q, k, v, dout)
    assert st_fwd == 0 and st_bwd == RANGE


def test_backward_in_range_is_not_reported(ra):
    q, k, v = wl.attn_qkv(1, 4, 2, 384, 384, 128, torch.bfloat16, seed=9)
    dout = wl.randn((1, 4, 384, 128), torch.Generator("cpu").manual_seed(10), torch.bfloat16)
    st_fwd, st_bwd = bwd(ra, q, k, v, dout)
    assert st_fwd == 0 and st_bwd == 0
