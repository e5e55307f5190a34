"""GPU parity: attn_fwd_causal_rope against the fp64 oracle.

Tolerances (max absolute error against the fp64 result): O <= 2e-2 for
bf16/fp16 inputs and <= 1e-4 for fp32 inputs; LSE <= 1e-3 for every dtype at
the default scale 1/sqrt(D) (for bf16/fp16 with a larger custom scale the LSE
bound grows by scale * sqrt(D), as the score error does).
Inputs are the seeded tensors of ``workloads``.
"""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

NEOX, GPTJ = 0, 1
TOL = {torch.float32: (1e-4, 1e-3), torch.bfloat16: (2e-2, 1e-3), torch.float16: (2e-2, 1e-3)}


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


def run_case(ra, orc, dt, B, Hq, Hkv, Sq, Sk, D, off, layout=NEOX, rot_dim=None, apply_rope=True,
             base=10000.0, seed=0, rows=None, scale=None, qkv=None, strided=False):
    q, k, v = qkv if qkv is not None else wl.attn_qkv(B, Hq, Hkv, Sq, Sk, D, dt, seed)
    r = rot_dim or D
    cos = sin = None
    if apply_rope:
        cos, sin = ra.make_tables(max(Sk, off + Sq), r, base)
    if strided:  # token-major [B, S, H, D] storage viewed as [B, H, S, D]
        qg = q.transpose(1, 2).contiguous().cuda().transpose(1, 2)
        kg = k.transpose(1, 2).contiguous().cuda().transpose(1, 2)
        vg = v.transpose(1, 2).contiguous().cuda().transpose(1, 2)
    else:
        qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    o, lse = ra.attn_fwd_causal_rope(qg, kg, vg, cos, sin, kv_offset=off, apply_rope=apply_rope,
                                     rot_dim=r if apply_rope else None, layout=layout,
                                     softmax_scale=scale)
    assert ra.ra_get_device_status() == 0
    o_ref, lse_ref = orc.attention(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                   kv_offset=off, apply_rope=apply_rope, rot_dim=r, base=base,
                                   layout=layout, scale=scale, rows=rows)
    og = o.float().cpu().numpy().reshape(-1, D)
    lg = lse.cpu().numpy().reshape(-1)
    if rows is not None:
        og, lg = og[rows], lg[rows]
    else:
        o_ref, lse_ref = o_ref.reshape(-1, D), lse_ref.reshape(-1)
    eo = np.abs(og - o_ref).max()
    el = np.abs(lg - lse_ref).max()
    to, tl = TOL[dt]
    if scale is not None and dt != torch.float32:
        # the fp16 rounding error of every score grows linearly with the scale:
        # the stated LSE bound applies at 1/sqrt(D) and scales with it
        tl *= max(1.0, scale * np.sqrt(D))
    assert np.isfinite(og).all() and np.isfinite(lg).all()
    assert eo <= to and el <= tl, f"O err {eo:.3g} (tol {to}), LSE err {el:.3g} (tol {tl})"
    return eo, el


# ------------------------------------------------------------------ fp32 path
def test_fp32_workload_full(ra, orc):
    """fp32, B=1 H=2 S=128 D=64, NeoX, base 1e4, positions 0..127, scale 1/8."""
    W = wl.FP32_ATTN
    run_case(ra, orc, torch.float32, W.B, W.Hq, W.Hkv, W.Sq, W.Sk, W.D, W.kv_offset,
             layout=W.layout, base=W.base, qkv=W.inputs(), scale=1 / 8)


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,off,layout,rot", [
    (1, 4, 2, 37, 50, 64, 13, GPTJ, None),
    (2, 2, 1, 70, 70, 32, 0, NEOX, 16),
    (1, 3, 3, 1, 90, 128, 89, NEOX, None),
    (1, 2, 1, 33, 33, 256, 0, GPTJ, 128),
    (1, 1, 1, 5, 9, 6, 2, NEOX, 4),
])
def test_fp32_cases(ra, orc, B, Hq, Hkv, Sq, Sk, D, off, layout, rot):
    run_case(ra, orc, torch.float32, B, Hq, Hkv, Sq, Sk, D, off, layout=layout, rot_dim=rot,
             seed=Sq + D)


def test_fp32_no_rope_matches_textbook(ra, orc):
    run_case(ra, orc, torch.float32, 1, 2, 2, 40, 60, 64, 20, apply_rope=False, seed=3)


# ------------------------------------------------------------ tensor-core path
TC_CASES = [
    # dt, B, Hq, Hkv, Sq, Sk, D, off, layout, rot
    (torch.bfloat16, 1, 1, 1, 1, 1, 64, 0, NEOX, None),
    (torch.bfloat16, 1, 2, 2, 128, 128, 64, 0, GPTJ, None),
    (torch.bfloat16, 1, 2, 1, 130, 130, 64, 0, NEOX, None),
    (torch.bfloat16, 2, 4, 2, 300, 300, 128, 0, NEOX, None),
    (torch.bfloat16, 1, 4, 1, 77, 300, 128, 223, GPTJ, None),
    (torch.bfloat16, 1, 8, 2, 200, 260, 128, 60, NEOX, 64),
    (torch.bfloat16, 1, 2, 2, 256, 256, 64, 0, GPTJ, 32),
    (torch.bfloat16, 1, 4, 4, 1, 1000, 128, 999, NEOX, None),
    (torch.bfloat16, 1, 3, 1, 129, 1500, 64, 1371, GPTJ, None),
    (torch.float16, 1, 4, 2, 190, 190, 128, 0, NEOX, None),
    (torch.float16, 2, 2, 2, 65, 100, 64, 35, GPTJ, None),
    # grids that fit on the SMs: one query tile per block, its key tiles
    # shared out between the two slots; odd and even tile counts, offsets,
    # ragged tiles, partial rotation, and (off = 129) rows with no admissible
    # key in slot 1's first tile
    (torch.bfloat16, 1, 3, 1, 700, 900, 64, 200, GPTJ, None),
    (torch.bfloat16, 2, 2, 2, 640, 640, 128, 0, NEOX, None),
    (torch.float16, 1, 1, 1, 1100, 1100, 128, 0, GPTJ, 64),
    (torch.bfloat16, 1, 2, 2, 300, 429, 64, 129, GPTJ, None),
    (torch.bfloat16, 1, 2, 1, 400, 400, 128, 0, NEOX, 64),
    # more blocks than SMs: adjacent tile pairs (one q head) and q-head pairs
    (torch.bfloat16, 1, 40, 40, 1000, 1000, 64, 0, NEOX, None),
    (torch.bfloat16, 2, 32, 8, 600, 600, 128, 0, NEOX, None),
    (torch.float16, 1, 64, 16, 640, 640, 64, 0, GPTJ, None),
    (torch.bfloat16, 1, 20, 20, 2000, 2000, 128, 0, GPTJ, None),
    # more blocks than SMs, D = 128, four and eight q-heads per kv head:
    # q-head pairs with ragged tiles, offsets and both layouts
    (torch.float16, 1, 32, 8, 1200, 1500, 128, 300, GPTJ, None),
    (torch.bfloat16, 1, 64, 8, 700, 777, 128, 77, NEOX, None),
    (torch.bfloat16, 3, 16, 4, 900, 900, 128, 0, GPTJ, None),
    # launch order in bands of four kv heads' head units, the last band
    # ragged: 18 units in bands of 8 (three batches), 10 units in bands of 4
    (torch.bfloat16, 3, 12, 3, 1200, 1300, 128, 100, NEOX, None),
    (torch.float16, 2, 10, 5, 2000, 2000, 64, 0, GPTJ, None),
]


@pytest.mark.parametrize("dt,B,Hq,Hkv,Sq,Sk,D,off,layout,rot", TC_CASES)
def test_tensor_core_cases(ra, orc, dt, B, Hq, Hkv, Sq, Sk, D, off, layout, rot):
    run_case(ra, orc, dt, B, Hq, Hkv, Sq, Sk, D, off, layout=layout, rot_dim=rot, seed=Sq * 3 + Sk)


@pytest.mark.parametrize("D", [64, 128])
def test_tensor_core_without_rope(ra, orc, D):
    """apply_rope = 0: plain causal flash attention (also the path for a cache
    of already-rotated keys)."""
    run_case(ra, orc, torch.bfloat16, 1, 4, 2, 260, 300, D, 40, apply_rope=False, seed=D)


@pytest.mark.parametrize("B,Hq,Hkv,S", [(2, 4, 2, 150), (2, 32, 8, 640)])
def test_tensor_core_strided_token_major(ra, orc, B, Hq, Hkv, S):
    """Q/K/V stored token-major [B, S, H, D] and passed as [B, H, S, D] views
    (a split-block grid, and a grid of q-head pairs past one wave)."""
    run_case(ra, orc, torch.bfloat16, B, Hq, Hkv, S, S, 128, 0, strided=True, seed=4)


def test_tensor_core_custom_scale(ra, orc):
    run_case(ra, orc, torch.bfloat16, 1, 2, 1, 140, 140, 64, 0, scale=0.3, seed=5)


@pytest.mark.parametrize("W", wl.SWEEP, ids=[w.name for w in wl.SWEEP])
def test_sweep_workloads_full(ra, orc, W):
    """bf16 GPT-J sweep B x 8 x S x 64 (S 512..4096, B 1..4): every row."""
    run_case(ra, orc, torch.bfloat16, W.B, W.Hq, W.Hkv, W.Sq, W.Sk, W.D, W.kv_offset,
             layout=W.layout, base=W.base, qkv=W.inputs())


def test_long_context_gqa_sampled_rows(ra, orc):
    """bf16 GQA 32 q-heads / 8 kv-heads, Sq 16384 new queries after a 4096-row
    cached prefix (Sk 20480), D 128, base 5e5, NeoX: full-size launch, checked
    on 1024 seeded random rows plus the first and last 128 rows of heads 0
    and 31."""
    W = wl.LONG_GQA
    rng = np.random.default_rng(77)
    n = W.B * W.Hq * W.Sq
    edge = []
    for h in (0, W.Hq - 1):
        base_row = h * W.Sq
        edge += list(range(base_row, base_row + 128)) + list(range(base_row + W.Sq - 128,
                                                                    base_row + W.Sq))
    rows = np.unique(np.concatenate([rng.integers(0, n, 1024), np.array(edge)]))
    run_case(ra, orc, torch.bfloat16, W.B, W.Hq, W.Hkv, W.Sq, W.Sk, W.D, W.kv_offset,
             layout=W.layout, base=W.base, qkv=W.inputs(), rows=rows)


def test_peak_extra_memory_bounded(ra):
    """Peak extra device memory of one call (beyond inputs and tables) stays
    within O + LSE: no rotated or expanded tensor is materialised."""
    B, Hq, Hkv, S, D = 1, 8, 8, 2048, 64
    q, k, v = [t.cuda() for t in wl.attn_qkv(B, Hq, Hkv, S, S, D, torch.bfloat16, 9)]
    cos, sin = ra.make_tables(S, D, 10000.0)
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    o, lse = ra.attn_fwd_causal_rope(q, k, v, cos, sin)
    torch.cuda.synchronize()
    extra = torch.cuda.max_memory_allocated() - base
    assert extra <= o.numel() * o.element_size() + lse.numel() * 4 + 1024


def test_rejections_with_real_buffers(ra):
    q, k, v = [t.cuda() for t in wl.attn_qkv(1, 2, 1, 16, 16, 64, torch.bfloat16, 1)]
    cos, sin = ra.make_tables(16, 64, 10000.0)
    with pytest.raises(ra.RAError) as e:
        ra.attn_fwd_causal_rope(q, k, v, cos, sin, kv_offset=-1)
    assert e.value.code == -1
    short_c, short_s = cos[:8], sin[:8]
    with pytest.raises(ra.RAError) as e:
        ra.attn_fwd_causal_rope(q, k, v, short_c.contiguous(), short_s.contiguous())
    assert e.value.code == -1
    q96 = torch.zeros(1, 2, 16, 96, dtype=torch.bfloat16, device="cuda")
    k96 = torch.zeros(1, 1, 16, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ra.RAError) as e:
        ra.attn_fwd_causal_rope(q96, k96, k96, apply_rope=False)
    assert e.value.code == -2
    assert ra.ra_get_device_status() == 0


@pytest.mark.parametrize("layout", [NEOX, GPTJ])
def test_unfused_rotate_then_flash_matches(ra, orc, layout):
    """The ablation path: rope_apply_qk into copies, then attention without
    RoPE.  Each stage is checked against the oracle on its own inputs: the
    materialised rotated Q/K (bf16, as rope_apply_qk returns them) fed to the
    no-RoPE kernel must match the oracle's attention of those same tensors at
    the standard tolerances, and its O must also match the fused result's
    oracle (bf16 rounding of the rotated operands moves LSE, not O, beyond
    the fused kernel's bound: the fused kernel keeps them in fp16)."""
    B, H, S, D = 2, 4, 300, 64
    q, k, v = wl.attn_qkv(B, H, H, S, S, D, torch.bfloat16, seed=31)
    cos, sin = ra.make_tables(S, D, 10000.0)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    qr, kr = torch.empty_like(qg), torch.empty_like(kg)
    pos = torch.arange(S, dtype=torch.int32, device="cuda")
    for b in range(B):
        ra.rope_apply_qk(qg[b].transpose(0, 1), kg[b].transpose(0, 1), pos, cos, sin,
                         layout=layout, q_out=qr[b].transpose(0, 1), k_out=kr[b].transpose(0, 1))
    o_u, lse_u = ra.attn_fwd_causal_rope(qr, kr, vg, apply_rope=False)
    assert ra.ra_get_device_status() == 0
    qr_c, kr_c = qr.float().cpu().numpy(), kr.float().cpu().numpy()
    o_ref_u, lse_ref_u = orc.attention(qr_c, kr_c, v.float().numpy(), apply_rope=False)
    assert np.abs(o_u.float().cpu().numpy() - o_ref_u).max() <= 2e-2
    assert np.abs(lse_u.cpu().numpy() - lse_ref_u).max() <= 1e-3
    o_ref, _ = orc.attention(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                             layout=layout)
    assert np.abs(o_u.float().cpu().numpy() - o_ref).max() <= 2e-2


def test_past_2g_elements_sampled_rows(ra, orc):
    """Q, K, V and O with more than 2^31 elements each (1040 x 16 x 1024 x 128,
    4.4 GB per tensor): 64-bit offsets in every tensor map and store.  One
    seeded batch is repeated along B on the device, so every batch computes
    the same attention; 256 sampled rows and the edge rows of the first and
    the last batch are checked against the oracle on that batch."""
    B, H, S, D = 1040, 16, 1024, 128
    qb, kb, vb = wl.attn_qkv(1, H, H, S, S, D, torch.bfloat16, 41)
    qg, kg, vg = [t.cuda().expand(B, H, S, D).contiguous() for t in (qb, kb, vb)]
    assert qg.numel() > 2 ** 31
    cos, sin = ra.make_tables(S, D, 10000.0)
    o, lse = ra.attn_fwd_causal_rope(qg, kg, vg, cos, sin)
    assert ra.ra_get_device_status() == 0
    del qg, kg, vg
    rng = np.random.default_rng(42)
    rows = np.unique(np.concatenate([rng.integers(0, H * S, 256), np.arange(128),
                                     np.arange(H * S - 128, H * S)]))
    o_ref, lse_ref = orc.attention(qb.float().numpy(), kb.float().numpy(), vb.float().numpy(),
                                   rows=rows)
    to, tl = TOL[torch.bfloat16]
    for bi in (0, B - 1):
        og = o[bi].reshape(-1, D)[torch.from_numpy(rows).cuda()].float().cpu().numpy()
        lg = lse[bi].reshape(-1)[torch.from_numpy(rows).cuda()].cpu().numpy()
        assert np.abs(og - o_ref).max() <= to
        assert np.abs(lg - lse_ref).max() <= tl
    del o, lse
    torch.cuda.empty_cache()
