"""GPU parity of attn_bwd_causal_rope against the fp64 backward oracle.

Tolerances: gradients compared normwise per tensor, max |got - ref| <=
tol * max(1, max |ref|) with tol = 1e-4 for fp32 (fp32 accumulation over at
most a few thousand unit-scale terms) and 2e-2 for bf16 / fp16 (outputs
rounded to the 16-bit dtype, rotated Q/K and dS rounded to fp16 and P to the
input dtype before their products, as in the forward's O bound)."""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

NEOX, GPTJ = 0, 1
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2, torch.float16: 2e-2}


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


def grads_case(ra, orc, dt, B, Hq, Hkv, Sq, Sk, D, off, layout, rot_dim, apply_rope=True,
               scale=None, seed=0, base=10000.0):
    q, k, v = wl.attn_qkv(B, Hq, Hkv, Sq, Sk, D, dt, seed=seed)
    g = torch.Generator("cpu").manual_seed(seed + 99)
    dout = wl.randn((B, Hq, Sq, D), g, dt)
    qg, kg, vg, dg = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    cos = sin = None
    if apply_rope:
        cos, sin = ra.make_tables(max(Sk, off + Sq), rot_dim, base)
    o, lse = ra.attn_fwd_causal_rope(qg, kg, vg, cos, sin, kv_offset=off, apply_rope=apply_rope,
                                     layout=layout, softmax_scale=scale)
    dq, dk, dv = ra.attn_bwd_causal_rope(qg, kg, vg, o, lse, dg, cos, sin, kv_offset=off,
                                         apply_rope=apply_rope, layout=layout,
                                         softmax_scale=scale)
    assert ra.ra_get_device_status() == 0
    want = orc.attention_bwd(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                             dout.float().numpy(), kv_offset=off, apply_rope=apply_rope,
                             rot_dim=rot_dim, base=base, layout=layout, scale=scale)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), want):
        err = np.abs(got.float().cpu().numpy().astype(np.float64) - ref).max()
        bound = TOL[dt] * max(1.0, np.abs(ref).max())
        assert err <= bound, (name, err, bound)
    return dq, dk, dv


FP32_CASES = [
    # B, Hq, Hkv, Sq, Sk, D, off, layout, rot_dim
    (1, 2, 2, 128, 128, 64, 0, NEOX, 64),     # the fp32 workload's shape
    (2, 4, 2, 50, 70, 64, 20, GPTJ, 32),      # GQA, offset, partial rotation
    (1, 3, 1, 33, 33, 96, 0, NEOX, 96),
    (1, 2, 1, 17, 40, 32, 5, GPTJ, 32),       # keys past the last query: zero gradient
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,off,layout,rot_dim", FP32_CASES)
def test_fp32_backward_matches_oracle(ra, orc, B, Hq, Hkv, Sq, Sk, D, off, layout, rot_dim):
    dq, dk, dv = grads_case(ra, orc, torch.float32, B, Hq, Hkv, Sq, Sk, D, off, layout, rot_dim,
                            seed=Sq + D)
    assert ra.ra_last_launch() == ["bwd_rowterm_kernel", "bwd_dq_simt_kernel",
                                   "bwd_dkdv_simt_kernel"]
    if Sk > off + Sq:
        assert bool((dk[:, :, off + Sq:] == 0).all()) and bool((dv[:, :, off + Sq:] == 0).all())


def test_fp32_backward_no_rope_custom_scale(ra, orc):
    grads_case(ra, orc, torch.float32, 1, 4, 2, 40, 60, 64, 20, NEOX, 64, apply_rope=False,
               scale=0.2, seed=3)


def test_fp32_fused_workload(ra, orc):
    W = wl.FP32_ATTN
    grads_case(ra, orc, torch.float32, W.B, W.Hq, W.Hkv, W.Sq, W.Sk, W.D, W.kv_offset, W.layout,
               W.r, seed=W.seed, base=W.base, scale=1.0 / 8)


TC_CASES = [
    # dt, B, Hq, Hkv, Sq, Sk, D, off, layout, rot_dim
    (torch.bfloat16, 1, 2, 2, 128, 128, 128, 0, NEOX, 128),
    (torch.bfloat16, 1, 4, 2, 300, 300, 128, 0, GPTJ, 128),
    (torch.float16, 2, 2, 1, 200, 456, 128, 256, NEOX, 128),
    (torch.bfloat16, 1, 2, 2, 257, 257, 64, 0, GPTJ, 64),
    (torch.float16, 1, 4, 4, 130, 200, 64, 70, NEOX, 32),
    (torch.bfloat16, 1, 8, 2, 512, 512, 128, 0, NEOX, 64),
    (torch.bfloat16, 1, 2, 1, 100, 400, 128, 100, GPTJ, 128),  # keys past the last query
    (torch.float16, 1, 4, 2, 190, 220, 128, 30, GPTJ, 48),     # GPT-J partial: unrotated tail
]


@pytest.mark.parametrize("dt,B,Hq,Hkv,Sq,Sk,D,off,layout,rot_dim", TC_CASES)
def test_tc_backward_matches_oracle(ra, orc, dt, B, Hq, Hkv, Sq, Sk, D, off, layout, rot_dim):
    grads_case(ra, orc, dt, B, Hq, Hkv, Sq, Sk, D, off, layout, rot_dim, seed=Sq + D + off)
    assert "bwd_dkdv_tc_kernel" in ra.ra_last_launch()
    assert "bwd_dq_tc_kernel" in ra.ra_last_launch()


def test_tc_backward_no_rope(ra, orc):
    grads_case(ra, orc, torch.bfloat16, 1, 4, 2, 200, 260, 128, 60, NEOX, 128, apply_rope=False,
               seed=8)


def test_tc_backward_mid_size_gqa_offset(ra, orc):
    """Every row of a mid-size case on the long-context paths: four q-heads
    per kv head, a 512-row cached prefix, base 5e5, NeoX, D = 128, 16 query
    tiles against 20 key tiles."""
    grads_case(ra, orc, torch.bfloat16, 1, 8, 2, 2048, 2560, 128, 512, NEOX, 128, seed=77,
               base=500000.0)


def sample_rows(rng, n_all, n, edge):
    """n seeded random flat rows plus the first and last `edge` rows."""
    pick = rng.choice(n_all, size=n, replace=False)
    return np.unique(np.concatenate([pick, np.arange(edge), np.arange(n_all - edge, n_all)]))


def test_tc_backward_long_context_workload_sampled(ra, orc):
    """The long-context GQA workload at full size, called exactly as the
    benchmark times it (same inputs, dO seeded seed + 7, caller workspace):
    dq on 1024 seeded query rows plus the first and last 128 of the tensor,
    dk and dv on 256 seeded key rows of one kv head plus its first and last
    64, against the selected-rows backward oracle."""
    W = wl.LONG_GQA
    dt = wl.DTYPES[W.dtype]
    q, k, v = W.inputs()
    g = torch.Generator("cpu").manual_seed(W.seed + 7)
    dout = wl.randn((W.B, W.Hq, W.Sq, W.D), g, dt)
    qg, kg, vg, dg = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    cos, sin = ra.make_tables(max(W.Sk, W.kv_offset + W.Sq), W.r, W.base)
    o, lse = ra.attn_fwd_causal_rope(qg, kg, vg, cos, sin, kv_offset=W.kv_offset,
                                     layout=W.layout)
    dq, dk, dv = (torch.empty_like(t) for t in (qg, kg, vg))
    wsb = int(ra.lib().attn_bwd_workspace_size(1, W.B, W.Hq, W.Hkv, W.Sq, W.Sk, W.D))
    wsp = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    ra.attn_bwd_causal_rope(qg, kg, vg, o, lse, dg, cos, sin, kv_offset=W.kv_offset,
                            layout=W.layout, dq=dq, dk=dk, dv=dv, workspace=wsp)
    assert ra.ra_get_device_status() == 0
    assert "bwd_dkdv_tc_kernel" in ra.ra_last_launch()
    rng = np.random.default_rng(W.seed)
    qrows = sample_rows(rng, W.B * W.Hq * W.Sq, 1024, 128)
    hk = int(rng.integers(0, W.Hkv))
    krows = hk * W.Sk + sample_rows(rng, W.Sk, 256, 64)
    ref_dq, ref_dk, ref_dv = orc.attention_bwd_rows(
        q.float().numpy(), k.float().numpy(), v.float().numpy(), dout.float().numpy(),
        dq_rows=qrows, dkv_rows=krows, kv_offset=W.kv_offset, base=W.base, layout=W.layout)
    got = {"dq": dq.float().cpu().numpy().reshape(-1, W.D)[qrows],
           "dk": dk.float().cpu().numpy().reshape(-1, W.D)[krows],
           "dv": dv.float().cpu().numpy().reshape(-1, W.D)[krows]}
    for name, ref in (("dq", ref_dq), ("dk", ref_dk), ("dv", ref_dv)):
        assert np.isfinite(got[name]).all(), name
        err = np.abs(got[name].astype(np.float64) - ref).max()
        bound = TOL[dt] * max(1.0, np.abs(ref).max())
        assert err <= bound, (name, err, bound)


def test_tc_backward_ragged_launch_bands_sampled(ra, orc):
    """Grids past one wave run in bands of four kv heads' work: with five kv
    heads the dK/dV grid (40 key tiles x 5 kv heads) has bands of 4 + 1 kv
    heads and the dQ grid (32 query tiles x 10 q-heads) bands of 8 + 2
    q-heads.  dq on 512 seeded query rows plus the first and last 64, dk/dv
    on 128 seeded key rows plus the first and last 32 of kv head 0 and of
    kv head 4 (the ragged band), against the selected-rows oracle."""
    B, Hq, Hkv, Sq, Sk, D, off, base = 1, 10, 5, 4096, 5120, 128, 1024, 500000.0
    dt = torch.bfloat16
    q, k, v = wl.attn_qkv(B, Hq, Hkv, Sq, Sk, D, dt, seed=61)
    g = torch.Generator("cpu").manual_seed(62)
    dout = wl.randn((B, Hq, Sq, D), g, dt)
    qg, kg, vg, dg = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    cos, sin = ra.make_tables(Sk, D, base)
    o, lse = ra.attn_fwd_causal_rope(qg, kg, vg, cos, sin, kv_offset=off)
    dq, dk, dv = ra.attn_bwd_causal_rope(qg, kg, vg, o, lse, dg, cos, sin, kv_offset=off)
    assert ra.ra_get_device_status() == 0
    assert "bwd_dkdv_tc_kernel" in ra.ra_last_launch()
    rng = np.random.default_rng(63)
    qrows = sample_rows(rng, B * Hq * Sq, 512, 64)
    krows = np.concatenate([hk * Sk + sample_rows(rng, Sk, 128, 32) for hk in (0, Hkv - 1)])
    ref_dq, ref_dk, ref_dv = orc.attention_bwd_rows(
        q.float().numpy(), k.float().numpy(), v.float().numpy(), dout.float().numpy(),
        dq_rows=qrows, dkv_rows=krows, kv_offset=off, base=base, layout=NEOX)
    got = {"dq": dq.float().cpu().numpy().reshape(-1, D)[qrows],
           "dk": dk.float().cpu().numpy().reshape(-1, D)[krows],
           "dv": dv.float().cpu().numpy().reshape(-1, D)[krows]}
    for name, ref in (("dq", ref_dq), ("dk", ref_dk), ("dv", ref_dv)):
        assert np.isfinite(got[name]).all(), name
        err = np.abs(got[name].astype(np.float64) - ref).max()
        bound = TOL[dt] * max(1.0, np.abs(ref).max())
        assert err <= bound, (name, err, bound)


def test_backward_rejections(ra):
    q = torch.zeros((1, 2, 8, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 2, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(ra.RAError):  # dq on top of q
        ra.attn_bwd_causal_rope(q, q, q, q, lse, q, apply_rope=False, dq=q)
    qd = torch.zeros((1, 2, 8, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ra.RAError) as e:  # tensor-core head sizes
        ra.attn_bwd_causal_rope(qd, qd, qd, qd, lse, qd, apply_rope=False)
    assert e.value.code == -2
