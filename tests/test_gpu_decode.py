"""GPU parity of the decoder step against the fp64 oracle: rope_append_kv
(rotated Q, rotated K and raw V written to the cache at each token's cache
position) and attn_decode (split-KV attention of the new queries over the
cache), separately and composed.

Tolerances: rotations as in the rope_apply tests (rope_check); V rows and
untouched cache rows bit-exact; attention O within 2e-2 (bf16/fp16) or 1e-4
(fp32) absolute and LSE within 1e-3 of the fp64 oracle, the bounds stated
for the fused attention."""
import numpy as np
import pytest
import torch

import workloads as wl
from rope_check import check_rotated

pytestmark = pytest.mark.gpu

NEOX, GPTJ = 0, 1
POSRANGE = -7
O_TOL = {torch.bfloat16: 2e-2, torch.float16: 2e-2, torch.float32: 1e-4}
LSE_TOL = 1e-3


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


def make_cache(ra, Hkv, D, dt, n_seqs, cap, layout, seed, fill=None):
    """A cache of n_seqs regions of `cap` rows separated by 3-row gaps.
    layout: 'token' [rows][Hkv][D], 'head' [Hkv][rows][D] storage seen as
    [rows][Hkv][D], 'inter' K and V interleaved per row [rows][2][Hkv][D].
    Rows hold seeded N(0,1) values, or `fill` everywhere."""
    rows = n_seqs * (cap + 3) + 5
    g = torch.Generator("cpu").manual_seed(seed)
    shape = {"token": (2, rows, Hkv, D), "head": (2, Hkv, rows, D), "inter": (rows, 2, Hkv, D)}
    buf = wl.randn(shape[layout], g, dt)
    if fill is not None:
        buf.fill_(fill)
    buf = buf.cuda()
    if layout == "token":
        k, v = buf[0], buf[1]
    elif layout == "head":
        k, v = buf[0].permute(1, 0, 2), buf[1].permute(1, 0, 2)
    else:
        k, v = buf[:, 0], buf[:, 1]
    starts = torch.tensor([5 + s * (cap + 3) for s in range(n_seqs)], dtype=torch.int64)
    return ra.KVCache(k, v, starts.cuda()), starts


def token_slots(T, n_seqs, cap, seed, identity):
    """(seq id, position) per token; no two tokens share a cache row."""
    rng = np.random.default_rng(seed)
    if identity:
        seq = np.arange(T)
    else:
        seq = rng.integers(0, n_seqs, size=T)
    pos = np.empty(T, dtype=np.int64)
    for s in np.unique(seq):
        idx = np.nonzero(seq == s)[0]
        pos[idx] = rng.choice(cap, size=idx.shape[0], replace=False)
    return seq.astype(np.int32), pos


APPEND_CASES = [
    # dt, Hq, Hkv, D, rot_dim, layout, cache layout
    (torch.bfloat16, 8, 2, 128, 128, NEOX, "token"),
    (torch.bfloat16, 8, 2, 128, 64, GPTJ, "head"),
    (torch.float16, 4, 4, 64, 32, NEOX, "inter"),
    (torch.float32, 6, 2, 64, 64, GPTJ, "token"),
    (torch.float32, 3, 1, 96, 16, NEOX, "inter"),
    (torch.bfloat16, 3, 1, 10, 6, NEOX, "token"),   # scalar kernel (no 16-byte slices)
    (torch.float16, 2, 2, 24, 12, GPTJ, "head"),    # scalar kernel
]


@pytest.mark.parametrize("q_mode", ["inplace", "out", "none"])
@pytest.mark.parametrize("ids", [False, True])
@pytest.mark.parametrize("dt,Hq,Hkv,D,rot_dim,layout,cl", APPEND_CASES)
def test_append_matches_oracle(ra, orc, dt, Hq, Hkv, D, rot_dim, layout, cl, q_mode, ids):
    n_seqs, cap, base = 5, 48, 10000.0
    T = 13 if ids else n_seqs
    cache, starts = make_cache(ra, Hkv, D, dt, n_seqs, cap, cl, seed=D + Hq)
    k0, v0 = cache.k.cpu(), cache.v.cpu()
    q, k, v = wl.decode_tokens(T, Hq, Hkv, D, dt, seed=17 + D)
    seq, pos = token_slots(T, n_seqs, cap, seed=rot_dim + T, identity=not ids)
    cos, sin = ra.make_tables(cap, rot_dim, base)
    qg = q.cuda() if q_mode != "none" else None
    qo = torch.full_like(qg, 3.0) if q_mode == "out" else None
    res = ra.rope_append_kv(cache, qg, k.cuda(), v.cuda(), torch.from_numpy(pos).cuda(), cos, sin,
                            seq_ids=torch.from_numpy(seq).cuda() if ids else None,
                            layout=layout, q_out=qo)
    assert ra.ra_get_device_status() == 0
    if q_mode != "none":
        check_rotated(res, q, pos, orc, rot_dim, base, layout)
        if q_mode == "out":
            assert torch.equal(qg.cpu(), q)
    rows = starts.numpy()[seq] + pos
    k1, v1 = cache.k.cpu(), cache.v.cpu()
    check_rotated(k1[rows], k, pos, orc, rot_dim, base, layout)
    assert torch.equal(v1[rows], v)
    keep = np.ones(k1.shape[0], dtype=bool)
    keep[rows] = False
    assert torch.equal(k1[keep], k0[keep]) and torch.equal(v1[keep], v0[keep])


def test_append_out_of_range_tokens_are_skipped(ra, orc):
    dt, Hq, Hkv, D = torch.bfloat16, 2, 2, 64
    cache, starts = make_cache(ra, Hkv, D, dt, 3, 16, "token", seed=5)
    k0 = cache.k.cpu()
    q, k, v = wl.decode_tokens(4, Hq, Hkv, D, dt, seed=6)
    seq = torch.tensor([0, 7, 1, 2], dtype=torch.int32)      # token 1: no such sequence
    pos = torch.tensor([3, 1, 16, 4], dtype=torch.int64)     # token 2: past the table
    cos, sin = ra.make_tables(16, D, 10000.0)
    qg = q.cuda()
    ra.rope_append_kv(cache, qg, k.cuda(), v.cuda(), pos.cuda(), cos, sin, seq_ids=seq.cuda())
    assert ra.ra_get_device_status() == POSRANGE
    assert ra.ra_get_device_status() == 0
    got = qg.cpu()
    assert torch.equal(got[1], q[1]) and torch.equal(got[2], q[2])   # skipped tokens untouched
    k1 = cache.k.cpu()
    for t in (0, 3):
        check_rotated(k1[int(starts[seq[t]]) + int(pos[t])][None], k[t][None],
                      pos[t:t + 1].numpy(), orc, D, 10000.0, NEOX)
    keep = np.ones(k1.shape[0], dtype=bool)
    keep[[int(starts[0]) + 3, int(starts[2]) + 4]] = False
    assert torch.equal(k1[keep], k0[keep])


def decode_inputs(ra, dt, B, Hq, Hkv, Sq, D, lens, cl, seed, nan_outside=True):
    """Cache holding seeded keys/values for each entry's sequence (entries map
    to sequences in reverse order) and NaN everywhere else; q [B,Hq,Sq,D]."""
    cap = max(lens) + 40
    cache, starts = make_cache(ra, Hkv, D, dt, B, cap, cl, seed,
                               fill=float("nan") if nan_outside else None)
    g = torch.Generator("cpu").manual_seed(seed + 1)
    ids = np.arange(B)[::-1].astype(np.int32).copy()
    for b, L in enumerate(lens):
        r0 = int(starts[ids[b]])
        cache.k[r0:r0 + L] = wl.randn((L, Hkv, D), g, dt).cuda()
        cache.v[r0:r0 + L] = wl.randn((L, Hkv, D), g, dt).cuda()
    q = wl.randn((B, Hq, Sq, D), g, dt)
    return cache, starts, ids, q


def check_decode(o, lse, want_o, want_lse, dt):
    err_o = np.abs(o.float().cpu().numpy().astype(np.float64) - want_o).max()
    err_l = np.abs(lse.cpu().numpy().astype(np.float64) - want_lse).max()
    assert err_o <= O_TOL[dt], err_o
    assert err_l <= LSE_TOL, err_l


DECODE_CASES = [
    # dt, B, Hq, Hkv, Sq, D, lens
    (torch.bfloat16, 3, 8, 1, 1, 128, [1, 130, 700]),
    (torch.bfloat16, 2, 32, 8, 1, 128, [5000, 333]),
    (torch.float16, 2, 16, 2, 4, 128, [4, 2000]),
    (torch.bfloat16, 1, 8, 8, 1, 128, [12000]),
    (torch.bfloat16, 2, 4, 4, 1, 64, [100, 1000]),
    (torch.float32, 2, 4, 2, 2, 64, [3, 900]),
    (torch.bfloat16, 1, 16, 1, 4, 128, [3000]),     # 64 query columns
    (torch.float16, 2, 20, 2, 4, 128, [700, 41]),   # 40 columns, padded to 64
    (torch.bfloat16, 2, 24, 2, 2, 128, [1500, 129]),  # 24 columns, padded to 32
    (torch.bfloat16, 1, 64, 1, 2, 128, [300]),      # 128 query rows per kv head
    (torch.float32, 1, 2, 1, 1, 256, [50]),
    (torch.float16, 2, 6, 3, 3, 40, [7, 64]),
]


@pytest.mark.parametrize("cl", ["token", "head", "inter"])
@pytest.mark.parametrize("dt,B,Hq,Hkv,Sq,D,lens", DECODE_CASES)
def test_decode_matches_oracle(ra, orc, dt, B, Hq, Hkv, Sq, D, lens, cl):
    cache, starts, ids, q = decode_inputs(ra, dt, B, Hq, Hkv, Sq, D, lens, cl, seed=B * D + Sq)
    kv_len = torch.tensor(lens, dtype=torch.int32)
    o, lse = ra.attn_decode(cache, q.cuda(), kv_len.cuda(), max(lens) + 7,
                            seq_ids=torch.from_numpy(ids).cuda())
    assert ra.ra_get_device_status() == 0
    want_o, want_lse = orc.decode_attention(q.float().numpy(), cache.k.float().cpu().numpy(),
                                            cache.v.float().cpu().numpy(), starts.numpy(),
                                            lens, seq_ids=ids)
    check_decode(o, lse, want_o, want_lse, dt)


def test_decode_token_major_queries_and_custom_scale(ra, orc):
    """Decode tokens laid out [B*Sq][Hq][D] (as rope_append_kv leaves them)
    viewed as [B,Hq,Sq,D] through strides; output written into a strided view."""
    dt, B, Hq, Hkv, Sq, D, lens = torch.bfloat16, 3, 8, 2, 2, 128, [40, 900, 2]
    cache, starts, ids, q = decode_inputs(ra, dt, B, Hq, Hkv, Sq, D, lens, "token", seed=9)
    qt = q.permute(0, 2, 1, 3).contiguous().cuda()              # [B, Sq, Hq, D]
    out = torch.zeros((B, Sq, Hq, D), dtype=dt, device="cuda")
    o, lse = ra.attn_decode(cache, qt.permute(0, 2, 1, 3), torch.tensor(lens, dtype=torch.int32).cuda(),
                            max(lens), seq_ids=torch.from_numpy(ids).cuda(), softmax_scale=0.05,
                            out=out.permute(0, 2, 1, 3))
    assert ra.ra_get_device_status() == 0
    want_o, want_lse = orc.decode_attention(q.float().numpy(), cache.k.float().cpu().numpy(),
                                            cache.v.float().cpu().numpy(), starts.numpy(), lens,
                                            seq_ids=ids, scale=0.05)
    check_decode(out.permute(0, 2, 1, 3), lse, want_o, want_lse, dt)


def test_decode_bad_entries_are_flagged_and_skipped(ra, orc):
    dt, B, Hq, Hkv, Sq, D = torch.bfloat16, 3, 4, 1, 2, 128
    lens = [10, 20, 30]
    cache, starts, ids, q = decode_inputs(ra, dt, B, Hq, Hkv, Sq, D, lens, "token", seed=4,
                                          nan_outside=False)
    kv_len = torch.tensor([10, 1, 30], dtype=torch.int32)      # entry 1: fewer keys than queries
    out = torch.full((B, Hq, Sq, D), 5.0, dtype=dt, device="cuda")
    ra.attn_decode(cache, q.cuda(), kv_len.cuda(), 30, seq_ids=torch.from_numpy(ids).cuda(), out=out)
    assert ra.ra_get_device_status() == POSRANGE
    assert ra.ra_get_device_status() == 0
    assert bool((out[1] == 5.0).all())
    want_o, _ = orc.decode_attention(q.float().numpy(), cache.k.float().cpu().numpy(),
                                     cache.v.float().cpu().numpy(), starts.numpy(), [10, 20, 30],
                                     seq_ids=ids)
    got = out.float().cpu().numpy()
    for b in (0, 2):
        assert np.abs(got[b] - want_o[b]).max() <= O_TOL[dt]


@pytest.mark.parametrize("dt,layout,rot_dim", [(torch.bfloat16, NEOX, 128), (torch.float16, GPTJ, 64),
                                               (torch.float32, NEOX, 32)])
def test_decode_step_end_to_end(ra, orc, dt, layout, rot_dim):
    """The decoder step end to end: the prefix and then the new tokens are
    appended (rotated K, raw V), the new queries rotated in place, and decode
    attention run over the cache.

    Reference: the oracle's fp64 rotation of the raw K and Q, rounded once to
    the cache dtype (the cache stores rotated K in its own dtype, section 2),
    then the oracle's decode attention; O and LSE within the attention
    bounds.  Also, O within the same bound of causal attention with RoPE
    applied inside to the raw tensors (the convention's equivalence; its LSE
    differs by the dtype rounding of the cached keys, up to ~2e-3 in bf16,
    so only O is compared there)."""
    B, Hq, Hkv, Sq, base = 2, 8, 2, 2, 500000.0
    D = 128 if dt != torch.float32 else 64
    lens = [37, 300]
    cap = max(lens) + 8
    cache, starts = make_cache(ra, Hkv, D, dt, B, cap, "token", seed=21, fill=float("nan"))
    cos, sin = ra.make_tables(cap, rot_dim, base)
    g = torch.Generator("cpu").manual_seed(22)
    raw = []
    for b, L in enumerate(lens):
        k = wl.randn((L, Hkv, D), g, dt)
        v = wl.randn((L, Hkv, D), g, dt)
        q = wl.randn((Sq, Hq, D), g, dt)
        raw.append((q, k, v))
        pre = L - Sq   # prefix first (no queries), then the step's new tokens
        ids = torch.full((pre,), b, dtype=torch.int32)
        ra.rope_append_kv(cache, None, k[:pre].cuda(), v[:pre].cuda(), torch.arange(pre).cuda(),
                          cos, sin, seq_ids=ids.cuda(), layout=layout)
    qn = torch.stack([r[0] for r in raw]).cuda()                      # [B, Sq, Hq, D]
    tok = lambda i: torch.cat([raw[b][i][lens[b] - Sq:] for b in range(B)]).cuda()
    pos = torch.cat([torch.arange(L - Sq, L) for L in lens]).cuda()
    ids = torch.arange(B, dtype=torch.int32).repeat_interleave(Sq).cuda()
    ra.rope_append_kv(cache, qn.view(B * Sq, Hq, D), tok(1), tok(2), pos, cos, sin, seq_ids=ids,
                      layout=layout)
    o, lse = ra.attn_decode(cache, qn.permute(0, 2, 1, 3),
                            torch.tensor(lens, dtype=torch.int32).cuda(), max(lens))
    assert ra.ra_get_device_status() == 0
    rnd = lambda x: torch.from_numpy(x).to(dt).float().numpy()
    for b, L in enumerate(lens):
        q, k, v = raw[b]
        k_rot = rnd(orc.rope_tokens(k.float().numpy(), np.arange(L), rot_dim=rot_dim, base=base,
                                    layout=layout))
        q_rot = rnd(orc.rope_tokens(q.float().numpy(), np.arange(L - Sq, L), rot_dim=rot_dim,
                                    base=base, layout=layout))
        want_o, want_lse = orc.decode_attention(q_rot.transpose(1, 0, 2)[None], k_rot,
                                                v.float().numpy(), [0], [L])
        check_decode(o[b:b + 1], lse[b:b + 1], want_o, want_lse, dt)
        fused_o, _ = orc.attention(q.float().numpy().transpose(1, 0, 2)[None],
                                   k.float().numpy().transpose(1, 0, 2)[None],
                                   v.float().numpy().transpose(1, 0, 2)[None],
                                   kv_offset=L - Sq, rot_dim=rot_dim, base=base, layout=layout)
        assert np.abs(o[b:b + 1].float().cpu().numpy() - fused_o).max() <= O_TOL[dt]


@pytest.mark.parametrize("dt,Hq,Hkv,Sq,D,want", [
    (torch.bfloat16, 16, 2, 1, 128, "attn_decode_tc_kernel"),
    (torch.float16, 16, 1, 4, 128, "attn_decode_tc_kernel"),
    (torch.bfloat16, 8, 2, 1, 64, "attn_decode_simt_kernel"),
    (torch.float32, 8, 2, 1, 128, "attn_decode_simt_kernel"),
])
def test_dispatch_runs_the_expected_kernel(ra, dt, Hq, Hkv, Sq, D, want):
    """bf16/fp16 with D = 128 run the tcgen05 split kernel (no silent
    CUDA-core fallback); other cases the CUDA-core kernel; long contexts add
    the merge."""
    lens = [3000, 100]
    cache, starts, ids, q = decode_inputs(ra, dt, 2, Hq, Hkv, Sq, D, lens, "token", seed=31)
    ra.attn_decode(cache, q.cuda(), torch.tensor(lens, dtype=torch.int32).cuda(), max(lens),
                   seq_ids=torch.from_numpy(ids).cuda())
    assert ra.ra_get_device_status() == 0
    assert ra.ra_last_launch() == [want, "attn_decode_merge_kernel"]
    _, kn, vn = wl.decode_tokens(1, 1, Hkv, D, dt, seed=3)
    ra.rope_append_kv(cache, None, kn.cuda(), vn.cuda(), torch.tensor([2], dtype=torch.int32).cuda(),
                      *ra.make_tables(8, D, 1e4))
    assert ra.ra_get_device_status() == 0
    assert ra.ra_last_launch() == ["rope_append_vec_kernel"]


def test_decode_workload_full_size_sampled(ra, orc):
    """The decode workload at full size (512 requests, contexts up to 131072
    keys, ~140 GB of bf16 K/V) in the launch configuration the benchmark
    times: append, then decode.  The longest, the shortest and two random
    requests are checked against the oracle, which rotates the new token's q
    and k itself (rounded to bf16, the cache's dtype) and reads the other
    cache rows from the seeded generator's output."""
    W = wl.DECODE_ATTN
    if torch.cuda.get_device_properties(0).total_memory < 180e9:
        pytest.skip("needs the GB300's memory")
    dev = torch.device("cuda")
    lens = W.kv_lens()
    B = lens.shape[0]
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    rows = int(lens.sum())
    g = torch.Generator(device=dev)
    g.manual_seed(W.seed)
    kc = torch.randn((rows, W.Hkv, W.D), generator=g, device=dev, dtype=torch.bfloat16)
    vc = torch.randn((rows, W.Hkv, W.D), generator=g, device=dev, dtype=torch.bfloat16)
    cache = ra.KVCache(kc, vc, torch.from_numpy(starts).to(dev))
    q, kn, vn = W.new_tokens()
    qg = q.cuda()
    pos = lens - 1
    cos, sin = ra.make_tables(W.table_rows, W.rot_dim, W.base)
    ra.rope_append_kv(cache, qg, kn.cuda(), vn.cuda(), torch.from_numpy(pos).to(torch.int32).cuda(),
                      cos, sin, layout=W.layout)
    o, lse = ra.attn_decode(cache, qg.view(B, 1, W.Hq, W.D).permute(0, 2, 1, 3),
                            torch.from_numpy(lens).to(torch.int32).cuda(), int(lens.max()))
    assert ra.ra_get_device_status() == 0
    rng = np.random.default_rng(0)
    picks = [int(np.argmax(lens)), int(np.argmin(lens)), *rng.choice(B, 2, replace=False).tolist()]
    rnd = lambda x: torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    for b in picks:
        L, r0 = int(lens[b]), int(starts[b])
        k_rows = kc[r0:r0 + L].float().cpu().numpy()
        v_rows = vc[r0:r0 + L].float().cpu().numpy()
        # the appended row: the GPU's must be the rotation of k_new; the oracle uses its own
        check_rotated(kc[r0 + L - 1:r0 + L].cpu(), kn[b:b + 1], pos[b:b + 1], orc, W.rot_dim,
                      W.base, W.layout)
        assert torch.equal(vc[r0 + L - 1].cpu(), vn[b])
        k_rows[L - 1] = rnd(orc.rope_tokens(kn[b:b + 1].float().numpy(), pos[b:b + 1],
                                            rot_dim=W.rot_dim, base=W.base, layout=W.layout))[0]
        v_rows[L - 1] = vn[b].float().numpy()
        q_rot = rnd(orc.rope_tokens(q[b:b + 1].float().numpy(), pos[b:b + 1], rot_dim=W.rot_dim,
                                    base=W.base, layout=W.layout))
        want_o, want_lse = orc.decode_attention(q_rot.transpose(1, 0, 2)[None], k_rows, v_rows,
                                                [0], [L])
        check_decode(o[b:b + 1], lse[b:b + 1], want_o, want_lse, torch.bfloat16)
    del kc, vc, cache
    torch.cuda.empty_cache()
