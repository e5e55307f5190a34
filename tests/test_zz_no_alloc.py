"""attn_decode_noalloc: decode attention for callers that cannot hand out
scratch memory (a device memory budget fixed at start-up, a framework that
owns every allocation): the split workspace lives in the library's static
device region, and the call allocates nothing.  The file name puts it last
in collection, so it runs both alone and after every other GPU test of a
session; it depends on no state those tests leave.

Each case makes two calls in a row with different inputs, the first one
larger (longer contexts, more key chunks), so that partial results the first
call leaves in the shared region would show up in the second.  Each result is
compared bit for bit with attn_decode on a caller workspace filled with NaN
(same plan, same kernels), and the second against the fp64 oracle.  Free
device memory (cudaMemGetInfo) must not change across the two calls."""
import numpy as np
import pytest
import torch

import workloads as wl

UNSUPPORTED = -2


@pytest.fixture(scope="module")
def ra():
    import __graft_entry__
    __graft_entry__.build()
    import rope_causal_attention_gb300 as m
    return m


def make_cache(ra, dt, B, Hkv, D, cap, seed):
    rows = B * cap
    g = torch.Generator("cpu").manual_seed(seed)
    k = wl.randn((rows, Hkv, D), g, dt).cuda()
    v = wl.randn((rows, Hkv, D), g, dt).cuda()
    starts = torch.arange(B, dtype=torch.int64) * cap
    return ra.KVCache(k, v, starts.cuda()), g


def reference(ra, cache, q, kv_len, max_len, ids):
    """attn_decode on a caller workspace whose every byte is 0xff (NaN)."""
    dt = q.dtype
    B, Hq, Sq, D = q.shape
    need = ra.attn_decode_workspace_size(dt, B, Hq, cache.Hkv, Sq, D, max_len)
    ws = torch.full((need,), 255, dtype=torch.uint8, device="cuda")
    o, lse = ra.attn_decode(cache, q, kv_len, max_len, seq_ids=ids, workspace=ws)
    assert ra.ra_get_device_status() == 0
    return o, lse


CASES = [
    # dt, B, Hq, Hkv, Sq, D, first lens, second lens (shorter: fewer key chunks)
    (torch.bfloat16, 3, 16, 2, 1, 128, [9000, 40, 5000], [1999, 700, 3]),  # tensor-core split
    (torch.float16, 2, 16, 1, 4, 128, [6000, 7], [300, 2500]),            # tensor-core, 64 cols
    (torch.bfloat16, 2, 8, 8, 2, 64, [3000, 900], [3, 1200]),             # CUDA-core split kernel
    (torch.float32, 1, 4, 2, 1, 128, [9000], [2100]),                     # CUDA-core, fp32
]


@pytest.mark.gpu
@pytest.mark.parametrize("dt,B,Hq,Hkv,Sq,D,lens1,lens2", CASES)
def test_noalloc_two_calls_match_attn_decode(ra, dt, B, Hq, Hkv, Sq, D, lens1, lens2):
    import oracle
    cap = max(lens1 + lens2) + 16
    cache, g = make_cache(ra, dt, B, Hkv, D, cap, seed=B * D + Sq)
    ids = torch.from_numpy(np.arange(B)[::-1].astype(np.int32).copy()).cuda()
    calls = []
    for lens in (lens1, lens2):
        q = wl.randn((B, Hq, Sq, D), g, dt).cuda()
        kv_len = torch.tensor(lens, dtype=torch.int32).cuda()
        max_len = max(lens) + 3
        assert ra.attn_decode_workspace_size(dt, B, Hq, Hkv, Sq, D, max_len) > 0
        calls.append((q, kv_len, max_len, reference(ra, cache, q, kv_len, max_len, ids)))
    # two calls in a row on the static region; the first call on the device
    # looks the region up, so the memory check starts after it
    outs = []
    free_before = None
    for n, (q, kv_len, max_len, _) in enumerate(calls):
        out = torch.full_like(calls[n][3][0], float("nan"))
        lse = torch.full_like(calls[n][3][1], float("nan"))
        if n == 1:
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
        ra.attn_decode_noalloc(cache, q, kv_len, max_len, out, lse=lse, seq_ids=ids)
        assert ra.ra_get_device_status() == 0
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    for (out, lse), (_, _, _, (want_o, want_lse)) in zip(outs, calls):
        assert torch.equal(out, want_o)
        assert torch.equal(lse, want_lse)
    # the second call against the fp64 oracle (O <= 2e-2 / 1e-4, LSE <= 1e-3)
    q, kv_len, _, _ = calls[1]
    kc, vc = cache.k.float().cpu().numpy(), cache.v.float().cpu().numpy()
    o_ref, lse_ref = oracle.decode_attention(q.float().cpu().numpy(), kc, vc,
                                             cache.seq_start.cpu().numpy(), lens2,
                                             seq_ids=ids.cpu().numpy())
    tol_o = 1e-4 if dt == torch.float32 else 2e-2
    assert np.abs(outs[1][0].float().cpu().numpy() - o_ref).max() <= tol_o
    assert np.abs(outs[1][1].cpu().numpy() - lse_ref).max() <= 1e-3


@pytest.mark.gpu
def test_noalloc_rejects_sizes_past_the_static_region(ra):
    """The decode workload needs ~1.2 GB of split workspace: refused before
    any launch, outputs untouched."""
    W = wl.DECODE_ATTN
    dt = torch.bfloat16
    need = ra.attn_decode_workspace_size(dt, W.B, W.Hq, W.Hkv, 1, W.D, W.table_rows)
    assert need > 32 * 2 ** 20  # RA_DECODE_STATIC_SCRATCH_BYTES
    cache, g = make_cache(ra, dt, W.B, W.Hkv, W.D, 2 + 16, seed=1)
    q = wl.randn((W.B, W.Hq, 1, W.D), g, dt).cuda()
    kv_len = torch.full((W.B,), 2, dtype=torch.int32).cuda()
    out = torch.zeros((W.B, W.Hq, 1, W.D), dtype=dt, device="cuda")
    with pytest.raises(ra.RAError) as e:
        ra.attn_decode_noalloc(cache, q, kv_len, W.table_rows, out)
    assert e.value.code == UNSUPPORTED
    assert bool((out == 0).all())
    assert ra.ra_get_device_status() == 0
