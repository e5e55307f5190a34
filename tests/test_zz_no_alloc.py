"""attn_decode_noalloc: the decode kernels with their split workspace in the
library's static device region (no allocation by the call).  The file name
puts it last in collection, so it runs both alone and after every other GPU
test of a session; it depends on no state those tests leave.

Each case runs the variant twice in a row and compares both results bit for
bit with attn_decode on a caller-allocated workspace (same plan, same
kernels), and checks that device memory in use did not change."""
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


def inputs(ra, dt, B, Hq, Hkv, Sq, D, lens, seed):
    cap = max(lens) + 16
    rows = B * cap
    g = torch.Generator("cpu").manual_seed(seed)
    k = wl.randn((rows, Hkv, D), g, dt).cuda()
    v = wl.randn((rows, Hkv, D), g, dt).cuda()
    starts = torch.arange(B, dtype=torch.int64) * cap
    cache = ra.KVCache(k, v, starts.cuda())
    q = wl.randn((B, Hq, Sq, D), g, dt).cuda()
    ids = torch.from_numpy(np.arange(B)[::-1].astype(np.int32).copy()).cuda()
    return cache, q, torch.tensor(lens, dtype=torch.int32).cuda(), ids


CASES = [
    # dt, B, Hq, Hkv, Sq, D, lens   (every case splits its keys: the static region is used)
    (torch.bfloat16, 3, 16, 2, 1, 128, [5000, 40, 1999]),   # tensor-core split kernel
    (torch.float16, 2, 16, 1, 4, 128, [3000, 7]),            # tensor-core, 64 query columns
    (torch.bfloat16, 2, 8, 8, 2, 64, [900, 3]),              # CUDA-core split kernel
    (torch.float32, 1, 4, 2, 1, 128, [6000]),                # CUDA-core, fp32
]


@pytest.mark.gpu
@pytest.mark.parametrize("dt,B,Hq,Hkv,Sq,D,lens", CASES)
def test_noalloc_equals_attn_decode_on_two_calls(ra, dt, B, Hq, Hkv, Sq, D, lens):
    cache, q, kv_len, ids = inputs(ra, dt, B, Hq, Hkv, Sq, D, lens, seed=B * D + Sq)
    max_len = max(lens) + 3
    assert ra.attn_decode_workspace_size(dt, B, Hq, Hkv, Sq, D, max_len) > 0
    want_o, want_lse = ra.attn_decode(cache, q, kv_len, max_len, seq_ids=ids)
    assert ra.ra_get_device_status() == 0
    out = torch.empty_like(want_o)
    lse = torch.empty_like(want_lse)
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    for _ in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        ra.attn_decode_noalloc(cache, q, kv_len, max_len, out, lse=lse, seq_ids=ids)
        assert ra.ra_get_device_status() == 0
        assert torch.equal(out, want_o)
        assert torch.equal(lse, want_lse)
    assert torch.cuda.memory_allocated() == before


@pytest.mark.gpu
def test_noalloc_rejects_sizes_past_the_static_region(ra):
    """The decode workload needs ~1.2 GB of split workspace: refused before
    any launch, outputs untouched."""
    W = wl.DECODE_ATTN
    dt = torch.bfloat16
    need = ra.attn_decode_workspace_size(dt, W.B, W.Hq, W.Hkv, 1, W.D, W.table_rows)
    assert need > 32 * 2 ** 20  # RA_DECODE_STATIC_SCRATCH_BYTES
    cache, q, kv_len, ids = inputs(ra, dt, W.B, W.Hq, W.Hkv, 1, W.D, [2] * W.B, seed=1)
    out = torch.zeros((W.B, W.Hq, 1, W.D), dtype=dt, device="cuda")
    with pytest.raises(ra.RAError) as e:
        ra.attn_decode_noalloc(cache, q, kv_len, W.table_rows, out)
    assert e.value.code == UNSUPPORTED
    assert bool((out == 0).all())
    assert ra.ra_get_device_status() == 0
