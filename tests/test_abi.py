"""C-ABI checks that need no GPU: the library loads, exports every function
that include/rope_attn.h declares, and rejects bad arguments on the host with
the documented codes before any CUDA call.

The rejection cases use placeholder addresses that the library never
dereferences (every case fails validation).  On a machine with a visible GPU
those cases are skipped and the GPU suite covers the error paths with real
buffers instead, so that a validation regression can never launch a kernel
on a placeholder address.
"""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rope_attn.h")

OK, INVALID, UNSUPPORTED, ALIGN, OVERLAP, CUDA, TIMEOUT, POSRANGE = 0, -1, -2, -3, -4, -5, -6, -7


@pytest.fixture(scope="module")
def L():
    from rope_causal_attention_gb300 import build as b
    b.build()
    import rope_causal_attention_gb300 as ra
    return ra.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["rope_tables_build", "rope_tables_build_scaled", "rope_apply_qk", "rope_append_kv",
              "attn_bwd_causal_rope", "attn_bwd_workspace_size",
              "attn_decode", "attn_decode_workspace_size", "attn_fwd_causal_rope",
              "ra_get_device_status", "ra_status_string", "ra_last_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in rope_attn.h but not exported"


def test_status_strings(L):
    for code in [OK, INVALID, UNSUPPORTED, ALIGN, OVERLAP, CUDA, TIMEOUT, POSRANGE]:
        s = L.ra_status_string(code).decode()
        assert s.startswith("RA_")
    assert L.ra_status_string(12345).decode() == "unknown ra_status"


no_gpu = pytest.mark.skipif(torch.cuda.is_available(),
                            reason="placeholder-address cases run only where no GPU is visible")

A = 0x10000000  # placeholder, 256-byte aligned, never dereferenced


def p(off):
    return ctypes.c_void_p(A + off)


def i64(*v):
    return (ctypes.c_int64 * len(v))(*v)


def rope(L, q=p(0), k=p(1 << 24), qo=None, ko=None, dt=1, T=4, Hq=2, Hkv=1, D=8, rot=8, lay=0,
         sq=(16, 8), sk=(8, 8), sqo=None, sko=None, pos=p(1 << 26), is64=0, rows=16):
    return L.rope_apply_qk(q, k, qo, ko, dt, T, Hq, Hkv, D, rot, lay,
                           i64(*sq) if sq else None, i64(*sk) if sk else None,
                           i64(*sqo) if sqo else None, i64(*sko) if sko else None, pos, is64,
                           p(1 << 27), p(1 << 28), rows, None)


@no_gpu
def test_tables_rejections(L):
    c, s = p(0), p(4096)
    assert L.rope_tables_build(c, s, -1, 8, 10000.0, 0, None) == INVALID
    assert L.rope_tables_build(c, s, 4, 7, 10000.0, 0, None) == INVALID
    assert L.rope_tables_build(c, s, 4, 0, 10000.0, 0, None) == INVALID
    assert L.rope_tables_build(c, s, 4, 8, 0.0, 0, None) == INVALID
    assert L.rope_tables_build(c, s, 4, 8, -2.0, 0, None) == INVALID
    assert L.rope_tables_build(c, s, 4, 8, float("nan"), 0, None) == INVALID
    assert L.rope_tables_build(None, s, 4, 8, 10000.0, 0, None) == INVALID
    assert L.rope_tables_build(p(2), s, 4, 8, 10000.0, 0, None) == ALIGN
    assert L.rope_tables_build(c, s, 0, 8, 10000.0, 0, None) == OK  # nothing to do
    for bad in (0.0, -4.0, float("nan"), float("inf")):
        assert L.rope_tables_build_scaled(c, s, 4, 8, 10000.0, 0, bad, None) == INVALID
    assert L.rope_tables_build_scaled(c, s, 4, 7, 10000.0, 0, 4.0, None) == INVALID
    assert L.rope_tables_build_scaled(c, s, 0, 8, 10000.0, 0, 4.0, None) == OK


@no_gpu
def test_rope_rejections(L):
    assert rope(L, D=7, rot=6) == INVALID                 # odd D
    assert rope(L, rot=10) == INVALID                     # rot_dim > D
    assert rope(L, rot=3) == INVALID                      # odd rot_dim
    assert rope(L, dt=9) == INVALID                       # dtype
    assert rope(L, lay=2) == INVALID                      # layout
    assert rope(L, q=None) == INVALID                     # Hq > 0 without q
    assert rope(L, pos=None) == INVALID
    assert rope(L, rows=0) == INVALID
    assert rope(L, sq=(-16, 8)) == INVALID
    assert rope(L, sq=None) == INVALID
    assert rope(L, T=0) == OK                             # empty batch: no launch
    # k written in place overlapping q's bytes
    assert rope(L, k=p(16)) == OVERLAP
    # q_out partially overlapping q
    assert rope(L, qo=p(2), sqo=(16, 8)) == OVERLAP
    # k_out landing on q
    assert rope(L, ko=p(0), sko=(8, 8)) == OVERLAP
    # misaligned positions (int64 needs 8 bytes)
    assert rope(L, pos=p((1 << 26) + 4), is64=1) == ALIGN
    # misaligned element pointer
    assert rope(L, q=p(1)) == ALIGN


def attn(L, dt=1, B=1, Hq=4, Hkv=2, Sq=8, Sk=8, D=64, off=0, rope_on=1, rot=64, lay=0, rows=8,
         q=p(0), k=p(1 << 22), v=p(1 << 23), o=p(1 << 24), lse=None, strides=None):
    sq = strides or (Hq * Sq * D, Sq * D, D)
    sk = strides or (Hkv * Sk * D, Sk * D, D)
    return L.attn_fwd_causal_rope(q, k, v, o, lse, dt, B, Hq, Hkv, Sq, Sk, D, off, rope_on, rot,
                                  lay, p(1 << 25), p(1 << 26), rows, ctypes.c_float(0.0),
                                  i64(*sq), i64(*sk), i64(*sk), i64(*sq), None)


@no_gpu
def test_attention_rejections(L):
    assert attn(L, off=-1) == INVALID         # rows without keys
    assert attn(L, Hq=3, Hkv=2) == INVALID    # Hq % Hkv
    assert attn(L, Sk=0) == INVALID
    assert attn(L, D=63, rot=62) == INVALID
    assert attn(L, rot=66) == INVALID
    assert attn(L, rows=7) == INVALID         # table shorter than positions used
    assert attn(L, Sk=10, rows=9) == INVALID
    assert attn(L, Sq=4, off=6, rows=9) == INVALID
    assert attn(L, dt=7) == INVALID
    assert attn(L, q=None) == INVALID
    assert attn(L, Sq=0) == OK                # no rows: no launch
    assert attn(L, D=96, rot=96) == UNSUPPORTED           # tensor-core head dims
    assert attn(L, dt=0, D=300, rot=300) == UNSUPPORTED    # fp32 path limit
    assert attn(L, rot=60) == UNSUPPORTED                 # NeoX rot_dim/2 % 8
    assert attn(L, o=p(8)) == OVERLAP                     # output on top of q
    assert attn(L, q=p(2)) == ALIGN
    assert attn(L, strides=(4 * 8 * 64, 8 * 64, 60)) == ALIGN  # row stride not multiple of 8


def kvc(k=A + (1 << 27), v=A + (1 << 28), ks=(16, 8), vs=(16, 8), rows=64, st=A + (1 << 29),
        n=4):
    from rope_causal_attention_gb300 import KVCacheDesc
    c = KVCacheDesc()
    c.k, c.v = k, v
    c.k_strides[0], c.k_strides[1] = ks
    c.v_strides[0], c.v_strides[1] = vs
    c.rows, c.seq_start, c.n_seqs = rows, st, n
    return c


def append(L, cache=None, q=p(0), qo=None, kn=p(1 << 22), vn=p(1 << 23), dt=1, T=4, Hq=2,
           Hkv=2, D=8, rot=8, lay=0, sq=(16, 8), sqo=None, skn=(16, 8), svn=(16, 8), ids=None,
           pos=p(1 << 24), is64=0, rows=16):
    c = kvc() if cache is None else cache
    return L.rope_append_kv(q, qo, kn, vn, ctypes.byref(c) if c is not False else None, dt, T,
                            Hq, Hkv, D, rot, lay, i64(*sq) if sq else None,
                            i64(*sqo) if sqo else None, i64(*skn) if skn else None,
                            i64(*svn) if svn else None, ids, pos, is64, p(1 << 25), p(1 << 26),
                            rows, None)


def test_decode_workspace_size(L):
    L.attn_decode_workspace_size.restype = ctypes.c_size_t
    bad = ctypes.c_size_t(-1).value
    assert L.attn_decode_workspace_size(1, 1, 8, 8, 1, 128, 100) == 0       # one chunk
    assert L.attn_decode_workspace_size(1, 1, 8, 3, 1, 128, 100) == bad     # Hq % Hkv
    assert L.attn_decode_workspace_size(1, 1, 8, 8, 0, 128, 100) == bad     # Sq
    assert L.attn_decode_workspace_size(1, 1, 8, 8, 1, 258, 100) == bad     # D > 256
    assert L.attn_decode_workspace_size(9, 1, 8, 8, 1, 128, 100) == bad     # dtype
    # long keys split into chunks: O partials (fp32 D per chunk) + one LSE per chunk
    n = L.attn_decode_workspace_size(1, 4, 64, 8, 1, 128, 131072)
    assert n != bad and n > 4 * 64 * 2 * 128 * 4


@no_gpu
def test_append_rejections(L):
    assert append(L, cache=False) == INVALID
    assert append(L, cache=kvc(k=0)) == INVALID
    assert append(L, cache=kvc(rows=0)) == INVALID
    assert append(L, cache=kvc(n=0)) == INVALID
    assert append(L, cache=kvc(ks=(4, 8))) == INVALID     # rows of the K cache overlap
    assert append(L, Hkv=0) == INVALID
    assert append(L, D=7, rot=6) == INVALID
    assert append(L, rot=10) == INVALID
    assert append(L, q=None) == INVALID                    # Hq > 0 without q
    assert append(L, kn=None) == INVALID
    assert append(L, pos=None) == INVALID
    assert append(L, rows=0) == INVALID
    assert append(L, skn=None) == INVALID
    assert append(L, sq=(-16, 8)) == INVALID
    assert append(L, T=0) == OK                            # nothing to do
    # cache V on top of cache K
    assert append(L, cache=kvc(v=A + (1 << 27) + 8)) == OVERLAP
    # cache K on top of k_new
    assert append(L, cache=kvc(k=A + (1 << 22))) == OVERLAP
    # q_out partially overlapping q
    assert append(L, qo=p(2), sqo=(16, 8)) == OVERLAP
    assert append(L, q=p(1)) == ALIGN
    assert append(L, pos=p((1 << 24) + 4), is64=1) == ALIGN


def decode(L, cache=None, q=p(0), o=p(1 << 22), lse=None, dt=1, B=2, Hq=4, Hkv=2, Sq=1, D=8,
           ids=None, kvl=p(1 << 24), maxl=32, sq=(32, 8, 32), so=(32, 8, 32), ws=None, wsb=0):
    c = kvc() if cache is None else cache
    return L.attn_decode(q, o, lse, ctypes.byref(c) if c is not False else None, dt, B, Hq, Hkv,
                         Sq, D, ids, kvl, maxl, ctypes.c_float(0.0), i64(*sq) if sq else None,
                         i64(*so) if so else None, ws, ctypes.c_size_t(wsb), None)


@no_gpu
def test_decode_rejections(L):
    assert decode(L, Hq=3) == INVALID                      # Hq % Hkv
    assert decode(L, Sq=0) == INVALID
    assert decode(L, D=7) == INVALID
    assert decode(L, D=258) == INVALID
    assert decode(L, maxl=0) == INVALID
    assert decode(L, Sq=4, maxl=3) == INVALID              # max_kv_len < Sq
    assert decode(L, q=None) == INVALID
    assert decode(L, kvl=None) == INVALID
    assert decode(L, cache=False) == INVALID
    assert decode(L, sq=None) == INVALID
    assert decode(L, dt=5) == INVALID
    assert decode(L, B=0) == OK                            # nothing to do
    # a long cache needs a workspace
    assert decode(L, maxl=100000) == INVALID
    assert decode(L, maxl=100000, ws=p(1 << 30), wsb=16) == INVALID   # too small
    need = L.attn_decode_workspace_size(1, 2, 4, 2, 1, 8, 100000)
    assert decode(L, maxl=100000, ws=ctypes.c_void_p(A + (1 << 30) + 8), wsb=need) == ALIGN
    assert decode(L, o=p(8)) == OVERLAP                    # output on top of q
    assert decode(L, o=ctypes.c_void_p(A + (1 << 27))) == OVERLAP      # output on the cache
    assert decode(L, q=p(1)) == ALIGN


@no_gpu
def test_decode_noalloc_rejections(L):
    """Sizes whose split workspace exceeds the static region are refused
    before any CUDA call; invalid sizes as in attn_decode."""
    c = kvc()
    call = lambda B, Hq, Hkv, maxl: L.attn_decode_noalloc(
        p(0), p(1 << 22), None, ctypes.byref(c), 1, B, Hq, Hkv, 1, 8, None, p(1 << 24), maxl,
        ctypes.c_float(0.0), i64(32, 8, 32), i64(32, 8, 32), None)
    assert call(512, 64, 8, 131072) == UNSUPPORTED
    assert call(2, 3, 2, 32) == INVALID      # Hq % Hkv
    assert call(2, 4, 2, 0) == INVALID       # max_kv_len


def test_backward_workspace_size(L):
    """D_i row terms always; fp16 rotated Q and K copies for 16-bit inputs."""
    L.attn_bwd_workspace_size.restype = ctypes.c_size_t
    up = lambda x: (x + 255) // 256 * 256
    B, Hq, Hkv, Sq, Sk, D = 2, 8, 2, 100, 300, 128
    assert L.attn_bwd_workspace_size(0, B, Hq, Hkv, ctypes.c_int64(Sq), ctypes.c_int64(Sk), D) == \
        up(B * Hq * Sq * 4)
    assert L.attn_bwd_workspace_size(1, B, Hq, Hkv, ctypes.c_int64(Sq), ctypes.c_int64(Sk), D) == \
        up(B * Hq * Sq * 4) + up(B * Hq * Sq * D * 2) + up(B * Hkv * Sk * D * 2)
    assert L.attn_bwd_workspace_size(7, B, Hq, Hkv, ctypes.c_int64(Sq), ctypes.c_int64(Sk), D) == \
        ctypes.c_size_t(-1).value
