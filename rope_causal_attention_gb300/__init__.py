"""Python binding of librope_attn.so (RoPE and causal attention with RoPE
fused in, for GB300 / sm_103a).

The functions mirror the C ABI in ``include/rope_attn.h`` one for one and do
argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and the current
stream.  There is no CPU path: a missing library or a non-CUDA tensor raises.

Layouts: ``NEOX`` rotates pairs (i, i + rot_dim/2); ``GPTJ`` rotates pairs
(2i, 2i+1) ("Write Triton Rope Kernel", Inputs the agent should gather
first, item 1).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["NEOX", "GPTJ", "RAError", "rope_tables_build", "rope_tables_build_scaled",
           "make_tables", "rope_apply_qk", "KVCache", "rope_append_kv", "attn_decode",
           "attn_decode_workspace_size", "attn_decode_noalloc", "ra_last_launch",
           "attn_fwd_causal_rope", "attn_bwd_causal_rope", "ra_get_device_status", "ra_status_string", "library_path",
           "lib"]

NEOX = 0
GPTJ = 1
_DT = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "librope_attn.so")
_lock = threading.Lock()
_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)


class KVCacheDesc(ctypes.Structure):
    """ctypes mirror of ra_kv_cache."""
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("k_strides", ctypes.c_int64 * 2), ("v_strides", ctypes.c_int64 * 2),
                ("rows", ctypes.c_int64), ("seq_start", ctypes.c_void_p),
                ("n_seqs", ctypes.c_int64)]


class RAError(RuntimeError):
    """A non-OK ra_status from the library: `code` is the status value, the
    message carries ra_status_string and the library's reason (ra_last_error)."""

    def __init__(self, code: int, msg: str):
        super().__init__(msg)
        self.code = code


def library_path() -> str:
    """Path of the shared library the binding loads (built in-tree by build())."""
    return _LIB_PATH


def lib():
    """The loaded ctypes library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise ImportError(
                    f"{_LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` (there is no CPU fallback)")
            L = ctypes.CDLL(_LIB_PATH)
            vp, i64, i32, f64, f32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                      ctypes.c_double, ctypes.c_float)
            L.rope_tables_build.argtypes = [vp, vp, i64, i32, f64, i32, vp]
            L.rope_tables_build.restype = i32
            L.rope_tables_build_scaled.argtypes = [vp, vp, i64, i32, f64, i32, f64, vp]
            L.rope_tables_build_scaled.restype = i32
            L.rope_apply_qk.argtypes = [vp, vp, vp, vp, i32, i64, i32, i32, i32, i32, i32,
                                        _i64p, _i64p, _i64p, _i64p, vp, i32, vp, vp, i64, vp]
            L.rope_apply_qk.restype = i32
            L.attn_fwd_causal_rope.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i64, i64,
                                               i32, i64, i32, i32, i32, vp, vp, i64, f32,
                                               _i64p, _i64p, _i64p, _i64p, vp]
            L.attn_fwd_causal_rope.restype = i32
            L.attn_bwd_workspace_size.argtypes = [i32, i32, i32, i32, i64, i64, i32]
            L.attn_bwd_workspace_size.restype = ctypes.c_size_t
            L.attn_bwd_causal_rope.argtypes = ([vp] * 9 + [i32, i32, i32, i32, i64, i64, i32, i64,
                                               i32, i32, i32, vp, vp, i64, f32] + [_i64p] * 8
                                              + [vp, ctypes.c_size_t, vp])
            L.attn_bwd_causal_rope.restype = i32
            cp = ctypes.POINTER(KVCacheDesc)
            i32p = ctypes.POINTER(ctypes.c_int32)
            L.rope_append_kv.argtypes = [vp, vp, vp, vp, cp, i32, i64, i32, i32, i32, i32, i32,
                                         _i64p, _i64p, _i64p, _i64p, vp, vp, i32, vp, vp, i64,
                                         vp]
            L.rope_append_kv.restype = i32
            L.attn_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i64]
            L.attn_decode_workspace_size.restype = ctypes.c_size_t
            L.attn_decode.argtypes = [vp, vp, vp, cp, i32, i32, i32, i32, i32, i32, vp, vp, i64,
                                      f32, _i64p, _i64p, vp, ctypes.c_size_t, vp]
            L.attn_decode.restype = i32
            L.attn_decode_noalloc.argtypes = [vp, vp, vp, cp, i32, i32, i32, i32, i32, i32, vp,
                                              vp, i64, f32, _i64p, _i64p, vp]
            L.attn_decode_noalloc.restype = i32
            L.ra_get_device_status.argtypes = [vp]
            L.ra_get_device_status.restype = i32
            L.ra_status_string.argtypes = [i32]
            L.ra_status_string.restype = ctypes.c_char_p
            L.ra_last_error.argtypes = []
            L.ra_last_error.restype = ctypes.c_char_p
            L.ra_last_launch.argtypes = []
            L.ra_last_launch.restype = ctypes.c_char_p
            _lib = L
    return _lib


def ra_status_string(code: int) -> str:
    """English name of an ra_status code."""
    return lib().ra_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != 0:
        L = lib()
        raise RAError(code, f"{what}: {L.ra_status_string(code).decode()} "
                            f"({L.ra_last_error().decode()})")


def _arr(vals):
    return (ctypes.c_int64 * len(vals))(*[int(x) for x in vals])


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(device, stream):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _cuda(t, name):
    if t is not None and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")


def rope_tables_build(cos_out: torch.Tensor, sin_out: torch.Tensor, base: float,
                      freq_dim: int = 0, stream=None, pos_scale: float = 1.0):
    """Fills fp32 tables [rows, rot_dim/2] with cos/sin((p / pos_scale) *
    base^(-2i/F)); pos_scale != 1 calls rope_tables_build_scaled (position
    interpolation)."""
    _cuda(cos_out, "cos_out")
    _cuda(sin_out, "sin_out")
    if (cos_out.dtype != torch.float32 or sin_out.shape != cos_out.shape or cos_out.dim() != 2
            or not cos_out.is_contiguous() or not sin_out.is_contiguous()):
        raise ValueError("tables must be contiguous fp32 [rows, rot_dim/2] of equal shape")
    rows, half = cos_out.shape
    if pos_scale == 1.0:
        _check(lib().rope_tables_build(_ptr(cos_out), _ptr(sin_out), rows, 2 * half, float(base),
                                       int(freq_dim), _stream(cos_out.device, stream)),
               "rope_tables_build")
    else:
        _check(lib().rope_tables_build_scaled(_ptr(cos_out), _ptr(sin_out), rows, 2 * half,
                                              float(base), int(freq_dim), float(pos_scale),
                                              _stream(cos_out.device, stream)),
               "rope_tables_build_scaled")
    return cos_out, sin_out


def rope_tables_build_scaled(cos_out, sin_out, base: float, pos_scale: float, freq_dim: int = 0,
                             stream=None):
    """Position-interpolated tables: cos/sin((p / pos_scale) * theta_i)."""
    return rope_tables_build(cos_out, sin_out, base, freq_dim, stream, pos_scale)


def make_tables(rows: int, rot_dim: int, base: float, freq_dim: int = 0, device="cuda",
                stream=None, pos_scale: float = 1.0):
    """Allocates and builds the cos/sin tables (fp32 [rows, rot_dim/2] each)."""
    c = torch.empty((rows, rot_dim // 2), dtype=torch.float32, device=device)
    s = torch.empty_like(c)
    return rope_tables_build(c, s, base, freq_dim, stream, pos_scale)


def rope_apply_qk(q, k, positions, cos, sin, rot_dim: int | None = None, layout: int = NEOX,
                  q_out=None, k_out=None, stream=None):
    """Rotates token-major q [T, Hq, D] and k [T, Hkv, D] (either may be None)
    at positions[t] in one launch; in place unless q_out / k_out are given.
    Returns (q result, k result)."""
    ref = q if q is not None else k
    if ref is None:
        raise ValueError("q or k required")
    for t, n in ((q, "q"), (k, "k"), (q_out, "q_out"), (k_out, "k_out"), (positions, "positions"),
                 (cos, "cos"), (sin, "sin")):
        _cuda(t, n)
    if positions.dtype not in (torch.int32, torch.int64) or positions.dim() != 1:
        raise ValueError("positions must be int32 or int64 [T]")
    T, _, D = ref.shape
    for t, n in ((q, "q"), (k, "k"), (q_out, "q_out"), (k_out, "k_out")):
        if t is not None and (t.dim() != 3 or t.shape[0] != T or t.shape[2] != D
                              or t.stride(2) != 1 or t.dtype != ref.dtype):
            raise ValueError(f"{n} must be [T, H, D] of one dtype with unit last stride")
    if q_out is not None and q is not None and q_out.shape != q.shape:
        raise ValueError("q_out shape must equal q's")
    if k_out is not None and k is not None and k_out.shape != k.shape:
        raise ValueError("k_out shape must equal k's")
    if positions.shape[0] != T:
        raise ValueError("one position per token required")
    if cos.dtype != torch.float32 or cos.shape != sin.shape or not cos.is_contiguous():
        raise ValueError("tables must be contiguous fp32 of equal shape")
    rot_dim = 2 * cos.shape[1] if rot_dim is None else int(rot_dim)
    if rot_dim != 2 * cos.shape[1]:
        raise ValueError("rot_dim must match the table width (rot_dim/2 columns)")
    Hq = q.shape[1] if q is not None else 0
    Hkv = k.shape[1] if k is not None else 0
    st = lambda t: _arr([t.stride(0), t.stride(1)]) if t is not None else None
    _check(lib().rope_apply_qk(
        _ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), _DT[ref.dtype], T, Hq, Hkv, D, rot_dim,
        int(layout), st(q), st(k), st(q_out), st(k_out), _ptr(positions),
        int(positions.dtype == torch.int64), _ptr(cos), _ptr(sin), cos.shape[0],
        _stream(ref.device, stream)), "rope_apply_qk")
    return (q_out if q_out is not None else q), (k_out if k_out is not None else k)


def attn_fwd_causal_rope(q, k, v, cos=None, sin=None, kv_offset: int = 0, apply_rope: bool = True,
                         rot_dim: int | None = None, layout: int = NEOX,
                         softmax_scale: float | None = None, out=None, lse=None,
                         return_lse: bool = True, stream=None):
    """Causal attention forward with RoPE fused in.  q [B,Hq,Sq,D];
    k, v [B,Hkv,Sk,D]; query row i sits at position kv_offset + i, key j at j.
    Returns (O [B,Hq,Sq,D] in q's dtype, LSE fp32 [B,Hq,Sq] or None)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (cos, "cos"), (sin, "sin"), (out, "out"),
                 (lse, "lse")):
        _cuda(t, n)
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, H, S, D]")
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    if k.shape != (B, Hkv, Sk, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, Sk, D] with q's B and D")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in _DT:
        raise ValueError("q, k, v must share one of fp32 / bf16 / fp16")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if t.stride(3) != 1:
            raise ValueError(f"{n} needs unit stride in the head dimension")
    if out is None:
        out = torch.empty((B, Hq, Sq, D), dtype=q.dtype, device=q.device)
    elif out.shape != (B, Hq, Sq, D) or out.dtype != q.dtype or out.stride(3) != 1:
        raise ValueError("out must be [B, Hq, Sq, D] in q's dtype with unit last stride")
    if return_lse and lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.shape != (B, Hq, Sq) or lse.dtype != torch.float32
                            or not lse.is_contiguous()):
        raise ValueError("lse must be contiguous fp32 [B, Hq, Sq]")
    if apply_rope:
        if cos is None or sin is None:
            raise ValueError("apply_rope needs the cos/sin tables")
        rot_dim = 2 * cos.shape[1] if rot_dim is None else int(rot_dim)
        if rot_dim != 2 * cos.shape[1]:
            raise ValueError("rot_dim must match the table width")
        rows = cos.shape[0]
    else:
        rot_dim, rows = D, 0
    s3 = lambda t: _arr([t.stride(0), t.stride(1), t.stride(2)])
    _check(lib().attn_fwd_causal_rope(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _DT[q.dtype], B, Hq, Hkv, Sq, Sk, D,
        int(kv_offset), int(bool(apply_rope)), rot_dim, int(layout), _ptr(cos), _ptr(sin), rows,
        float(softmax_scale) if softmax_scale is not None else 0.0, s3(q), s3(k), s3(v), s3(out),
        _stream(q.device, stream)), "attn_fwd_causal_rope")
    return out, lse


def attn_bwd_causal_rope(q, k, v, o, lse, dout, cos=None, sin=None, kv_offset: int = 0,
                         apply_rope: bool = True, rot_dim: int | None = None, layout: int = NEOX,
                         softmax_scale: float | None = None, dq=None, dk=None, dv=None,
                         workspace=None, stream=None):
    """Gradients of attn_fwd_causal_rope with respect to the raw q, k, v.
    o and lse come from the forward call with the same arguments; dout is
    dL/dO like o.  Returns (dq, dk, dv) in q's dtype."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (lse, "lse"), (dout, "dout"),
                 (cos, "cos"), (sin, "sin"), (dq, "dq"), (dk, "dk"), (dv, "dv"),
                 (workspace, "workspace")):
        _cuda(t, n)
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, H, S, D]")
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    if k.shape != (B, Hkv, Sk, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, Sk, D] with q's B and D")
    if o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("o and dout must have q's shape")
    for t, n in ((k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        if t.dtype != q.dtype:
            raise ValueError(f"{n} must have q's dtype")
    if q.dtype not in _DT:
        raise ValueError("dtype must be fp32 / bf16 / fp16")
    if lse.shape != (B, Hq, Sq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B, Hq, Sq]")
    outs = []
    for t, ref, n in ((dq, q, "dq"), (dk, k, "dk"), (dv, v, "dv")):
        if t is None:
            t = torch.empty(ref.shape, dtype=ref.dtype, device=ref.device)
        elif t.shape != ref.shape or t.dtype != ref.dtype:
            raise ValueError(f"{n} must match its input's shape and dtype")
        outs.append(t)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout"), *zip(outs, ("dq", "dk", "dv"))):
        if t.stride(3) != 1:
            raise ValueError(f"{n} needs unit stride in the head dimension")
    if apply_rope:
        if cos is None or sin is None:
            raise ValueError("apply_rope needs the cos/sin tables")
        rot_dim = 2 * cos.shape[1] if rot_dim is None else int(rot_dim)
        if rot_dim != 2 * cos.shape[1]:
            raise ValueError("rot_dim must match the table width")
        rows = cos.shape[0]
    else:
        rot_dim, rows = D, 0
    need = int(lib().attn_bwd_workspace_size(_DT[q.dtype], B, Hq, Hkv, Sq, Sk, D))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    s3 = lambda t: _arr([t.stride(0), t.stride(1), t.stride(2)])
    _check(lib().attn_bwd_causal_rope(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(outs[0]), _ptr(outs[1]),
        _ptr(outs[2]), _DT[q.dtype], B, Hq, Hkv, Sq, Sk, D, int(kv_offset), int(bool(apply_rope)),
        rot_dim, int(layout), _ptr(cos), _ptr(sin), rows,
        float(softmax_scale) if softmax_scale is not None else 0.0,
        s3(q), s3(k), s3(v), s3(o), s3(dout), s3(outs[0]), s3(outs[1]), s3(outs[2]),
        _ptr(workspace), wbytes, _stream(q.device, stream)), "attn_bwd_causal_rope")
    return tuple(outs)


class KVCache:
    """A decoder KV cache: k and v are [rows, Hkv, D] views (any strides with a
    unit last stride; e.g. token-major tensors, or head-major storage
    permuted to that shape), seq_start int64 [n_seqs] on the device holds each
    sequence's first row; the key at position j of sequence s is row
    seq_start[s] + j."""

    def __init__(self, k: torch.Tensor, v: torch.Tensor, seq_start: torch.Tensor):
        for t, n in ((k, "k"), (v, "v"), (seq_start, "seq_start")):
            _cuda(t, n)
        if k.dim() != 3 or v.shape != k.shape or k.dtype != v.dtype or k.dtype not in _DT:
            raise ValueError("k and v must be [rows, Hkv, D] of one of fp32 / bf16 / fp16")
        if k.stride(2) != 1 or v.stride(2) != 1:
            raise ValueError("cache rows need a unit last stride")
        if seq_start.dtype != torch.int64 or seq_start.dim() != 1 or not seq_start.is_contiguous():
            raise ValueError("seq_start must be contiguous int64 [n_seqs]")
        self.k, self.v, self.seq_start = k, v, seq_start

    @property
    def Hkv(self):
        return self.k.shape[1]

    @property
    def D(self):
        return self.k.shape[2]

    def desc(self) -> KVCacheDesc:
        d = KVCacheDesc()
        d.k, d.v = self.k.data_ptr(), self.v.data_ptr()
        d.k_strides[0], d.k_strides[1] = self.k.stride(0), self.k.stride(1)
        d.v_strides[0], d.v_strides[1] = self.v.stride(0), self.v.stride(1)
        d.rows = self.k.shape[0]
        d.seq_start = self.seq_start.data_ptr()
        d.n_seqs = self.seq_start.shape[0]
        return d


def rope_append_kv(cache: KVCache, q, k_new, v_new, positions, cos, sin, seq_ids=None,
                   layout: int = NEOX, q_out=None, stream=None):
    """Rotates q [T,Hq,D] (in place unless q_out), writes rot(k_new) and v_new
    ([T,Hkv,D]) into the cache rows seq_start[seq_ids[t]] + positions[t]
    (seq_ids None: token t is sequence t).  q may be None.  Returns q's result."""
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (positions, "positions"),
                 (cos, "cos"), (sin, "sin"), (seq_ids, "seq_ids"), (q_out, "q_out")):
        _cuda(t, n)
    if k_new.dim() != 3 or v_new.shape != k_new.shape:
        raise ValueError("k_new and v_new must be [T, Hkv, D]")
    T, Hkv, D = k_new.shape
    dt = cache.k.dtype
    if k_new.dtype != dt or v_new.dtype != dt or (q is not None and q.dtype != dt):
        raise ValueError("q, k_new, v_new must have the cache's dtype")
    if Hkv != cache.Hkv or D != cache.D:
        raise ValueError("k_new heads / head size must match the cache")
    for t, n in ((q, "q"), (q_out, "q_out"), (k_new, "k_new"), (v_new, "v_new")):
        if t is not None and (t.dim() != 3 or t.shape[0] != T or t.shape[2] != D
                              or t.stride(2) != 1):
            raise ValueError(f"{n} must be [T, H, D] with unit last stride")
    if q_out is not None and (q is None or q_out.shape != q.shape or q_out.dtype != q.dtype):
        raise ValueError("q_out must match q")
    if positions.dtype not in (torch.int32, torch.int64) or positions.shape != (T,):
        raise ValueError("positions must be int32 or int64 [T]")
    if seq_ids is not None and (seq_ids.dtype != torch.int32 or seq_ids.shape != (T,)
                                or not seq_ids.is_contiguous()):
        raise ValueError("seq_ids must be contiguous int32 [T]")
    if cos.dtype != torch.float32 or cos.shape != sin.shape or not cos.is_contiguous():
        raise ValueError("tables must be contiguous fp32 of equal shape")
    rot_dim = 2 * cos.shape[1]
    Hq = q.shape[1] if q is not None else 0
    st = lambda t: _arr([t.stride(0), t.stride(1)]) if t is not None else None
    d = cache.desc()
    _check(lib().rope_append_kv(
        _ptr(q), _ptr(q_out), _ptr(k_new), _ptr(v_new), ctypes.byref(d), _DT[dt], T, Hq, Hkv, D,
        rot_dim, int(layout), st(q), st(q_out), st(k_new), st(v_new), _ptr(seq_ids),
        _ptr(positions), int(positions.dtype == torch.int64), _ptr(cos), _ptr(sin), cos.shape[0],
        _stream(k_new.device, stream)), "rope_append_kv")
    return q_out if q_out is not None else q


def attn_decode_workspace_size(dtype, B: int, Hq: int, Hkv: int, Sq: int, D: int,
                               max_kv_len: int) -> int:
    """Workspace bytes attn_decode needs on the current device."""
    n = lib().attn_decode_workspace_size(_DT[dtype], B, Hq, Hkv, Sq, D, int(max_kv_len))
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid decode sizes")
    return int(n)


def attn_decode(cache: KVCache, q, kv_len, max_kv_len: int, seq_ids=None,
                softmax_scale: float | None = None, out=None, lse=None, return_lse: bool = True,
                workspace=None, stream=None):
    """Decode attention over the cache (rotated K, raw V).  q [B,Hq,Sq,D]
    (already rotated; any strides with unit last stride), kv_len int32 [B]
    keys of each entry (the Sq new ones included), max_kv_len >= max(kv_len).
    Query i of entry b sits at kv_len[b] - Sq + i.  Returns (O, LSE or None)."""
    for t, n in ((q, "q"), (kv_len, "kv_len"), (seq_ids, "seq_ids"), (out, "out"), (lse, "lse"),
                 (workspace, "workspace")):
        _cuda(t, n)
    if q.dim() != 4 or q.stride(3) != 1:
        raise ValueError("q must be [B, Hq, Sq, D] with unit last stride")
    B, Hq, Sq, D = q.shape
    if q.dtype != cache.k.dtype or D != cache.D:
        raise ValueError("q must have the cache's dtype and head size")
    if kv_len.dtype != torch.int32 or kv_len.shape != (B,) or not kv_len.is_contiguous():
        raise ValueError("kv_len must be contiguous int32 [B]")
    if seq_ids is not None and (seq_ids.dtype != torch.int32 or seq_ids.shape != (B,)
                                or not seq_ids.is_contiguous()):
        raise ValueError("seq_ids must be contiguous int32 [B]")
    if out is None:
        out = torch.empty((B, Hq, Sq, D), dtype=q.dtype, device=q.device)
    elif out.shape != (B, Hq, Sq, D) or out.dtype != q.dtype or out.stride(3) != 1:
        raise ValueError("out must be [B, Hq, Sq, D] in q's dtype with unit last stride")
    if return_lse and lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.shape != (B, Hq, Sq) or lse.dtype != torch.float32
                            or not lse.is_contiguous()):
        raise ValueError("lse must be contiguous fp32 [B, Hq, Sq]")
    need = attn_decode_workspace_size(q.dtype, B, Hq, cache.Hkv, Sq, D, max_kv_len)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    s3 = lambda t: _arr([t.stride(0), t.stride(1), t.stride(2)])
    d = cache.desc()
    _check(lib().attn_decode(
        _ptr(q), _ptr(out), _ptr(lse), ctypes.byref(d), _DT[q.dtype], B, Hq, cache.Hkv, Sq, D,
        _ptr(seq_ids), _ptr(kv_len), int(max_kv_len),
        float(softmax_scale) if softmax_scale is not None else 0.0, s3(q), s3(out),
        _ptr(workspace), wbytes, _stream(q.device, stream)), "attn_decode")
    return out, lse


def attn_decode_noalloc(cache: KVCache, q, kv_len, max_kv_len: int, out, lse=None, seq_ids=None,
                        softmax_scale: float | None = None, stream=None):
    """attn_decode with the split workspace in the library's static device
    region: neither this function nor the library allocates (out, and lse
    if wanted, are the caller's).  Returns (out, lse)."""
    for t, n in ((q, "q"), (kv_len, "kv_len"), (seq_ids, "seq_ids"), (out, "out"), (lse, "lse")):
        _cuda(t, n)
    if q.dim() != 4 or q.stride(3) != 1:
        raise ValueError("q must be [B, Hq, Sq, D] with unit last stride")
    B, Hq, Sq, D = q.shape
    if q.dtype != cache.k.dtype or D != cache.D:
        raise ValueError("q must have the cache's dtype and head size")
    if kv_len.dtype != torch.int32 or kv_len.shape != (B,) or not kv_len.is_contiguous():
        raise ValueError("kv_len must be contiguous int32 [B]")
    if seq_ids is not None and (seq_ids.dtype != torch.int32 or seq_ids.shape != (B,)
                                or not seq_ids.is_contiguous()):
        raise ValueError("seq_ids must be contiguous int32 [B]")
    if out is None or out.shape != (B, Hq, Sq, D) or out.dtype != q.dtype or out.stride(3) != 1:
        raise ValueError("out must be [B, Hq, Sq, D] in q's dtype with unit last stride")
    if lse is not None and (lse.shape != (B, Hq, Sq) or lse.dtype != torch.float32
                            or not lse.is_contiguous()):
        raise ValueError("lse must be contiguous fp32 [B, Hq, Sq]")
    s3 = lambda t: _arr([t.stride(0), t.stride(1), t.stride(2)])
    d = cache.desc()
    _check(lib().attn_decode_noalloc(
        _ptr(q), _ptr(out), _ptr(lse), ctypes.byref(d), _DT[q.dtype], B, Hq, cache.Hkv, Sq, D,
        _ptr(seq_ids), _ptr(kv_len), int(max_kv_len),
        float(softmax_scale) if softmax_scale is not None else 0.0, s3(q), s3(out),
        _stream(q.device, stream)), "attn_decode_noalloc")
    return out, lse


def ra_last_launch() -> list[str]:
    """Kernels the last attention / append / decode call on this thread launched."""
    return lib().ra_last_launch().decode().split()


def ra_get_device_status(stream=None, device=None) -> int:
    """Synchronises the stream and returns (and clears) the device status code."""
    return int(lib().ra_get_device_status(_stream(device, stream)))
