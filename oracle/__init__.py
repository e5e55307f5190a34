"""fp64 CPU oracle for RoPE and causal softmax attention.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg may import this package.  It shares no
code with the CUDA library (``rope_causal_attention_gb300``) and never imports
it; the two meet only through the seeded generators in ``workloads``.

Contents
--------
* ``rope_freqs``, ``rope_tables``, ``rope_rows``: the rotation itself, in the C
  library built from ``oracle.c`` (fp64, libm).
* ``attention``: naive two-pass causal softmax attention with optional RoPE,
  for all rows or a selected subset (C, fp64, threaded over rows).
* ``decode_attention``: the decoder step's attention over a KV cache of
  already-rotated keys (per sequence, the same naive attention).
* ``attention_bwd`` (``oracle.backward``): gradients of the fused RoPE
  attention, probabilities rebuilt from Q and K (numpy, fp64);
  ``attention_bwd_rows``: selected query / key rows of the same gradients,
  for problems too large to differentiate densely.
* ``tiled_attention`` (``oracle.tiled``): the Q-block-outer / K-block-inner
  online-softmax recurrence, used only to show that the recurrence reaches
  the naive result.

Sources (page title, section):
* "RoPE and FlashAttention: relative positions and online softmax",
  sections 1, 2, 4 and 5.
* "Write Triton Rope Kernel", Required reasoning process and Correctness
  requirements.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .tiled import tiled_attention  # noqa: F401

NEOX = 0
GPTJ = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles ``oracle.c`` into ``_build/liboracle.so`` (gcc, fp64, no FMA
    contraction so that x86_64 and aarch64 give the same bits)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            fp = ctypes.POINTER(ctypes.c_float)
            lp = ctypes.POINTER(ctypes.c_int64)
            i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.oracle_rope_freqs.argtypes = [i32, i32, f64, dp]
            lib.oracle_rope_freqs.restype = None
            lib.oracle_rope_tables.argtypes = [i64, i32, i32, f64, dp, dp]
            lib.oracle_rope_tables.restype = None
            lib.oracle_rope_tables_scaled.argtypes = [i64, i32, i32, f64, f64, dp, dp]
            lib.oracle_rope_tables_scaled.restype = None
            lib.oracle_rope_rows.argtypes = [dp, i64, i32, lp, i32, i32, f64, i32, dp]
            lib.oracle_rope_rows.restype = i32
            lib.oracle_attention.argtypes = [fp, fp, fp, i32, i32, i32, i64, i64, i32, i64,
                                             i32, i32, i32, f64, i32, f64, lp, i64, dp, dp, i32]
            lib.oracle_attention.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def rope_freqs(rot_dim: int, base: float, freq_dim: int = 0) -> np.ndarray:
    """theta_i = base**(-2i/F), i < rot_dim/2 (F = freq_dim or rot_dim)."""
    out = np.empty(rot_dim // 2, dtype=np.float64)
    _load().oracle_rope_freqs(rot_dim, freq_dim, float(base), _ptr(out, ctypes.c_double))
    return out


def rope_tables(rows: int, rot_dim: int, base: float, freq_dim: int = 0):
    """fp64 cos and sin of p*theta_i, each [rows, rot_dim/2]."""
    half = rot_dim // 2
    c = np.empty((rows, half), dtype=np.float64)
    s = np.empty((rows, half), dtype=np.float64)
    _load().oracle_rope_tables(rows, rot_dim, freq_dim, float(base),
                               _ptr(c, ctypes.c_double), _ptr(s, ctypes.c_double))
    return c, s


def rope_tables_scaled(rows: int, rot_dim: int, base: float, pos_scale: float,
                       freq_dim: int = 0):
    """fp64 cos and sin of (p / pos_scale) * theta_i (position interpolation)."""
    half = rot_dim // 2
    c = np.empty((rows, half), dtype=np.float64)
    s = np.empty((rows, half), dtype=np.float64)
    _load().oracle_rope_tables_scaled(rows, rot_dim, freq_dim, float(base), float(pos_scale),
                                      _ptr(c, ctypes.c_double), _ptr(s, ctypes.c_double))
    return c, s


def rope_rows(x, positions, rot_dim: int | None = None, base: float = 10000.0,
              layout: int = NEOX, freq_dim: int = 0) -> np.ndarray:
    """Rotates every row x[..., r, :] at positions[r] (positions broadcast over
    the leading dims).  Returns fp64 of x's shape; the input is not modified."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    D = x.shape[-1]
    rot_dim = D if rot_dim is None else rot_dim
    pos = np.asarray(positions, dtype=np.int64)
    if pos.ndim != 1 or pos.shape[0] != x.shape[-2]:
        raise ValueError("one absolute position per row required")
    lead = int(np.prod(x.shape[:-2], dtype=np.int64))
    pos_all = np.ascontiguousarray(np.tile(pos, lead))
    y = np.empty_like(x)
    rc = _load().oracle_rope_rows(_ptr(x, ctypes.c_double), pos_all.shape[0], D,
                                  _ptr(pos_all, ctypes.c_int64), rot_dim, freq_dim,
                                  float(base), layout, _ptr(y, ctypes.c_double))
    if rc != 0:
        raise ValueError("invalid RoPE arguments (D and rot_dim even, 2<=rot_dim<=D, base>0)")
    return y


def rope_tokens(x, positions, rot_dim: int | None = None, base: float = 10000.0,
                layout: int = NEOX, freq_dim: int = 0) -> np.ndarray:
    """Token-major [T, H, D] input: token t of every head rotated at positions[t]."""
    x = np.asarray(x, dtype=np.float64)
    T, H, D = x.shape
    pos = np.repeat(np.asarray(positions, dtype=np.int64), H)
    y = rope_rows(x.reshape(T * H, D), pos, rot_dim, base, layout, freq_dim)
    return y.reshape(T, H, D)


def attention(q, k, v, kv_offset: int = 0, apply_rope: bool = True, rot_dim: int | None = None,
              base: float = 10000.0, layout: int = NEOX, scale: float | None = None,
              freq_dim: int = 0, rows=None, nthreads: int | None = None):
    """Causal attention, fp64.  q [B,Hq,Sq,D]; k, v [B,Hkv,Sk,D] (any real dtype,
    upcast exactly through float32).  Query row i sits at absolute position
    kv_offset + i and sees keys j <= kv_offset + i (j < Sk); key j sits at j.

    rows: None for every row (returns O [B,Hq,Sq,D], LSE [B,Hq,Sq]) or an array
    of flat row indices (b*Hq + h)*Sq + i (returns O [n,D], LSE [n])."""
    q = np.ascontiguousarray(np.asarray(q, dtype=np.float32))
    k = np.ascontiguousarray(np.asarray(k, dtype=np.float32))
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    if k.shape != (B, Hkv, Sk, D) or v.shape != k.shape:
        raise ValueError("q [B,Hq,Sq,D], k and v [B,Hkv,Sk,D] required")
    rot_dim = D if rot_dim is None else rot_dim
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    full = rows is None
    sel = (np.arange(B * Hq * Sq, dtype=np.int64) if full
           else np.ascontiguousarray(np.asarray(rows, dtype=np.int64)))
    o = np.empty((sel.shape[0], D), dtype=np.float64)
    lse = np.empty(sel.shape[0], dtype=np.float64)
    rc = _load().oracle_attention(
        _ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
        B, Hq, Hkv, Sq, Sk, D, int(kv_offset), int(bool(apply_rope)), rot_dim, freq_dim,
        float(base), layout, scale, _ptr(sel, ctypes.c_int64), sel.shape[0],
        _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
        nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"invalid attention arguments (oracle rc={rc})")
    if full:
        return o.reshape(B, Hq, Sq, D), lse.reshape(B, Hq, Sq)
    return o, lse


def decode_attention(q, k_cache, v_cache, seq_start, kv_len, seq_ids=None,
                     scale: float | None = None, nthreads: int | None = None):
    """Attention of a decoder step over a KV cache, fp64 ("RoPE and
    FlashAttention: relative positions and online softmax", section 2: the
    cache holds rotated K and raw V, new queries are rotated before the
    product; section 5: the offset causal mask).

    q [B,Hq,Sq,D] holds the (already rotated) new queries; k_cache, v_cache
    [rows, Hkv, D].  Entry b reads cache sequence s = seq_ids[b] (default b):
    L = kv_len[b] keys at rows seq_start[s] + j, j < L; its query i sits at
    position L - Sq + i and sees keys j <= L - Sq + i.  Nothing is rotated
    here.  Returns O [B,Hq,Sq,D] and LSE [B,Hq,Sq] (natural log, scale
    included)."""
    q = np.asarray(q)
    B, Hq, Sq, D = q.shape
    o = np.empty((B, Hq, Sq, D), dtype=np.float64)
    lse = np.empty((B, Hq, Sq), dtype=np.float64)
    for b in range(B):
        s = int(seq_ids[b]) if seq_ids is not None else b
        L = int(kv_len[b])
        r0 = int(seq_start[s])
        kb = np.asarray(k_cache[r0:r0 + L]).transpose(1, 0, 2)[None]
        vb = np.asarray(v_cache[r0:r0 + L]).transpose(1, 0, 2)[None]
        ob, lb = attention(q[b:b + 1], kb, vb, kv_offset=L - Sq, apply_rope=False, scale=scale,
                           nthreads=nthreads)
        o[b], lse[b] = ob[0], lb[0]
    return o, lse


from .backward import attention_bwd, attention_bwd_rows  # noqa: E402,F401
