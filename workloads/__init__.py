"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no RoPE or attention arithmetic: it only draws random
numbers, positions and request lengths, and names the workloads.  Both the
CUDA path and the fp64 oracle consume what it produces; neither is imported
here.

Recipe (all workloads):
* q, then k, then v drawn as float32 N(0, 1) from ``torch.Generator('cpu')``
  seeded with ``seed``, then cast to the workload's dtype;
* request lengths, start offsets and positions from
  ``numpy.random.default_rng(seed)``.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

NEOX = 0
GPTJ = 1

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def randn(shape, gen: torch.Generator, dtype: torch.dtype) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(dtype)


def attn_qkv(B, Hq, Hkv, Sq, Sk, D, dtype=torch.bfloat16, seed=0):
    """q [B,Hq,Sq,D], k and v [B,Hkv,Sk,D], CPU, drawn in that order."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = randn((B, Hq, Sq, D), g, dtype)
    k = randn((B, Hkv, Sk, D), g, dtype)
    v = randn((B, Hkv, Sk, D), g, dtype)
    return q, k, v


def rope_qk(T, Hq, Hkv, D, dtype=torch.bfloat16, seed=0):
    """Token-major q [T,Hq,D] and k [T,Hkv,D], CPU, drawn in that order."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = randn((T, Hq, D), g, dtype)
    k = randn((T, Hkv, D), g, dtype)
    return q, k


def decode_tokens(T, Hq, Hkv, D, dtype=torch.bfloat16, seed=0):
    """Token-major new-token q [T,Hq,D], k and v [T,Hkv,D], CPU, drawn in that order."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = randn((T, Hq, D), g, dtype)
    k = randn((T, Hkv, D), g, dtype)
    v = randn((T, Hkv, D), g, dtype)
    return q, k, v


def request_lengths(n_req: int, total: int, max_len: int, rng: np.random.Generator):
    """Lengths drawn uniform in [1, max_len], then moved by +-1 on randomly
    chosen requests (kept within [1, max_len]) until they sum to ``total``."""
    if not (n_req <= total <= n_req * max_len):
        raise ValueError("total tokens out of reach for these lengths")
    L = rng.integers(1, max_len + 1, size=n_req).astype(np.int64)
    diff = int(L.sum()) - total
    while diff != 0:
        r = int(rng.integers(0, n_req))
        if diff > 0 and L[r] > 1:
            L[r] -= 1
            diff -= 1
        elif diff < 0 and L[r] < max_len:
            L[r] += 1
            diff += 1
    return L


def continuous_batch_positions(n_req: int, total: int, max_len: int, table_rows: int, seed: int):
    """Packed per-token positions for ``n_req`` requests: request r holds
    L_r tokens at positions start_r .. start_r + L_r - 1, with start_r uniform
    in [0, table_rows - L_r] so that every position has a table row.
    Returns (positions int64 [total], lengths, starts)."""
    rng = np.random.default_rng(seed)
    L = request_lengths(n_req, total, max_len, rng)
    starts = np.array([rng.integers(0, table_rows - int(l) + 1) for l in L], dtype=np.int64)
    pos = np.concatenate([np.arange(s, s + l, dtype=np.int64) for s, l in zip(starts, L)])
    return pos, L, starts


def decode_positions(n_tokens: int, max_pos: int, seed: int):
    """One token per request at a position uniform in [0, max_pos]."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, max_pos + 1, size=n_tokens).astype(np.int64)


@dataclass(frozen=True)
class AttnWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    D: int
    dtype: str
    layout: int
    base: float
    kv_offset: int
    seed: int
    rot_dim: int = 0  # 0: full D

    @property
    def r(self) -> int:
        return self.rot_dim or self.D

    def flops(self) -> float:
        """QK^T and PV multiply-adds over admissible (i, j) pairs: 4*D per pair
        per query head."""
        pairs = 0
        for i in range(self.Sq):
            pairs += min(self.Sk, self.kv_offset + i + 1)
        return 4.0 * self.D * pairs * self.B * self.Hq

    def inputs(self):
        return attn_qkv(self.B, self.Hq, self.Hkv, self.Sq, self.Sk, self.D,
                        DTYPES[self.dtype], self.seed)


@dataclass(frozen=True)
class RopeWorkload:
    name: str
    T: int
    Hq: int
    Hkv: int
    D: int
    rot_dim: int
    layout: int
    base: float
    table_rows: int
    dtype: str
    seed: int
    kind: str = "batch"  # "batch": continuous batching; "decode": one token per request
    n_req: int = 0
    max_len: int = 0
    in_place: bool = True
    extra: dict = field(default_factory=dict)

    def positions(self) -> np.ndarray:
        if self.kind == "decode":
            return decode_positions(self.T, self.table_rows - 1, self.seed)
        return continuous_batch_positions(self.n_req, self.T, self.max_len,
                                          self.table_rows, self.seed)[0]

    def inputs(self):
        return rope_qk(self.T, self.Hq, self.Hkv, self.D, DTYPES[self.dtype], self.seed)

    def algorithmic_bytes(self) -> int:
        """Bytes a rotation must move: read and write the rotated dims of every
        q and k head, one position per token and one cos and one sin row per
        token.  The untouched tail of an in-place call is not moved."""
        es = torch.tensor([], dtype=DTYPES[self.dtype]).element_size()
        heads = self.Hq + self.Hkv
        moved_dims = self.rot_dim if self.in_place else self.D
        return (2 * self.T * heads * moved_dims * es + 4 * self.T
                + 2 * 4 * (self.rot_dim // 2) * self.T)


@dataclass(frozen=True)
class DecodeWorkload:
    """One decoder step over a KV cache: B requests, Sq new tokens each; the
    new token of request b sits at positions()[b] and its context holds
    kv_lens()[b] = position + Sq keys (the new ones included)."""
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    D: int
    rot_dim: int
    layout: int
    base: float
    table_rows: int
    dtype: str
    seed: int

    def positions(self) -> np.ndarray:
        """Position of each request's first new token (uniform, so that the
        last new token still has a table row)."""
        return decode_positions(self.B, self.table_rows - self.Sq, self.seed)

    def kv_lens(self) -> np.ndarray:
        return self.positions() + self.Sq

    def new_tokens(self):
        """Token-major q [B*Sq,Hq,D], k and v [B*Sq,Hkv,D] of the new tokens."""
        return decode_tokens(self.B * self.Sq, self.Hq, self.Hkv, self.D, DTYPES[self.dtype],
                             self.seed)

    def cache_bytes(self, lens=None) -> int:
        es = torch.tensor([], dtype=DTYPES[self.dtype]).element_size()
        lens = self.kv_lens() if lens is None else lens
        return int(lens.sum()) * self.Hkv * self.D * es * 2

    def algorithmic_bytes(self, lens=None) -> int:
        """Bytes the decode attention must move: read every cached K and V row
        of every request once, read q, write O and LSE, read kv_len and
        seq_start."""
        es = torch.tensor([], dtype=DTYPES[self.dtype]).element_size()
        lens = self.kv_lens() if lens is None else lens
        B = lens.shape[0]
        return (self.cache_bytes(lens) + 2 * B * self.Hq * self.Sq * self.D * es
                + 4 * B * self.Hq * self.Sq + 12 * B)


# --------------------------------------------------------------- named workloads
FP32_ATTN = AttnWorkload("fp32_attn_1x2x128x64_neox", 1, 2, 2, 128, 128, 64, "f32", NEOX,
                         10000.0, 0, 1001)

SWEEP_SHAPES = [(1, 512), (1, 1024), (1, 2048), (1, 4096), (2, 1024), (4, 1024)]
SWEEP = [AttnWorkload(f"bf16_attn_{B}x8x{S}x64_gptj", B, 8, 8, S, S, 64, "bf16", GPTJ,
                      10000.0, 0, 1002) for B, S in SWEEP_SHAPES]

CB_ROPE = RopeWorkload("bf16_rope_cb_T65536_32q8kv_D128", 65536, 32, 8, 128, 128, NEOX,
                       10000.0, 32768, "bf16", 1003, kind="batch", n_req=256, max_len=512)

DECODE_ROPE = RopeWorkload("bf16_rope_decode_T512_64q8kv_D128_r64", 512, 64, 8, 128, 64, NEOX,
                           10000.0, 131072, "bf16", 1004, kind="decode")

LONG_GQA = AttnWorkload("bf16_attn_gqa_1x32q8kv_Sq16384_Sk20480_D128_off4096", 1, 32, 8, 16384,
                        20480, 128, "bf16", NEOX, 500000.0, 4096, 1005)

# the decode rope workload's 512 requests (64 q / 8 kv heads, D = 128, r = 64,
# positions uniform over the 131072-row table) taken one step further: each
# request attends over its whole context, ~137 GB of bf16 K and V in all
DECODE_ATTN = DecodeWorkload("bf16_decode_512req_64q8kv_D128_ctx_upto131072", 512, 64, 8, 1, 128,
                             64, NEOX, 10000.0, 131072, "bf16", 1004)

ALL_ATTN = [FP32_ATTN, *SWEEP, LONG_GQA]
ALL_ROPE = [CB_ROPE, DECODE_ROPE]
