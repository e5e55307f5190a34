"""Seeded randomized parity of the tensor-core forward and backward against
the fp64 oracle: shapes, dtypes, layouts, partial rotation, offsets, keys
past the last query and kv-head groupings drawn from a fixed generator, so
that the cases are the same on every run.  Sizes span single-tile grids,
split blocks (one wave) and head-pair grids launched in bands (more blocks
than SMs).  Bounds as in test_gpu_attention / test_gpu_backward."""
import numpy as np
import pytest
import torch

import workloads as wl
from test_gpu_attention import orc, ra, run_case  # noqa: F401  (fixtures)
from test_gpu_backward import grads_case

pytestmark = pytest.mark.gpu

NEOX, GPTJ = 0, 1


def _cases(seed, n, max_work, max_sq):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        dt = [torch.bfloat16, torch.float16][rng.integers(2)]
        D = int(rng.choice([64, 128]))
        G = int(rng.choice([1, 2, 3, 4, 8]))
        Hkv = int(rng.integers(1, 9))
        Hq = Hkv * G
        if Hq > 32:
            continue
        B = int(rng.integers(1, 4))
        Sq = int(rng.integers(1, max_sq + 1))
        off = int(rng.integers(0, 600)) if rng.random() < 0.6 else 0
        extra = int(rng.integers(1, 200)) if rng.random() < 0.2 else 0
        Sk = Sq + off + extra
        if B * Hq * Sq * Sk * D > max_work:
            continue
        layout = int(rng.integers(2))
        rot = int(rng.choice([D, D // 2, D // 4]))
        out.append((dt, B, Hq, Hkv, Sq, Sk, D, off, layout, rot))
    return out


FWD = _cases(2026, 48, 4e10, 1600)
BWD = _cases(2027, 16, 2e9, 600)


def _id(c):
    dt, B, Hq, Hkv, Sq, Sk, D, off, layout, rot = c
    return (f"{'bf16' if dt == torch.bfloat16 else 'fp16'}-{B}x{Hq}q{Hkv}kv-"
            f"Sq{Sq}-Sk{Sk}-D{D}-off{off}-{'neox' if layout == NEOX else 'gptj'}-r{rot}")


@pytest.mark.parametrize("case", FWD, ids=[_id(c) for c in FWD])
def test_forward_random_case(ra, orc, case):
    dt, B, Hq, Hkv, Sq, Sk, D, off, layout, rot = case
    run_case(ra, orc, dt, B, Hq, Hkv, Sq, Sk, D, off, layout=layout, rot_dim=rot,
             seed=Sq * 7 + Sk + D)


@pytest.mark.parametrize("case", BWD, ids=[_id(c) for c in BWD])
def test_backward_random_case(ra, orc, case):
    dt, B, Hq, Hkv, Sq, Sk, D, off, layout, rot = case
    grads_case(ra, orc, dt, B, Hq, Hkv, Sq, Sk, D, off, layout, rot, seed=Sq * 5 + Sk + D)
