"""Shared check of a rotated tensor against the fp64 oracle (used by the GPU
tests of rope_apply_qk and rope_append_kv).

Tolerances: fp32 outputs within 1e-5 absolute of the fp64 result; bf16/fp16
within one ulp of the exact value plus 2^-21 x (|lo| + |hi|) of the pair's
inputs, with more than 99.9 % of outputs exactly the correctly rounded value;
dims past rot_dim bit-identical.
"""
import numpy as np
import torch

NEOX, GPTJ = 0, 1


def pair_partner(D, rot_dim, layout):
    """Index of the other member of each dim's rotation pair (itself past rot_dim)."""
    idx = np.arange(D)
    half = rot_dim // 2
    part = idx.copy()
    if layout == NEOX:
        part[:half] = idx[:half] + half
        part[half:rot_dim] = idx[half:rot_dim] - half
    else:
        part[:rot_dim] = idx[:rot_dim] ^ 1
    return part


def ulp_of(v, dtype):
    """Spacing of `dtype` numbers at |v| (v float64 array)."""
    mant = {torch.bfloat16: 7, torch.float16: 10}[dtype]
    emin = {torch.bfloat16: -126, torch.float16: -14}[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** emin)))
    return 2.0 ** (e - mant)


def check_rotated(got, x, pos, orc, rot_dim, base, layout, freq_dim=0):
    """got: GPU result (any dtype); x: input (CPU, same dtype).

    fp32: max |got - exact| <= 1e-5.  bf16/fp16: |got - exact| <= one ulp of
    the exact value plus 2^-21 * (|lo| + |hi|) of the pair's inputs, and more
    than 99.9% of outputs equal to the correctly rounded value.  The allowance
    covers the fp32 evaluation with fp32 cos/sin, whose absolute error scales
    with the pair's inputs and can exceed an ulp of an output that nearly
    cancels (lo*c - hi*s close to 0)."""
    want = orc.rope_tokens(x.float().numpy(), np.asarray(pos), rot_dim=rot_dim, base=base,
                           layout=layout, freq_dim=freq_dim)
    got = got.cpu()
    if got.dtype == torch.float32:
        err = np.abs(got.numpy().astype(np.float64) - want).max()
        assert err <= 1e-5, err
    else:
        g = got.float().numpy().astype(np.float64)
        xf = x.float().numpy().astype(np.float64)
        part = pair_partner(x.shape[-1], rot_dim, layout)
        mag = np.abs(xf) + np.abs(xf[..., part])
        bound = ulp_of(want, got.dtype) + 2.0 ** -21 * mag
        excess = np.abs(g - want) - bound
        assert excess.max() <= 0, f"worst excess over bound {excess.max():.3g}"
        exact = got == torch.from_numpy(want).to(got.dtype)
        assert float(exact.float().mean()) > 0.999
    # tail untouched / copied bit for bit
    assert torch.equal(got[..., rot_dim:], x[..., rot_dim:])
