"""Planted mistakes: each broken single-head attention must fail at least one pin.

The mutants are small, deliberately wrong restatements of the definition, run
on the CPU only.  They show that the pins in test_oracle.py would catch a
dropped term, a wrong sign or index, a transposed operand or a wrong log base
had one slipped into the oracle.
"""
import numpy as np
import pytest

from test_oracle import PINS


def _attn(q, k, v, scale, causal, bug):
    Sq, Sk = q.shape[0], k.shape[0]
    s = (q @ k.T) if bug != "no_scale" else (q @ k.T)
    if bug != "no_scale":
        s = scale * s
    if bug == "transposed" and Sq == Sk:
        s = s.T
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    vis = np.ones_like(s, dtype=bool)
    if causal:
        vis = {"mask_flipped": j >= i, "mask_strict": j < i}.get(bug, j <= i)
        if bug == "mask_strict":
            vis = vis | ((i == 0) & (j == 0))   # keep row 0 defined
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.where(vis, np.exp(s - m), 0.0)
    if bug == "softmax_axis0":
        z = e.sum(axis=0, keepdims=True)
        p = e / np.where(z == 0, 1, z)
    else:
        z = e.sum(axis=1, keepdims=True)
        p = e if bug == "no_normalise" else e / z
    vv = v[::-1] if bug == "v_reversed" else v
    o = p @ vv
    zz = e.sum(axis=1)
    if bug == "lse_no_max":
        lse = np.log(zz)
    elif bug == "lse_log2":
        lse = m[:, 0] + np.log2(zz)
    elif bug == "lse_unscaled":
        lse = m[:, 0] / (scale if scale else 1.0) + np.log(zz)
    else:
        lse = m[:, 0] + np.log(zz)
    return o, lse


BUGS = ["no_scale", "transposed", "mask_flipped", "mask_strict", "softmax_axis0",
        "no_normalise", "v_reversed", "lse_no_max", "lse_log2", "lse_unscaled"]


def test_correct_restatement_passes_all_pins():
    for pin in PINS:
        pin(lambda q, k, v, s, c: _attn(q, k, v, s, c, None))


@pytest.mark.parametrize("bug", BUGS)
def test_mutant_is_caught(bug):
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(lambda q, k, v, s, c: _attn(q, k, v, s, c, bug))
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {bug!r}"
