"""Pins of the oracle's sliding-window + global-rows mask (CPU only).

The mask is the hybrid of page "长文本处理性能断层真相", §2.5: a local window
for every query, full attention for the first global_tokens queries, spliced
row-wise.  Each pin is a function of a single-head callable
``fn(q, k, v, scale, causal, window_left, window_right, global_q) -> (O, LSE)``
and checks it against something other than the oracle's own mask: closed forms
(a window of one or two keys), a library routine (torch's fp64 SDPA) run on the
slice of keys a row may see, the page's own row-wise splice of a full and a
windowed result, and invariance under changes to keys outside the band.
Broken variants of the mask (off-by-one band ends, swapped sides, global rows
ignored or read as global keys) must each fail at least one pin.
"""
import math

import numpy as np
import pytest
import torch

from oracle.sdpa_oracle import attention_dense, attention_one_head, attention_varlen

TOL = 1e-12


def _oracle(q, k, v, scale, causal, wl, wr, g):
    return attention_one_head(q, k, v, scale, causal, window_left=wl, window_right=wr,
                              global_q=g)


def _rng(seed):
    return np.random.default_rng(seed)


def _sdpa_rows(q, k, v, scale):
    """torch fp64 SDPA of every row of q over all of k/v, plus its logsumexp."""
    qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(x))[None] for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0].numpy()
    lse = torch.logsumexp(scale * (qt[0] @ kt[0].T), dim=-1).numpy()
    return o, lse


def _band(i, Sk, causal, wl, wr):
    lo = 0 if wl < 0 else max(0, i - wl)
    hi = Sk if wr < 0 else min(Sk, i + wr + 1)
    if causal:
        hi = min(hi, i + 1)
    return lo, hi


# ----------------------------------------------------------------------------- pins
def pin_self_only(fn):
    """A window of one key (the query itself): O_i = V_i, LSE_i = s_ii."""
    r = _rng(1)
    S, D = 9, 5
    q, k, v = r.normal(size=(S, D)), r.normal(size=(S, D)), r.normal(size=(S, D + 2))
    for causal, wl, wr in ((True, 0, 0), (True, 0, -1), (False, 0, 0)):
        o, lse = fn(q, k, v, 0.7, causal, wl, wr, 0)
        np.testing.assert_allclose(o, v[:S], rtol=0, atol=TOL)
        np.testing.assert_allclose(lse, 0.7 * np.einsum("id,id->i", q, k), rtol=0, atol=TOL)


def pin_two_keys(fn):
    """Causal window of two keys: row i >= 1 is a logistic mix of V_{i-1} and V_i."""
    r = _rng(2)
    S, D = 8, 4
    q, k, v = r.normal(size=(S, D)), r.normal(size=(S, D)), r.normal(size=(S, D))
    sc = 0.9
    o, lse = fn(q, k, v, sc, True, 1, 0, 0)
    np.testing.assert_allclose(o[0], v[0], rtol=0, atol=TOL)
    for i in range(1, S):
        a, b = sc * q[i] @ k[i - 1], sc * q[i] @ k[i]
        wa = 1.0 / (1.0 + math.exp(b - a))
        np.testing.assert_allclose(o[i], wa * v[i - 1] + (1 - wa) * v[i], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[i], max(a, b) + math.log1p(math.exp(-abs(a - b))),
                                   rtol=0, atol=1e-12)


def pin_row_equals_sdpa_on_slice(fn):
    """Each windowed row is plain attention (torch SDPA) over the keys its band holds."""
    for seed, (S, D, causal, wl, wr) in enumerate([(13, 4, True, 3, 0), (13, 4, False, 2, 4),
                                                     (11, 3, False, 0, 3), (12, 5, True, 5, -1),
                                                     (10, 4, False, -1, 2), (10, 4, False, 3, -1)]):
        r = _rng(10 + seed)
        q, k, v = r.normal(size=(S, D)), r.normal(size=(S, D)), r.normal(size=(S, D))
        o, lse = fn(q, k, v, 0.6, causal, wl, wr, 0)
        for i in range(S):
            lo, hi = _band(i, S, causal, wl, wr)
            oi, li = _sdpa_rows(q[i:i + 1], k[lo:hi], v[lo:hi], 0.6)
            np.testing.assert_allclose(o[i], oi[0], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[i], li[0], rtol=0, atol=1e-12)


def pin_wide_window_is_plain(fn):
    """A band wider than the sequence changes nothing: equals torch SDPA (causal or not)."""
    r = _rng(3)
    S, D = 10, 4
    q, k, v = r.normal(size=(S, D)), r.normal(size=(S, D)), r.normal(size=(S, D))
    for causal in (False, True):
        o, lse = fn(q, k, v, 0.5, causal, S - 1, S - 1 if not causal else 0, 0)
        qt, kt, vt = (torch.from_numpy(x)[None] for x in (q, k, v))
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=0.5,
                                                               is_causal=causal)[0].numpy()
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
        s = 0.5 * (q @ k.T)
        if causal:
            s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
        np.testing.assert_allclose(lse, torch.logsumexp(torch.from_numpy(s), -1).numpy(),
                                   rtol=0, atol=1e-12)


def pin_global_rows_splice(fn):
    """The page's composition: rows < G from full attention, rows >= G from the window."""
    r = _rng(4)
    S, D, G = 14, 4, 3
    q, k, v = r.normal(size=(S, D)), r.normal(size=(S, D)), r.normal(size=(S, D))
    for causal, wl, wr in ((False, 2, 2), (True, 4, 0), (False, 1, -1)):
        o, lse = fn(q, k, v, 0.8, causal, wl, wr, G)
        o_win, lse_win = fn(q, k, v, 0.8, causal, wl, wr, 0)
        np.testing.assert_allclose(o[G:], o_win[G:], rtol=0, atol=TOL)
        np.testing.assert_allclose(lse[G:], lse_win[G:], rtol=0, atol=TOL)
        for i in range(G):
            hi = i + 1 if causal else S
            oi, li = _sdpa_rows(q[i:i + 1], k[:hi], v[:hi], 0.8)
            np.testing.assert_allclose(o[i], oi[0], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[i], li[0], rtol=0, atol=1e-12)


def pin_outside_keys_irrelevant(fn):
    """Changing keys and values outside row i's band leaves row i unchanged."""
    r = _rng(5)
    S, D, wl, wr = 12, 3, 2, 1
    q, k, v = r.normal(size=(S, D)), r.normal(size=(S, D)), r.normal(size=(S, D))
    o, lse = fn(q, k, v, 1.0, False, wl, wr, 0)
    for i in (0, 5, 11):
        lo, hi = _band(i, S, False, wl, wr)
        k2, v2 = k.copy(), v.copy()
        outside = np.r_[0:lo, hi:S]
        k2[outside] += 10.0
        v2[outside] -= 7.0
        o2, lse2 = fn(q, k2, v2, 1.0, False, wl, wr, 0)
        np.testing.assert_allclose(o2[i], o[i], rtol=0, atol=TOL)
        np.testing.assert_allclose(lse2[i], lse[i], rtol=0, atol=TOL)


WINDOW_PINS = [pin_self_only, pin_two_keys, pin_row_equals_sdpa_on_slice,
               pin_wide_window_is_plain, pin_global_rows_splice, pin_outside_keys_irrelevant]


@pytest.mark.parametrize("pin", WINDOW_PINS, ids=lambda f: f.__name__)
def test_window_pin(pin):
    pin(_oracle)


def test_default_window_is_the_unwindowed_oracle():
    r = _rng(6)
    q, k, v = r.normal(size=(9, 4)), r.normal(size=(7, 4)), r.normal(size=(7, 4))
    for causal in (False, True):
        a = attention_one_head(q, k, v, 0.3, causal)
        b = attention_one_head(q, k, v, 0.3, causal, window_left=-1, window_right=-1, global_q=0)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)


def test_dense_and_varlen_wrappers_pass_the_window_through():
    r = _rng(7)
    B, S, H, D = 2, 9, 2, 4
    q, k, v = (r.normal(size=(B, S, H, D)) for _ in range(3))
    o, lse = attention_dense(q, k, v, 0.4, True, window_left=2, window_right=0, global_q=1)
    for b in range(B):
        for h in range(H):
            ob, lb = attention_one_head(q[b, :, h], k[b, :, h], v[b, :, h], 0.4, True,
                                        window_left=2, window_right=0, global_q=1)
            np.testing.assert_array_equal(o[b, :, h], ob)
            np.testing.assert_array_equal(lse[b, h], lb)
    cu = np.array([0, 4, 9], dtype=np.int32)
    qv, kv, vv = (x.reshape(B * S, H, D)[:9] for x in (q, k, v))
    ov, lv = attention_varlen(qv, kv, vv, cu, cu, 0.4, False, window_left=1, window_right=2,
                              global_q=2)
    for s0, s1 in ((0, 4), (4, 9)):
        for h in range(H):
            ob, lb = attention_one_head(qv[s0:s1, h], kv[s0:s1, h], vv[s0:s1, h], 0.4, False,
                                        window_left=1, window_right=2, global_q=2)
            np.testing.assert_array_equal(ov[s0:s1, h], ob)
            np.testing.assert_array_equal(lv[h, s0:s1], lb)


# ------------------------------------------------------------------ planted mistakes
def _mutant(q, k, v, scale, causal, wl, wr, g, bug):
    Sq, Sk = q.shape[0], k.shape[0]
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    if bug == "sides_swapped":
        wl, wr = wr, wl
    band = i >= (g + 1 if bug == "global_off_by_one" else g)
    if bug == "global_ignored":
        band = np.ones_like(band)
    vis = np.ones((Sq, Sk), dtype=bool)
    if wl >= 0:
        left = (j > i - wl) if bug == "left_exclusive" else (j >= i - wl)
        vis &= ~band | left
    if wr >= 0:
        right = (j < i + wr) if bug == "right_exclusive" else (j <= i + wr)
        vis &= ~band | right
    if bug == "global_keys":  # global tokens read as keys every query sees
        vis |= j < g
    if causal:
        vis &= j <= i
    s = np.where(vis, scale * (q @ k.T), -np.inf)
    has = vis.any(axis=1)
    m = np.where(has, s.max(axis=1), 0.0)
    e = np.where(vis, np.exp(s - m[:, None]), 0.0)
    z = e.sum(axis=1)
    o = (e / np.where(has, z, 1.0)[:, None]) @ v
    with np.errstate(divide="ignore"):
        lse = np.where(has, m + np.log(np.where(has, z, 1.0)), -np.inf)
    return o, lse


WINDOW_BUGS = ["left_exclusive", "right_exclusive", "sides_swapped", "global_ignored",
               "global_keys", "global_off_by_one"]


def test_correct_window_restatement_passes():
    for pin in WINDOW_PINS:
        pin(lambda *a: _mutant(*a, None))


@pytest.mark.parametrize("bug", WINDOW_BUGS)
def test_window_mutant_is_caught(bug):
    caught = []
    for pin in WINDOW_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(lambda *a: _mutant(*a, bug))
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {bug!r}"
