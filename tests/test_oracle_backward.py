"""Pins of the oracle's attention backward (CPU only).

Page "Multi-Head Attention的计算本质与性能瓶颈", §3.3 reserves the backward
interface and says masked connections carry no gradient; the gradient itself is
calculus on the forward definition.  Pins: torch autograd through fp64 SDPA (a
library routine), central finite differences of the pinned forward oracle,
closed forms (constant V, a single key, zero scale), the gradient mask (keys
receive gradient only from queries that see them), and planted mistakes.
"""
import numpy as np
import pytest
import torch

from oracle.sdpa_oracle import (attention_backward_dense, attention_backward_one_head,
                                attention_one_head)


def _rng(seed):
    return np.random.default_rng(seed)


def _torch_grads(q, k, v, do, scale, causal):
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    Sq, Sk = q.shape[0], k.shape[0]
    mask = None
    if causal:
        mask = torch.arange(Sk)[None, :] <= torch.arange(Sq)[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt[None], kt[None], vt[None],
                                                         attn_mask=None if mask is None
                                                         else mask[None], scale=scale)[0]
    o.backward(torch.tensor(do))
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def pin_torch_autograd(fn):
    for seed, (Sq, Sk, D, causal) in enumerate([(7, 7, 4, False), (9, 9, 5, True),
                                                (6, 11, 3, False), (12, 12, 8, True),
                                                (11, 6, 4, False)]):
        r = _rng(seed)
        q, k, v = r.normal(size=(Sq, D)), r.normal(size=(Sk, D)), r.normal(size=(Sk, D + 1))
        do = r.normal(size=(Sq, D + 1))
        got = fn(q, k, v, do, 0.45, causal)
        ref = _torch_grads(q, k, v, do, 0.45, causal)
        for g, rr in zip(got, ref):
            np.testing.assert_allclose(g, rr, rtol=0, atol=1e-11)


def pin_finite_differences(fn):
    r = _rng(20)
    Sq, Sk, D = 4, 5, 3
    q, k, v = r.normal(size=(Sq, D)), r.normal(size=(Sk, D)), r.normal(size=(Sk, D))
    do = r.normal(size=(Sq, D))
    for causal in (False, True):
        dq, dk, dv = fn(q, k, v, do, 0.8, causal)

        def loss(q_, k_, v_):
            o, _ = attention_one_head(q_, k_, v_, 0.8, causal)
            return float((o * do).sum())

        eps = 1e-6
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += eps
                xm[idx] -= eps
                args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
                args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            np.testing.assert_allclose(g, num, rtol=0, atol=1e-7)


def pin_closed_forms(fn):
    r = _rng(21)
    q, k, do = r.normal(size=(6, 4)), r.normal(size=(6, 4)), r.normal(size=(6, 3))
    v = np.tile(r.normal(size=(1, 3)), (6, 1))          # constant V: O does not move
    dq, dk, dv = fn(q, k, v, do, 0.7, False)
    np.testing.assert_allclose(dq, 0, atol=1e-12)
    np.testing.assert_allclose(dk, 0, atol=1e-12)
    dq, dk, dv = fn(q, k[:1], r.normal(size=(1, 3)), do, 0.7, False)   # one key
    np.testing.assert_allclose(dv, do.sum(axis=0, keepdims=True), atol=1e-12)
    np.testing.assert_allclose(dq, 0, atol=1e-12)
    np.testing.assert_allclose(dk, 0, atol=1e-12)
    vv = r.normal(size=(6, 3))
    dq, dk, dv = fn(q, k, vv, do, 0.0, False)            # zero scale: uniform P
    np.testing.assert_allclose(dq, 0, atol=1e-12)
    np.testing.assert_allclose(dk, 0, atol=1e-12)
    np.testing.assert_allclose(dv, np.tile(do.mean(axis=0), (6, 1)), atol=1e-12)


def pin_gradient_mask(fn):
    """Causal: key j gets gradient only from queries i >= j, query i only from keys <= i."""
    r = _rng(22)
    S, D = 8, 4
    q, k, v, do = (r.normal(size=(S, D)) for _ in range(4))
    dq, dk, dv = fn(q, k, v, do, 0.6, True)
    do2 = do.copy()
    do2[:5] += 3.0                       # queries 0..4 change their output gradient
    dq2, dk2, dv2 = fn(q, k, v, do2, 0.6, True)
    np.testing.assert_allclose(dk2[5:], dk[5:], atol=1e-12)   # keys 5..7: unseen by 0..4
    np.testing.assert_allclose(dv2[5:], dv[5:], atol=1e-12)
    k2, v2 = k.copy(), v.copy()
    k2[6:] += 2.0
    v2[6:] -= 1.0                        # keys 6, 7 change
    dq3, _, _ = fn(q, k2, v2, do, 0.6, True)
    np.testing.assert_allclose(dq3[:6], dq[:6], atol=1e-12)   # queries 0..5 never see them


BWD_PINS = [pin_torch_autograd, pin_finite_differences, pin_closed_forms, pin_gradient_mask]


@pytest.mark.parametrize("pin", BWD_PINS, ids=lambda f: f.__name__)
def test_backward_pin(pin):
    pin(attention_backward_one_head)


def test_dense_wrapper_matches_one_head():
    r = _rng(23)
    B, S, H, D = 2, 7, 3, 4
    q, k, v, do = (r.normal(size=(B, S, H, D)) for _ in range(4))
    dq, dk, dv = attention_backward_dense(q, k, v, do, 0.3, True)
    for b in range(B):
        for h in range(H):
            g = attention_backward_one_head(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h],
                                            0.3, True)
            for x, y in zip((dq[b, :, h], dk[b, :, h], dv[b, :, h]), g):
                np.testing.assert_array_equal(x, y)


def _mutant(q, k, v, do, scale, causal, bug):
    _, _, p = attention_one_head(q, k, v, scale, causal, return_p=True)
    dv = (p @ do) if bug == "dv_untransposed" else p.T @ do
    dp = do @ v.T
    row = (dp * p).sum(axis=1, keepdims=True)
    ds = p * dp if bug == "no_row_term" else p * (dp - row)
    dq = (ds @ k) if bug == "dq_no_scale" else scale * (ds @ k)
    dk = scale * (ds @ q) if bug == "dk_wrong_side" else scale * (ds.T @ q)
    if bug == "row_term_colwise":
        ds = p * (dp - (dp * p).sum(axis=0, keepdims=True))
        dq, dk = scale * (ds @ k), scale * (ds.T @ q)
    return dq, dk, dv


BWD_BUGS = ["dv_untransposed", "no_row_term", "dq_no_scale", "dk_wrong_side",
            "row_term_colwise"]


@pytest.mark.parametrize("bug", BWD_BUGS)
def test_backward_mutant_is_caught(bug):
    caught = []
    for pin in BWD_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(lambda *a: _mutant(*a, bug))
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {bug!r}"
