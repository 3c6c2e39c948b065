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
                                attention_backward_sampled, attention_backward_varlen,
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


# ------------------------------------------------------------ packed sequences
def test_varlen_equal_lengths_is_the_dense_batch():
    """B sequences of one length packed back to back: the dense batch, bit for bit."""
    r = _rng(31)
    B, S, H, D = 3, 6, 2, 4
    q, k, v, do = (r.normal(size=(B, S, H, D)) for _ in range(4))
    cu = np.arange(0, (B + 1) * S, S, dtype=np.int32)
    for causal in (False, True):
        dense = attention_backward_dense(q, k, v, do, 0.4, causal)
        packed = attention_backward_varlen(*(x.reshape(B * S, H, D) for x in (q, k, v, do)),
                                           cu, cu, 0.4, causal)
        for x, y in zip(dense, packed):
            np.testing.assert_array_equal(x.reshape(B * S, H, D), y)


def test_varlen_sequences_are_independent():
    """Perturbing one sequence's inputs leaves every other sequence's gradients unchanged,
    and each sequence's gradients are those of its own slices."""
    r = _rng(32)
    H, D = 2, 3
    cq = np.array([0, 5, 5, 12, 15], dtype=np.int32)
    ck = np.array([0, 4, 8, 8, 14], dtype=np.int32)
    q, do = r.normal(size=(16, H, D)), r.normal(size=(16, H, D))   # row 15: no sequence
    k, v = r.normal(size=(14, H, D)), r.normal(size=(14, H, D))
    g = attention_backward_varlen(q, k, v, do, cq, ck, 0.7, True)
    assert np.all(np.isnan(g[0][15]))
    # sequence 1 has keys but no queries, sequence 2 queries but no keys
    assert np.all(g[1][4:8] == 0) and np.all(g[2][4:8] == 0) and np.all(g[0][5:12] == 0)
    k2, v2 = k.copy(), v.copy()
    k2[8:14] += 3.0
    v2[8:14] -= 2.0
    g2 = attention_backward_varlen(q, k2, v2, do, cq, ck, 0.7, True)
    for x, y in zip(g, g2):
        np.testing.assert_array_equal(x[:5], y[:5])
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b:b + 2].tolist() + ck[b:b + 2].tolist()
        if q1 == q0 or k1 == k0:
            continue
        for h in range(H):
            ref = attention_backward_one_head(q[q0:q1, h], k[k0:k1, h], v[k0:k1, h],
                                              do[q0:q1, h], 0.7, True)
            for x, y in zip((g[0][q0:q1, h], g[1][k0:k1, h], g[2][k0:k1, h]), ref):
                np.testing.assert_array_equal(x, y)


def test_varlen_matches_torch_autograd_on_a_ragged_batch():
    """The packed gradients equal torch autograd through a block-diagonal masked SDPA."""
    r = _rng(33)
    H, D = 2, 4
    cq = np.array([0, 3, 9, 10], dtype=np.int32)
    ck = np.array([0, 5, 9, 13], dtype=np.int32)
    q, do = r.normal(size=(10, H, D)), r.normal(size=(10, H, D))
    k, v = r.normal(size=(13, H, D)), r.normal(size=(13, H, D))
    g = attention_backward_varlen(q, k, v, do, cq, ck, 0.5, True)
    mask = np.zeros((10, 13), dtype=bool)
    for b in range(3):
        for i in range(cq[b], cq[b + 1]):
            for j in range(ck[b], ck[b + 1]):
                mask[i, j] = (j - ck[b]) <= (i - cq[b])
    qt, kt, vt = (torch.tensor(x.transpose(1, 0, 2), requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt,
                                                         attn_mask=torch.from_numpy(mask),
                                                         scale=0.5)
    o.backward(torch.from_numpy(do.transpose(1, 0, 2)))
    for x, t in zip(g, (qt, kt, vt)):
        np.testing.assert_allclose(x, t.grad.numpy().transpose(1, 0, 2), rtol=0, atol=1e-12)


# ------------------------------------------------------------- sampled outputs
@pytest.mark.parametrize("causal,Sq,Sk", [(True, 37, 37), (False, 29, 41), (True, 30, 45),
                                          (False, 40, 23)])
def test_sampled_backward_equals_the_full_backward(causal, Sq, Sk):
    """dQ at sampled rows and dK, dV at sampled keys from the needed score rows only equal
    the full backward at those rows and keys."""
    r = _rng(41 + Sq)
    D = 5
    q, do = r.normal(size=(Sq, D)), r.normal(size=(Sq, D + 1))
    k, v = r.normal(size=(Sk, D)), r.normal(size=(Sk, D + 1))
    full = attention_backward_one_head(q, k, v, do, 0.45, causal)
    q_rows = np.array([0, 3, Sq // 2, Sq - 1])
    k_rows = np.array([Sk - 1, Sk - 5, Sk // 3])
    dq, dk, dv = attention_backward_sampled(q, k, v, do, 0.45, causal, q_rows, k_rows)
    np.testing.assert_allclose(dq, full[0][q_rows], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, full[1][k_rows], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, full[2][k_rows], rtol=0, atol=1e-12)


def test_sampled_backward_reads_only_the_rows_it_needs():
    """Causal, keys at the end: changing queries (and their dO) that see none of the sampled
    keys and are not sampled themselves leaves the sampled outputs unchanged."""
    r = _rng(47)
    S, D = 60, 4
    q, k, v, do = (r.normal(size=(S, D)) for _ in range(4))
    q_rows, k_rows = np.array([2, 5]), np.array([55, 58])
    a = attention_backward_sampled(q, k, v, do, 0.6, True, q_rows, k_rows)
    q2, do2 = q.copy(), do.copy()
    q2[10:50] += 3.0   # rows 10..49 see no key >= 55 and are not sampled
    do2[10:50] -= 1.0
    b = attention_backward_sampled(q2, k, v, do2, 0.6, True, q_rows, k_rows)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


# ------------------------------------------------- the caller's forward output
def test_row_term_from_the_exact_output_is_the_gradient():
    """rowsum(dP * P) = rowsum(dO * O) for the exact O, so handing the oracle's own
    forward output as the caller's O reproduces the autograd-pinned gradient."""
    for seed, (Sq, Sk, D, causal) in enumerate([(9, 9, 5, True), (6, 11, 3, False),
                                                (12, 12, 8, True)]):
        r = _rng(40 + seed)
        q, k, v = r.normal(size=(Sq, D)), r.normal(size=(Sk, D)), r.normal(size=(Sk, D + 1))
        do = r.normal(size=(Sq, D + 1))
        o, _ = attention_one_head(q, k, v, 0.6, causal)
        ref = _torch_grads(q, k, v, do, 0.6, causal)
        got = attention_backward_one_head(q, k, v, do, 0.6, causal, o=o)
        for g, rr in zip(got, ref):
            np.testing.assert_allclose(g, rr, rtol=0, atol=1e-11)


def test_gradient_is_affine_in_the_callers_output_and_dv_ignores_it():
    """The caller's O enters only through the row term, linearly: equal steps in O give
    equal steps in dQ and dK, and dV does not depend on it."""
    r = _rng(50)
    Sq, Sk, D = 10, 13, 6
    q, k, v, do = r.normal(size=(Sq, D)), r.normal(size=(Sk, D)), r.normal(size=(Sk, D)), \
        r.normal(size=(Sq, D))
    o, _ = attention_one_head(q, k, v, 0.4, True)
    step = r.normal(size=o.shape) * 1e-2
    g0, g1, g2 = (attention_backward_one_head(q, k, v, do, 0.4, True, o=o + t * step)
                  for t in (0.0, 1.0, 2.0))
    for i in (0, 1):
        np.testing.assert_allclose(g2[i] - g1[i], g1[i] - g0[i], rtol=0, atol=1e-13)
        assert np.abs(g1[i] - g0[i]).max() > 1e-6  # the row term does move them
    np.testing.assert_array_equal(g0[2], g1[2])


def test_returned_terms_reproduce_the_gradients():
    """P and dS returned by the oracle are the terms of its own products."""
    r = _rng(60)
    Sq, Sk, D = 8, 8, 4
    q, k, v, do = (r.normal(size=(S, D)) for S in (Sq, Sk, Sk, Sq))
    dq, dk, dv, p, ds = attention_backward_one_head(q, k, v, do, 0.7, True, return_terms=True)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.triu(p, 1) == 0) and np.all(np.triu(ds, 1) == 0)  # causal: masked
    np.testing.assert_allclose(dq, 0.7 * ds @ k, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, 0.7 * ds.T @ q, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, p.T @ do, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ds.sum(axis=1), 0.0, rtol=0, atol=1e-12)  # softmax Jacobian rows


def test_dense_and_packed_wrappers_pass_the_callers_output():
    r = _rng(70)
    B, S, H, D = 2, 9, 2, 4
    q, k, v, do = (r.normal(size=(B, S, H, D)) for _ in range(4))
    o = r.normal(size=(B, S, H, D))
    dense = attention_backward_dense(q, k, v, do, 0.5, True, o=o)
    one = attention_backward_one_head(q[1, :, 1], k[1, :, 1], v[1, :, 1], do[1, :, 1], 0.5, True,
                                      o=o[1, :, 1])
    for a, b in zip(dense, one):
        np.testing.assert_array_equal(a[1, :, 1], b)
    cu = np.array([0, S, 2 * S], dtype=np.int32)
    flat = lambda x: x.reshape(B * S, H, D)  # noqa: E731
    packed = attention_backward_varlen(flat(q), flat(k), flat(v), flat(do), cu, cu, 0.5, True,
                                       o=flat(o))
    for a, b in zip(dense, packed):
        np.testing.assert_allclose(flat(a), b, rtol=0, atol=1e-13)


def test_sampled_backward_terms_are_the_full_terms_at_its_rows():
    r = _rng(80)
    Sq = Sk = 40
    D = 5
    q, k, v, do = (r.normal(size=(Sq, D)) for _ in range(4))
    dq, dk, dv, p, ds = attention_backward_one_head(q, k, v, do, 0.5, True, return_terms=True)
    o_full, _ = attention_one_head(q, k, v, 0.5, True)
    q_rows, k_rows = np.array([1, 17, 39]), np.array([30, 39])
    _, _, _, rows, p_s, ds_s, o_s = attention_backward_sampled(q, k, v, do, 0.5, True, q_rows,
                                                               k_rows, return_terms=True)
    assert set(q_rows) <= set(rows) and set(range(30, 40)) <= set(rows)
    np.testing.assert_allclose(p_s, p[rows], rtol=0, atol=1e-13)
    np.testing.assert_allclose(ds_s, ds[rows], rtol=0, atol=1e-13)
    np.testing.assert_allclose(o_s, o_full[rows], rtol=0, atol=1e-13)
