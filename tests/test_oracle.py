"""Pins of the fp64 oracle against things other than itself (CPU only).

Each pin is written as a function of a single-head attention callable
``fn(q, k, v, scale, causal) -> (O, LSE)`` so the same pins can be run against
deliberately broken variants (test_oracle_mutants below) to show that a
plausible mistake in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle.sdpa_oracle import attention_dense, attention_one_head, attention_varlen
from scaled_dot_product_tcgen05_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
TOL = 1e-12


def _oracle(q, k, v, scale, causal):
    return attention_one_head(q, k, v, scale, causal)


def _rng(seed):
    return np.random.default_rng(seed)


def brute_force(q, k, v, scale, causal):
    """Pure-Python loops straight from the definition (tiny inputs only)."""
    Sq, D = q.shape
    Sk, Dv = v.shape
    O, L = [], []
    for i in range(Sq):
        s = []
        for j in range(Sk):
            if causal and j > i:
                continue
            s.append((j, scale * math.fsum(float(q[i, d]) * float(k[j, d]) for d in range(D))))
        if not s:
            O.append([0.0] * Dv)
            L.append(-math.inf)
            continue
        mx = max(x for _, x in s)
        w = [(j, math.exp(x - mx)) for j, x in s]
        z = math.fsum(e for _, e in w)
        O.append([math.fsum(e * float(v[j, c]) for j, e in w) / z for c in range(Dv)])
        L.append(mx + math.log(z))
    return np.array(O), np.array(L)


# ----------------------------------------------------------------------------- pins
def pin_bruteforce(fn):
    for seed, (Sq, Sk, D) in enumerate([(1, 1, 1), (3, 5, 2), (8, 8, 8), (5, 3, 4), (7, 7, 3),
                                        (6, 9, 5)]):
        r = _rng(seed)
        q, k, v = r.normal(size=(Sq, D)), r.normal(size=(Sk, D)), r.normal(size=(Sk, D + 1))
        for causal in (False, True):
            scale = 0.7
            o, l = fn(q, k, v, scale, causal)
            ob, lb = brute_force(q, k, v, scale, causal)
            assert np.allclose(o, ob, rtol=0, atol=TOL), ("bruteforce O", Sq, Sk, D, causal)
            assert np.allclose(l, lb, rtol=0, atol=TOL), ("bruteforce LSE", Sq, Sk, D, causal)


def pin_constant_v(fn):
    r = _rng(10)
    q, k = r.normal(size=(9, 4)), r.normal(size=(9, 4))
    c = r.normal(size=(3,))
    v = np.tile(c, (9, 1))
    for causal in (False, True):
        o, _ = fn(q, k, v, 0.5, causal)
        assert np.allclose(o, np.tile(c, (9, 1)), rtol=0, atol=1e-14), "constant V"


def pin_causal_first_row(fn):
    r = _rng(11)
    q, k, v = r.normal(size=(6, 5)), r.normal(size=(6, 5)), r.normal(size=(6, 5))
    scale = 0.9
    o, l = fn(q, k, v, scale, True)
    assert np.allclose(o[0], v[0], rtol=0, atol=1e-15), "causal row 0 = V[0]"
    assert abs(l[0] - scale * float(q[0] @ k[0])) <= 1e-14, "causal LSE_0 = s_00"


def pin_shift_invariance(fn):
    # K has a constant column kappa, so adding delta_i to Q[i, dstar] adds
    # scale*delta_i*kappa to every score of row i: O unchanged, LSE shifted.
    r = _rng(12)
    Sq, Sk, D, dstar, kappa, scale = 7, 7, 4, 2, 1.5, 0.8
    q, k, v = r.normal(size=(Sq, D)), r.normal(size=(Sk, D)), r.normal(size=(Sk, 3))
    k[:, dstar] = kappa
    delta = r.normal(size=(Sq,)) * 3.0
    q2 = q.copy()
    q2[:, dstar] += delta
    for causal in (False, True):
        o1, l1 = fn(q, k, v, scale, causal)
        o2, l2 = fn(q2, k, v, scale, causal)
        assert np.allclose(o1, o2, rtol=0, atol=1e-12), "shift: O"
        assert np.allclose(l2 - l1, scale * delta * kappa, rtol=0, atol=1e-12), "shift: LSE"


def pin_single_key(fn):
    r = _rng(13)
    q, k, v = r.normal(size=(5, 3)), r.normal(size=(1, 3)), r.normal(size=(1, 4))
    o, l = fn(q, k, v, 1.3, False)
    assert np.allclose(o, np.tile(v[0], (5, 1)), rtol=0, atol=1e-15), "Sk=1 O"
    assert np.allclose(l, 1.3 * (q @ k[0]), rtol=0, atol=1e-14), "Sk=1 LSE"


def pin_two_keys(fn):
    r = _rng(14)
    q, k, v = r.normal(size=(4, 3)), r.normal(size=(2, 3)), r.normal(size=(2, 2))
    scale = 0.6
    o, l = fn(q, k, v, scale, False)
    s0, s1 = scale * (q @ k[0]), scale * (q @ k[1])
    sig = 1.0 / (1.0 + np.exp(s1 - s0))             # weight of key 0
    exp_o = sig[:, None] * v[0] + (1 - sig)[:, None] * v[1]
    assert np.allclose(o, exp_o, rtol=0, atol=1e-14), "Sk=2 O"
    assert np.allclose(l, np.logaddexp(s0, s1), rtol=0, atol=1e-14), "Sk=2 LSE"


def pin_zero_scale(fn):
    r = _rng(15)
    q, k, v = r.normal(size=(6, 3)), r.normal(size=(6, 3)), r.normal(size=(6, 2))
    o, l = fn(q, k, v, 0.0, True)
    for i in range(6):
        assert np.allclose(o[i], v[: i + 1].mean(axis=0), rtol=0, atol=1e-14), "scale 0 O"
        assert abs(l[i] - math.log(i + 1)) <= 1e-14, "scale 0 LSE"
    o, l = fn(q, k, v, 0.0, False)
    assert np.allclose(o, np.tile(v.mean(axis=0), (6, 1)), rtol=0, atol=1e-14)
    assert np.allclose(l, math.log(6), rtol=0, atol=1e-14)


def pin_key_permutation(fn):
    r = _rng(16)
    q, k, v = r.normal(size=(5, 4)), r.normal(size=(8, 4)), r.normal(size=(8, 3))
    perm = r.permutation(8)
    o1, l1 = fn(q, k, v, 0.7, False)
    o2, l2 = fn(q, k[perm], v[perm], 0.7, False)
    assert np.allclose(o1, o2, rtol=0, atol=1e-13) and np.allclose(l1, l2, rtol=0, atol=1e-13)


def pin_causal_prefix(fn):
    r = _rng(17)
    q, k, v = r.normal(size=(7, 4)), r.normal(size=(7, 4)), r.normal(size=(7, 3))
    o, l = fn(q, k, v, 0.9, True)
    for i in range(7):
        oi, li = fn(q[i:i + 1], k[: i + 1], v[: i + 1], 0.9, False)
        assert np.allclose(o[i], oi[0], rtol=0, atol=1e-14), "causal prefix O"
        assert abs(l[i] - li[0]) <= 1e-14, "causal prefix LSE"


def pin_torch_sdpa(fn):
    """Library cross-check: torch's own SDPA and logsumexp on the CPU in fp64."""
    r = _rng(18)
    for (Sq, Sk, D, causal) in [(16, 16, 8, False), (16, 16, 8, True), (9, 13, 5, False),
                                (13, 9, 5, True)]:
        q, k, v = r.normal(size=(Sq, D)), r.normal(size=(Sk, D)), r.normal(size=(Sk, D))
        scale = 1 / math.sqrt(D)
        o, l = fn(q, k, v, scale, causal)
        tq, tk, tv = (torch.from_numpy(x)[None, None] for x in (q, k, v))
        ot = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                              scale=scale)[0, 0].numpy()
        s = scale * torch.from_numpy(q) @ torch.from_numpy(k).T
        if causal:
            s = s.masked_fill(torch.ones(Sq, Sk, dtype=torch.bool).triu(1), -math.inf)
        lt = torch.logsumexp(s, dim=-1).numpy()
        assert np.allclose(o, ot, rtol=0, atol=1e-12), ("torch sdpa O", Sq, Sk, causal)
        assert np.allclose(l, lt, rtol=0, atol=1e-12), ("torch logsumexp", Sq, Sk, causal)


def pin_golden(fn):
    g = json.load(open(GOLDEN))
    for key in ("two_key_example", "causal_three_rows"):
        e = g[key]
        q, k, v = (np.array(e[n], dtype=np.float64) for n in ("q", "k", "v"))
        o, l = fn(q, k, v, e["scale"], key == "causal_three_rows")
        assert np.allclose(o, np.array(e["o"]), rtol=0, atol=1e-12), key
        assert np.allclose(l, np.array(e["lse"]), rtol=0, atol=1e-12), key


PINS = [pin_bruteforce, pin_constant_v, pin_causal_first_row, pin_shift_invariance,
        pin_single_key, pin_two_keys, pin_zero_scale, pin_key_permutation, pin_causal_prefix,
        pin_torch_sdpa, pin_golden]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(_oracle)


def test_rows_of_p_sum_to_one():
    r = _rng(19)
    q, k, v = r.normal(size=(12, 6)), r.normal(size=(15, 6)), r.normal(size=(15, 6))
    for causal in (False, True):
        _, _, p = attention_one_head(q, k, v, 0.4, causal, return_p=True)
        assert np.all(np.abs(p.sum(axis=1) - 1.0) <= 1e-12)
        assert np.all(p >= 0)
        if causal:
            assert np.all(p[np.triu_indices(12, 1, 15)] == 0.0)


def test_empty_key_rows():
    q = np.ones((3, 2))
    o, l = attention_one_head(q, np.zeros((0, 2)), np.zeros((0, 2)), 1.0, False)
    assert np.all(o == 0) and np.all(np.isneginf(l))


# ------------------------------------------------------------------- batch wrappers
def test_dense_layout_matches_torch():
    """attention_dense on [B,S,H,D] vs torch SDPA on the [B,H,S,D] permutation."""
    g = torch.Generator().manual_seed(5)
    B, S, H, D = 2, 11, 3, 4
    q, k, v = (torch.randn(B, S, H, D, generator=g, dtype=torch.float64) for _ in range(3))
    for causal in (False, True):
        o, l = attention_dense(q, k, v, 0.5, causal)
        ot = torch.nn.functional.scaled_dot_product_attention(
            q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2), is_causal=causal,
            scale=0.5).transpose(1, 2).numpy()
        s = 0.5 * q.transpose(1, 2) @ k.transpose(1, 2).transpose(-1, -2)
        if causal:
            s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), -math.inf)
        assert np.allclose(o, ot, rtol=0, atol=1e-12)
        assert np.allclose(l, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def test_dense_subset_equals_full():
    g = torch.Generator().manual_seed(6)
    q, k, v = (torch.randn(1, 20, 4, 8, generator=g, dtype=torch.float64) for _ in range(3))
    o, l = attention_dense(q, k, v, 0.3, True)
    os_, ls = attention_dense(q, k, v, 0.3, True, heads=[1, 3], rows=[0, 7, 19])
    for h in (1, 3):
        for i in (0, 7, 19):
            assert np.array_equal(os_[0, i, h], o[0, i, h]) and ls[0, h, i] == l[0, h, i]
    assert np.isnan(os_[0, 1, 1]).all() and np.isnan(os_[0, 0, 0]).all()


def _varlen_case(seed, lens_q, lens_k, H=2, D=4):
    g = torch.Generator().manual_seed(seed)
    cq = W.cu_seqlens_from_lengths(lens_q)
    ck = W.cu_seqlens_from_lengths(lens_k)
    q = torch.randn(int(cq[-1]), H, D, generator=g, dtype=torch.float64)
    k = torch.randn(int(ck[-1]), H, D, generator=g, dtype=torch.float64)
    v = torch.randn(int(ck[-1]), H, D, generator=g, dtype=torch.float64)
    return q, k, v, cq, ck


def test_varlen_equals_dense_per_sequence():
    lens = [5, 1, 9, 3]
    q, k, v, cq, ck = _varlen_case(7, lens, lens)
    for causal in (False, True):
        o, l = attention_varlen(q, k, v, cq, ck, 0.6, causal)
        for b, L in enumerate(lens):
            a, e = int(cq[b]), int(cq[b + 1])
            od, ld = attention_dense(q[None, a:e], k[None, a:e], v[None, a:e], 0.6, causal)
            assert np.array_equal(o[a:e], od[0]) and np.array_equal(l[:, a:e], ld[0])


def test_varlen_no_cross_sequence_leak():
    """Changing sequence 0's keys must not change any other sequence's output."""
    lens = [6, 4, 7]
    q, k, v, cq, ck = _varlen_case(8, lens, lens)
    o1, l1 = attention_varlen(q, k, v, cq, ck, 0.5, False)
    k2, v2 = k.clone(), v.clone()
    k2[:6] += 3.0
    v2[:6] -= 2.0
    o2, l2 = attention_varlen(q, k2, v2, cq, ck, 0.5, False)
    assert np.array_equal(o1[6:], o2[6:]) and np.array_equal(l1[:, 6:], l2[:, 6:])
    assert not np.allclose(o1[:6], o2[:6])


def test_varlen_sequence_permutation():
    lens = [3, 7, 2]
    q, k, v, cq, ck = _varlen_case(9, lens, lens)
    o, l = attention_varlen(q, k, v, cq, ck, 0.5, True)
    order = [2, 0, 1]
    segs = [(int(cq[b]), int(cq[b + 1])) for b in range(3)]
    idx = torch.cat([torch.arange(*segs[b]) for b in order])
    cp = W.cu_seqlens_from_lengths([lens[b] for b in order])
    o2, l2 = attention_varlen(q[idx], k[idx], v[idx], cp, cp, 0.5, True)
    assert np.array_equal(o2, o[idx.numpy()]) and np.array_equal(l2, l[:, idx.numpy()])


def test_varlen_empty_sequences():
    q, k, v, cq, ck = _varlen_case(10, [3, 0, 2], [3, 0, 0])
    o, l = attention_varlen(q, k, v, cq, ck, 0.5, True)
    assert np.all(o[3:5] == 0) and np.all(np.isneginf(l[:, 3:5]))
    assert np.all(np.isfinite(o[:3]))


# ------------------------------------------------------------------- FLOP accounting
def test_flop_formula_matches_pages_worked_example():
    e = json.load(open(GOLDEN))["roofline_worked_example"]
    f = W.attention_flops(1, 1, e["seq_len"], e["seq_len"], e["head_dim"], causal=False)
    assert f == 4 * 2048 ** 2 * 64
    assert round(f / 1e9, 2) == round(e["flops_printed"] / 1e9, 2)
    assert e["seq_len"] * e["head_dim"] * 2 * 3 == e["bytes_printed"]
    # the page divides its rounded 1.07e9 by the bytes: 1360.6 -> "1360"
    assert abs(e["flops_printed"] / e["bytes_printed"] - e["intensity_printed"]) < 1.0
    assert abs(f / e["bytes_printed"] / e["intensity_printed"] - 1) < 0.005
    assert W.attention_flops(2, 3, 64, 64, 64, causal=True) == 2 * 3 * 4 * 64 * 64 * 64 / 2
    assert W.varlen_flops([64, 32], 2, 64, True) == (W.attention_flops(1, 2, 64, 64, 64, True)
                                                     + W.attention_flops(1, 2, 32, 32, 64, True))


# ------------------------------------------------------------------- input generator
def test_inputs_are_seeded_and_headwise():
    wl = W.standard_workloads()["tiny_causal"]
    a = W.make_inputs(wl)
    b = W.make_inputs(wl)
    c = W.make_inputs(wl, heads=[1])
    assert torch.equal(a["q"], b["q"]) and a["q"].dtype == torch.float16
    assert torch.equal(a["k"][:, :, 1], c["k"][:, :, 1])
    assert torch.count_nonzero(c["k"][:, :, 0]) == 0
    vl = W.standard_workloads()["varlen_causal"]
    lens = W.varlen_lengths(vl)
    assert len(lens) == 16 and int(lens.min()) >= 128 and int(lens.max()) <= 4096
    heads, rows = W.sampled_heads_rows(W.standard_workloads()["long64k_causal"])
    assert len(heads) == 4 and len(rows) == 256 and rows[0] == 0 and rows[-1] == 65535
