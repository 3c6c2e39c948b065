"""Pins of the oracle's decode (KV cache) and partial-merge functions (CPU only).

Decode: the Sq new queries are the last Sq positions of a sequence whose cache
holds L keys (page "长文本处理性能断层真相", §2.2, the KV cache that grows with
the sequence).  Merge: attention over a union of disjoint key sets rebuilt from
the per-set (O, LSE) pairs, the combine step of ring attention (same page,
§1).  Pins: the last rows of a full causal forward, torch fp64 SDPA with a
bottom-right causal mask, a one-key cache, the merge identity over random key
partitions (and against torch), closed forms for equal and empty parts, and
planted mistakes in both functions.
"""
import math

import numpy as np
import pytest
import torch

from oracle.sdpa_oracle import attention_decode, attention_dense, merge_partials


def _rng(seed):
    return np.random.default_rng(seed)


def _cache(seed, B, Sq, Sk, H, D):
    r = _rng(seed)
    return (r.normal(size=(B, Sq, H, D)), r.normal(size=(B, Sk, H, D)),
            r.normal(size=(B, Sk, H, D)))


def test_decode_is_the_last_rows_of_a_causal_forward():
    r = _rng(1)
    B, S, H, D, Sq = 2, 23, 2, 5, 4
    q, k, v = (r.normal(size=(B, S, H, D)) for _ in range(3))
    o_full, l_full = attention_dense(q, k, v, 0.4, True)
    o, lse = attention_decode(q[:, S - Sq:], k, v, None, 0.4, True)
    np.testing.assert_allclose(o, o_full[:, S - Sq:], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, l_full[:, :, S - Sq:], rtol=0, atol=1e-12)


def test_decode_matches_torch_bottom_right_causal():
    q, k, v = _cache(2, 3, 5, 40, 2, 6)
    lens = [40, 17, 5]
    o, lse = attention_decode(q, k, v, np.array(lens), 0.3, True)
    for b, L in enumerate(lens):
        for h in range(2):
            qt = torch.from_numpy(q[b, :, h])
            kt, vt = torch.from_numpy(k[b, :L, h]), torch.from_numpy(v[b, :L, h])
            mask = torch.arange(L)[None, :] <= (L - 5 + torch.arange(5))[:, None]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qt[None], kt[None], vt[None], attn_mask=mask[None], scale=0.3)[0]
            np.testing.assert_allclose(o[b, :, h], ref.numpy(), rtol=0, atol=1e-12)
            s = torch.where(mask, 0.3 * qt @ kt.T, torch.tensor(-math.inf, dtype=torch.float64))
            np.testing.assert_allclose(lse[b, h], torch.logsumexp(s, -1).numpy(), rtol=0,
                                       atol=1e-12)


def test_decode_non_causal_sees_the_whole_cache():
    q, k, v = _cache(3, 2, 3, 30, 1, 4)
    o, lse = attention_decode(q, k, v, np.array([30, 11]), 0.5, False)
    for b, L in enumerate((30, 11)):
        qt, kt, vt = (torch.from_numpy(x) for x in (q[b, :, 0], k[b, :L, 0], v[b, :L, 0]))
        ref = torch.nn.functional.scaled_dot_product_attention(qt[None], kt[None], vt[None],
                                                               scale=0.5)[0]
        np.testing.assert_allclose(o[b, :, 0], ref.numpy(), rtol=0, atol=1e-12)


def test_decode_short_and_empty_caches():
    q, k, v = _cache(4, 3, 4, 10, 2, 3)
    o, lse = attention_decode(q, k, v, np.array([1, 2, 0]), 0.7, True)
    # one key: only the last query has a non-negative position; it sees key 0
    np.testing.assert_allclose(o[0, 3], v[0, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, :, 3], 0.7 * np.einsum("hd,hd->h", q[0, 3], k[0, 0]),
                               rtol=0, atol=1e-12)
    assert np.all(o[0, :3] == 0) and np.all(np.isneginf(lse[0, :, :3]))
    assert np.all(o[1, :2] == 0) and np.all(np.isneginf(lse[1, :, :2]))
    assert np.all(o[2] == 0) and np.all(np.isneginf(lse[2]))


def _split_results(q, k, v, cuts, scale):
    """Non-causal attention of every query over each key slice [cuts[i], cuts[i+1])."""
    os_, ls_ = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        if b == a:
            os_.append(np.zeros(q.shape[:-1] + (v.shape[-1],)))
            ls_.append(np.full(q.shape[:-1], -np.inf))
            continue
        o, l = attention_dense(q[None], k[None, a:b], v[None, a:b], scale, False)
        os_.append(o[0])
        ls_.append(l[0].transpose(1, 0))
    return np.stack(os_), np.stack(ls_)


def test_merge_of_a_partition_equals_attention_over_all_keys():
    r = _rng(5)
    S, Sk, H, D = 6, 37, 2, 4
    q, k, v = r.normal(size=(S, H, D)), r.normal(size=(Sk, H, D)), r.normal(size=(Sk, H, D))
    o_all, l_all = attention_dense(q[None], k[None], v[None], 0.6, False)
    for cuts in ([0, 37], [0, 10, 37], [0, 1, 2, 20, 37], [0, 0, 15, 15, 37]):
        op, lp = _split_results(q, k, v, cuts, 0.6)
        o, lse = merge_partials(op, lp)
        np.testing.assert_allclose(o, o_all[0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, l_all[0].transpose(1, 0), rtol=0, atol=1e-12)


def test_merge_closed_forms():
    o = np.array([[[1.0, 2.0]], [[3.0, 6.0]]])          # two parts, one row
    l = np.array([[0.25], [0.25]])
    mo, ml = merge_partials(o, l)
    np.testing.assert_allclose(mo, [[2.0, 4.0]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(ml, [0.25 + math.log(2.0)], rtol=0, atol=1e-15)
    mo, ml = merge_partials(o, np.array([[-np.inf], [1.5]]))   # one empty part
    np.testing.assert_allclose(mo, [[3.0, 6.0]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(ml, [1.5], rtol=0, atol=1e-15)
    mo, ml = merge_partials(o, np.array([[-np.inf], [-np.inf]]))  # nothing visible
    assert np.all(mo == 0) and np.isneginf(ml).all()
    mo, ml = merge_partials(o, np.array([[700.0], [-700.0]]))  # no overflow
    np.testing.assert_allclose(mo, [[1.0, 2.0]], rtol=0, atol=1e-12)


def _merge_mutant(o_parts, lse_parts, bug):
    o, lp = np.asarray(o_parts, float), np.asarray(lse_parts, float)
    m = lp.max(axis=0)
    w = np.exp(lp - m[None])
    if bug == "no_renormalise":
        return (w[..., None] * o).sum(0), m + np.log(w.sum(0))
    if bug == "plain_mean":
        return o.mean(0), m + np.log(w.sum(0))
    if bug == "lse_max_only":
        return (w[..., None] * o).sum(0) / w.sum(0)[..., None], m
    if bug == "log2_weights":
        w2 = np.exp2(lp - m[None])
        return (w2[..., None] * o).sum(0) / w2.sum(0)[..., None], m + np.log(w2.sum(0))
    raise ValueError(bug)


@pytest.mark.parametrize("bug", ["no_renormalise", "plain_mean", "lse_max_only",
                                 "log2_weights"])
def test_merge_mutants_fail_the_partition_identity(bug):
    r = _rng(6)
    q, k, v = r.normal(size=(5, 1, 3)), r.normal(size=(20, 1, 3)), r.normal(size=(20, 1, 3))
    o_all, l_all = attention_dense(q[None], k[None], v[None], 0.9, False)
    op, lp = _split_results(q, k, v, [0, 7, 20], 0.9)
    o, lse = _merge_mutant(op, lp, bug)
    ok = np.allclose(o, o_all[0], atol=1e-9) and np.allclose(lse, l_all[0].T, atol=1e-9)
    assert not ok, f"the partition identity misses the planted mistake {bug!r}"
