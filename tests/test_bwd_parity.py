"""GPU parity of the attention backward against the fp64 oracle.

The backward (page "Multi-Head Attention的计算本质与性能瓶颈", §3.3: a reserved
backward interface; masked connections carry no gradient) takes Q, K, V, O,
dO and the forward's LSE.  Here O and LSE come from attn_fwd on the GPU, and
the oracle's gradients from the exact fp64 definition.

Tolerance (from the arithmetic), per gradient:
  * mean |err| <= 1e-2 of the RMS of the reference gradient.  The kernel
    rounds P and dS to the input dtype (relative u = 2^-9 for bf16, 2^-11 for
    fp16) before the products that consume them and rounds dQ, dK, dV on
    output; every other step is fp32.  A gradient entry sums many such terms
    with random signs, so its mean error is about u of its RMS (0.002 for
    bf16): 5x margin.
  * max |err| <= 0.15 (bf16), 0.06 (fp16) of max(the RMS of the reference
    gradient, the RMS of the same row of the reference).  Each entry's error
    is a relative rounding error of its own row's terms (P and dS rounded, D =
    rowsum(dO * O) from the 16-bit O the forward returned, the method's input,
    which is off by up to u * |dO| |O|), so it scales with the row: in rows
    whose softmax is nearly one-hot dP - D nearly cancels and the error of D
    reaches dS unattenuated (dQ_i up to scale * dD * max|K|, 0.05-0.09 of the
    RMS observed on the causal cases), and the first rows of each causal
    sequence, where attention rests on a few keys, carry gradients far above
    the tensor's RMS and errors in proportion (packed batches, with one such
    start per sequence, reached 0.20 of the tensor RMS and stay within 0.15 of
    their own rows').  The row scale falls back to the tensor RMS where a
    row's exact gradient is near zero (a one-hot row's dQ).
"""
import math
import warnings

import numpy as np
import pytest
import torch

import scaled_dot_product_tcgen05_gb300 as pkg
from oracle.sdpa_oracle import attention_backward_dense, attention_backward_varlen

pytestmark = pytest.mark.gpu

BF, FP = torch.bfloat16, torch.float16
DEV = "cuda:0"
MEAN_REL = 1e-2
MAX_REL = {torch.bfloat16: 0.15, torch.float16: 0.06}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkg.load_library()


def _case(seed, B, H, Sq, Sk, D, dt):
    g = torch.Generator().manual_seed(seed)
    mk = lambda S: torch.randn(B, S, H, D, generator=g).to(dt)  # noqa: E731
    return mk(Sq), mk(Sk), mk(Sk), mk(Sq)


def compare_grads(got, ref, what):
    stats = {}
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        with np.errstate(invalid="ignore"):  # unwritten rows (keys of no sequence) may be NaN
            gg = g.float().cpu().numpy().astype(np.float64)
        sel = ~np.isnan(r)
        assert np.all(np.isfinite(gg[sel])), f"{what}: non-finite {name}"
        rms = max(float(np.sqrt(np.mean(r[sel] ** 2))), 1e-30)
        with warnings.catch_warnings():  # rows of no sequence are all NaN
            warnings.simplefilter("ignore", RuntimeWarning)
            row_rms = np.sqrt(np.nanmean(r ** 2, axis=-1, keepdims=True)) * np.ones_like(r)
        d = np.abs(gg[sel] - r[sel])
        scale_row = np.maximum(rms, np.nan_to_num(row_rms[sel]))
        stats[name] = (float(d.mean() / rms), float((d / scale_row).max()), float(d.max() / rms))
        bound = MAX_REL[g.dtype]
        assert stats[name][0] <= MEAN_REL and stats[name][1] <= bound, f"{what}: {name} {stats}"
    print(what, stats)
    return stats


def _run(q, k, v, do, causal, scale):
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = pkg.attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = pkg.attn_bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale)
    st = pkg.attn_check()
    assert st == pkg.ATTN_OK, pkg.status_string(st)
    return dq, dk, dv


CASES = [
    # (B, H, Sq, Sk, D, dtype, causal)
    (1, 2, 256, 256, 128, BF, True),
    (1, 2, 256, 256, 128, BF, False),
    (2, 2, 300, 300, 64, FP, True),
    (1, 3, 128, 384, 128, BF, False),
    (1, 2, 400, 200, 64, BF, False),
    (2, 1, 129, 129, 128, FP, False),
    (1, 2, 200, 300, 128, BF, True),     # keys 200.. seen by no query: zero dK, dV
    (1, 2, 300, 200, 64, FP, True),
    (1, 1, 1, 1, 64, BF, True),
    (1, 4, 1024, 1024, 128, BF, True),
    (2, 2, 777, 777, 64, BF, True),
]


def _id(c):
    return "B{}H{}q{}k{}D{}{}{}".format(c[0], c[1], c[2], c[3], c[4],
                                        "bf" if c[5] == BF else "fp", "c" if c[6] else "")


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_bwd_parity(case):
    B, H, Sq, Sk, D, dt, causal = case
    q, k, v, do = _case(Sq * 5 + Sk + D, B, H, Sq, Sk, D, dt)
    scale = 1.0 / math.sqrt(D)
    got = _run(q, k, v, do, causal, scale)
    ref = attention_backward_dense(q, k, v, do, scale, causal)
    compare_grads(got, ref, _id(case))
    if causal and Sk > Sq:  # keys no query sees get exactly zero gradient
        assert torch.all(got[1][:, Sq:] == 0) and torch.all(got[2][:, Sq:] == 0)


def test_bwd_peaked_scores():
    """Q, K ~ N(0, 16): a peaked softmax stresses P = exp(S - LSE) recomputation."""
    g = torch.Generator().manual_seed(77)
    B, H, S, D = 1, 2, 512, 128
    q = (torch.randn(B, S, H, D, generator=g) * 4).to(BF)
    k = (torch.randn(B, S, H, D, generator=g) * 4).to(BF)
    v = torch.randn(B, S, H, D, generator=g).to(BF)
    do = torch.randn(B, S, H, D, generator=g).to(BF)
    got = _run(q, k, v, do, True, 1 / math.sqrt(D))
    ref = attention_backward_dense(q, k, v, do, 1 / math.sqrt(D), True)
    compare_grads(got, ref, "peaked")


def test_bwd_dk_dv_deterministic():
    q, k, v, do = _case(3, 1, 2, 600, 600, 128, BF)
    a = _run(q, k, v, do, True, 0.09)
    b = _run(q, k, v, do, True, 0.09)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert torch.allclose(a[0].float(), b[0].float(), atol=1e-2, rtol=0)


# ------------------------------------------------------------ packed sequences
def _packed_case(seed, lens_q, lens_k, H, D, dt, lead=0, tail=0):
    """Packed batch with ``lead`` rows before and ``tail`` rows after the sequences
    (rows of no sequence, finite values)."""
    g = torch.Generator().manual_seed(seed)
    cq = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32) + lead
    ck = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32) + lead
    Tq, Tk = int(cq[-1]) + tail, int(ck[-1]) + tail
    mk = lambda T: torch.randn(T, H, D, generator=g).to(dt)  # noqa: E731
    return mk(Tq), mk(Tk), mk(Tk), mk(Tq), cq, ck


def _run_packed(q, k, v, do, cq, ck, causal, scale, poison_outside=True):
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    cqd, ckd = (torch.from_numpy(c).to(DEV) for c in (cq, ck))
    o, lse = pkg.attn_fwd(qd, kd, vd, causal=causal, scale=scale, cu_seqlens_q=cqd,
                          cu_seqlens_k=ckd)
    if poison_outside:  # the forward leaves these rows unwritten: anything may be there
        for sl in (slice(0, int(cq[0])), slice(int(cq[-1]), q.shape[0])):
            o[sl] = float("nan")
            lse[:, sl] = float("nan")
    dq, dk, dv = pkg.attn_bwd(qd, kd, vd, o, dod, lse, causal=causal, scale=scale,
                              cu_seqlens_q=cqd, cu_seqlens_k=ckd)
    st = pkg.attn_check()
    assert st == pkg.ATTN_OK, pkg.status_string(st)
    return dq, dk, dv


VARLEN_CASES = [
    # (lens_q, lens_k, H, D, dtype, causal, lead, tail)
    ([300, 0, 129, 1, 700], [300, 50, 129, 1, 700], 2, 128, BF, True, 0, 0),
    ([200, 513, 64], [333, 100, 64], 2, 64, FP, False, 0, 0),
    ([128, 256], [128, 256], 2, 128, BF, True, 0, 0),
    ([37, 90, 200], [37, 0, 150], 2, 128, BF, True, 0, 0),      # a sequence without keys
    ([150, 300], [170, 260], 2, 64, BF, True, 20, 33),         # rows of no sequence
    ([1000, 3, 517], [1000, 400, 517], 1, 128, FP, False, 5, 0),
]


def _vid(c):
    return "q{}k{}H{}D{}{}{}l{}t{}".format("-".join(map(str, c[0])), "-".join(map(str, c[1])),
                                          c[2], c[3], "bf" if c[4] == BF else "fp",
                                          "c" if c[5] else "", c[6], c[7])


@pytest.mark.parametrize("case", VARLEN_CASES, ids=_vid)
def test_bwd_varlen_parity(case):
    lens_q, lens_k, H, D, dt, causal, lead, tail = case
    q, k, v, do, cq, ck = _packed_case(sum(lens_q) + 7 * sum(lens_k), lens_q, lens_k, H, D, dt,
                                       lead, tail)
    scale = 1.0 / math.sqrt(D)
    got = _run_packed(q, k, v, do, cq, ck, causal, scale)
    ref = attention_backward_varlen(q, k, v, do, cq, ck, scale, causal)
    compare_grads(got, ref, _vid(case))
    dq = got[0].float().cpu()
    assert torch.all(dq[:int(cq[0])] == 0) and torch.all(dq[int(cq[-1]):] == 0)
    for b in range(len(lens_q)):  # keys no query sees: exactly zero
        k0, k1 = int(ck[b]), int(ck[b + 1])
        unseen = k0 + (min(lens_q[b], lens_k[b]) if causal else (lens_k[b] if lens_q[b] else 0))
        if unseen < k1:
            assert torch.all(got[1][unseen:k1] == 0) and torch.all(got[2][unseen:k1] == 0)


def test_bwd_varlen_equal_lengths_match_dense():
    """Sequences of one length packed back to back, with the same O and LSE, give the
    dense call's dK, dV bit for bit (dQ's fp32 reduce-adds may land in another order)."""
    B, S, H, D = 3, 333, 2, 128
    q, k, v, do = (t.to(DEV) for t in _case(91, B, H, S, S, D, BF))
    scale = 1.0 / math.sqrt(D)
    o, lse = pkg.attn_fwd(q, k, v, causal=True, scale=scale)
    dense = pkg.attn_bwd(q, k, v, o, do, lse, causal=True, scale=scale)
    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device=DEV)
    flat = lambda t: t.reshape(B * S, H, D)  # noqa: E731
    packed = pkg.attn_bwd(flat(q), flat(k), flat(v), flat(o), flat(do),
                          lse.permute(1, 0, 2).reshape(H, B * S).contiguous(), causal=True,
                          scale=scale, cu_seqlens_q=cu, cu_seqlens_k=cu)
    st = pkg.attn_check()
    assert st == pkg.ATTN_OK, pkg.status_string(st)
    assert torch.equal(flat(dense[1]), packed[1]) and torch.equal(flat(dense[2]), packed[2])
    assert torch.allclose(flat(dense[0]).float(), packed[0].float(), atol=1e-2, rtol=0)


def test_bwd_varlen_malformed_bounds_are_reported():
    """Decreasing sequence bounds: the call does no work and attn_check reports them."""
    q, k, v, do, cq, ck = _packed_case(5, [200, 100], [200, 100], 2, 128, BF)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    good_q, good_k = (torch.from_numpy(c).to(DEV) for c in (cq, ck))
    o, lse = pkg.attn_fwd(qd, kd, vd, causal=True, cu_seqlens_q=good_q, cu_seqlens_k=good_k)
    assert pkg.attn_check() == pkg.ATTN_OK
    bad_q = torch.tensor([0, 250, 200], dtype=torch.int32, device=DEV)
    pkg.attn_bwd(qd, kd, vd, o, dod, lse, causal=True, cu_seqlens_q=bad_q, cu_seqlens_k=good_k)
    assert pkg.attn_check() == pkg.ATTN_ERR_BAD_SEQLENS
    assert pkg.attn_check() == pkg.ATTN_OK  # the error word was cleared


def test_bwd_many_units_per_cta_dense():
    """16 heads x 16 key tiles = 256 units on at most 152 CTAs: every CTA runs several
    units, so K/V reloads, accumulator hand-over and barrier phases cross unit bounds."""
    B, H, S, D = 1, 16, 2048, 128
    q, k, v, do = _case(123, B, H, S, S, D, BF)
    scale = 1.0 / math.sqrt(D)
    got = _run(q, k, v, do, True, scale)
    heads = [0, 7, 15]
    ref = attention_backward_dense(q, k, v, do, scale, True, heads=heads)
    compare_grads([g[:, :, heads] for g in got], [r[:, :, heads] for r in ref], "dense 256 units")


def test_bwd_many_units_per_cta_packed():
    """A packed batch of 9000 tokens over 8 heads (about 600 units): the sequence walk,
    per-sequence tile offsets and dQ rows across sequences with several units per CTA."""
    lens = [3000, 17, 2500, 1, 3482]
    H, D = 8, 128
    q, k, v, do, cq, ck = _packed_case(77, lens, lens, H, D, BF, lead=3, tail=5)
    scale = 1.0 / math.sqrt(D)
    got = _run_packed(q, k, v, do, cq, ck, True, scale)
    heads = [1, 6]
    ref = attention_backward_varlen(q, k, v, do, cq, ck, scale, True, heads=heads)
    compare_grads([g[:, heads] for g in got], [r[:, heads] for r in ref], "packed 600 units")


def test_bwd_full_size_sampled():
    """The benchmarked problem (B=1 H=32 S=16384 D=128 bf16 causal) in the bench's launch
    configuration: dQ at seeded query rows and dK, dV at the last keys of two heads, from
    the oracle's sampled backward."""
    from oracle.sdpa_oracle import attention_backward_sampled
    from scaled_dot_product_tcgen05_gb300 import workloads as W
    wl = W.standard_workloads()["bwd16k_causal"]
    inp = W.make_inputs(wl)
    q, k, v, do = inp["q"], inp["k"], inp["v"], inp["do"]
    got = _run(q, k, v, do, True, wl.scale)
    S = wl.Sq
    rng = np.random.default_rng(16384)
    q_rows = np.union1d(rng.choice(S, 24, replace=False), [0, 1, 127, 128, 8191, S - 1])
    k_rows = np.union1d(np.arange(S - 64, S), [S - 129, S - 1000])
    for h in (0, 17):
        ref = attention_backward_sampled(q[0, :, h], k[0, :, h], v[0, :, h], do[0, :, h],
                                         wl.scale, True, q_rows, k_rows)
        sub = [got[0][0, q_rows, h], got[1][0, k_rows, h], got[2][0, k_rows, h]]
        compare_grads(sub, list(ref), f"bwd16k head {h}")
