"""GPU parity of the attention backward against the fp64 oracle.

The backward (page "Multi-Head Attention的计算本质与性能瓶颈", §3.3: a reserved
backward interface; masked connections carry no gradient) takes Q, K, V, the
forward's O and LSE, and dO.  In the parity cases O and LSE are the oracle's
forward rounded to what a forward hands over (O in the input dtype, LSE in
fp32), built on the host; the reference is the oracle's gradient computed from
that same O (its row term rowsum(dO * O) uses the O the backward is given).

Tolerance, derived a priori from where the kernel rounds (nothing is fitted
to observed errors).  The kernel rounds P to the input dtype (P~) before
dV = P~^T dO, forms dS = P~ (dP - D) from that rounded P~ and rounds it before
dQ = scale dS K and dK = scale dS^T Q, and rounds every output; everything else
is fp32 (exact 16-bit products, fp32 accumulation).  A rounded
value x carries an error of at most u|x| (u = 2^-8 bf16, 2^-11 fp16) plus eta
(half the spacing of the subnormals, 2^-25 for fp16), and a value below the
smallest normal (2^-14 for fp16) may be lost altogether (an error of |x|: the
tensor cores may flush such operands).  So, per element, to first order:
  |err dQ_id| <= scale sum_j e_S(i, j) |K_jd| + u |dQ_id| + eta
  |err dK_jd| <= scale sum_i e_S(i, j) |Q_id| + u |dK_jd| + eta
  |err dV_jd| <=       sum_i e(P_ij) |dO_id| + u |dV_jd| + eta
with e_S(i, j) = e(dS_ij) + |dP_ij - D_i| e(P_ij) (the rounding of dS and that
of the P~ it is formed from),
and e(x) = (u + gamma + rho_ij) |x| + eta on visible entries, gamma = n 2^-24
for the fp32 accumulation of n terms and rho_ij = delta + g scale sum_d
|Q_id| |K_jd| the relative error of the recomputed P (g = 2 D 2^-24 for an
fp32 dot product over the head dim, whose error lands in the exponent;
delta = 2^-16 for ex2.approx and the split bias terms); dS also carries
P_ij g (sum_d |dO_id| |V_jd| + sum_d |dO_id| |O_id|), the fp32 error of
dP - D (it dominates where dS is exactly 0, as in a causal row 0).  Checks:
  * every element: |err| <= 2 W (2: room for second-order terms);
  * every row of 128 (or 64) elements: R = sqrt(mean (err / sigma)^2) <= 2.5,
    where sigma is the standard deviation of the same sum of independent
    roundings (an error uniform in [-u|x|, u|x|] has variance u^2 x^2 / 3);
    possibly lost subnormal terms are functions of the data, not independent
    roundings, and enter sigma as if they all added up.
    R is about 1 when many roundings add up; a row whose error comes from one
    rounded term and the output rounding reaches at most sqrt(6) = 2.45 (each
    error at its maximum, sqrt(3) sigma), hence the 2.5;
  * every row: t = |sum_d err_d ref_d| / (its standard deviation under the same
    model) <= 6.  A row error along the row itself (a scaled row) adds up
    coherently in t, the roundings do not: t is a sum of independent terms, at
    most sqrt(3 m) for a row of m rounded terms (<= 6 for m <= 12) and close to
    N(0, 1) when many terms add up (6 sigma beyond).  A 1 % error in one row of
    dQ, dK or dV gives t of 20 or more, so it fails.
At full size (the benchmarked 16K problem, O from the GPU forward), the error of
the forward's O enters D; it is bounded a priori by the forward's own rounding,
u (sum_j P_ij |V_jd| + 2 |O_id|) per element of O, and only the per-element
check applies there (that term is systematic within a row).
"""
import math

import numpy as np
import pytest
import torch

import scaled_dot_product_tcgen05_gb300 as pkg
from oracle.sdpa_oracle import (attention_backward_one_head, attention_dense,
                                attention_varlen)

pytestmark = pytest.mark.gpu

BF, FP = torch.bfloat16, torch.float16
DEV = "cuda:0"
U = {BF: 2.0 ** -8, FP: 2.0 ** -11}
ETA = {BF: 2.0 ** -134, FP: 2.0 ** -25}
TINY = {BF: 2.0 ** -126, FP: 2.0 ** -14}  # smallest normal value
DELTA = 2.0 ** -16
W_FACTOR = 2.0
R_MAX = 2.5
T_MAX = 6.0


def _f64(x):
    return x.double().cpu().numpy() if torch.is_tensor(x) else np.asarray(x, dtype=np.float64)


class GradBounds:
    """Reference gradients of one (sequence, head) with their a-priori bounds."""

    def __init__(self, q, k, v, do, scale, causal, dt, o_in=None):
        q, k, v, do = (_f64(x) for x in (q, k, v, do))
        dq, dk, dv, p, ds = attention_backward_one_head(
            q, k, v, do, scale, causal, o=None if o_in is None else _f64(o_in), return_terms=True)
        u, eta = U[dt], ETA[dt]
        gam = max(q.shape[0], k.shape[0]) * 2.0 ** -24   # fp32 sums over queries or keys
        g_d = 2 * q.shape[1] * 2.0 ** -24                # fp32 sums over the head dim
        vis = (p > 0).astype(np.float64)
        o_abs = np.abs(_f64(o_in)) if o_in is not None else np.abs(p @ v)
        # relative error of the recomputed P: the score's fp32 dot product (an error in
        # the exponent) plus DELTA
        rel_p = DELTA + g_d * scale * (np.abs(q) @ np.abs(k).T)
        # absolute error of dP - D in fp32 (both dot products over the head dim)
        e_dpd = g_d * (np.abs(do) @ np.abs(v).T + (np.abs(do) * o_abs).sum(axis=1, keepdims=True))
        tiny = TINY[dt]

        def e_cvt(x):  # conversion to the dtype (subnormals kept)
            return u * np.abs(x) + eta * vis

        def e_opnd(x):  # the same, as an MMA operand: a subnormal may also be lost
            ax = np.abs(x)
            return np.where(ax < tiny, ax, u * ax) + eta * vis

        def v_cvt(x):  # variance of independent conversions
            return (u * u / 3) * x * x + (eta * eta / 3) * vis

        # A lost subnormal term is a function of the data, not an independent
        # rounding: those terms are taken as adding up coherently (worst case).
        lost_s = np.where(np.abs(ds) < tiny, np.abs(ds), 0.0) * vis
        lost_p = np.where(p < tiny, p, 0.0) * vis
        # dS = P~ (dP - D) is formed from the rounded P~ of the dV product
        dpd = np.where(vis > 0, ds / np.where(vis > 0, p, 1.0), 0.0)

        e_s = e_opnd(ds) + np.abs(dpd) * e_cvt(p) + (gam + rel_p) * np.abs(ds) + p * e_dpd
        e_p = e_opnd(p) + (gam + rel_p) * p
        w = [scale * e_s @ np.abs(k), scale * e_s.T @ np.abs(q), e_p.T @ np.abs(do)]
        # standard deviations: an fp32 sum of n terms errs like a random walk, sqrt(n)
        # roundings rather than the worst case's n
        shrink = 1.0 / np.sqrt(q.shape[1])
        v_s = (np.where(np.abs(ds) < tiny, 0.0, v_cvt(ds)) + dpd ** 2 * v_cvt(p)
               + ((shrink * rel_p) ** 2 / 3) * ds ** 2 + (shrink * p * e_dpd) ** 2 / 3)
        v_p = np.where(p < tiny, 0.0, v_cvt(p)) + ((shrink * rel_p) ** 2 / 3) * p ** 2
        var = [scale ** 2 * v_s @ k ** 2 + (scale * lost_s @ np.abs(k)) ** 2,
               scale ** 2 * v_s.T @ q ** 2 + (scale * lost_s.T @ np.abs(q)) ** 2,
               v_p.T @ do ** 2 + (lost_p.T @ np.abs(do)) ** 2]
        # variance of each row's error projected on the reference row (t statistic):
        # the rounding of term (i, j) moves row i of dQ along scale * K_j, row j of dK
        # along scale * Q_i and row j of dV along dO_i
        c_q = scale * (dq @ k.T)            # [query i, key j]: (scale K_j) . dQ_i
        c_k = scale * (dk @ q.T)            # [key j, query i]: (scale Q_i) . dK_j
        c_v = dv @ do.T                     # [key j, query i]: dO_i . dV_j
        out = (u * u / 3 + DELTA ** 2)
        self.var_t = [(v_s * c_q ** 2).sum(axis=1) + (lost_s * np.abs(c_q)).sum(axis=1) ** 2
                      + out * (dq ** 4).sum(axis=1),
                      (v_s.T * c_k ** 2).sum(axis=1) + (lost_s.T * np.abs(c_k)).sum(axis=1) ** 2
                      + out * (dk ** 4).sum(axis=1),
                      (v_p.T * c_v ** 2).sum(axis=1) + (lost_p.T * np.abs(c_v)).sum(axis=1) ** 2
                      + out * (dv ** 4).sum(axis=1)]
        self.ref = (dq, dk, dv)
        self.w = [wi + u * np.abs(g) + eta for wi, g in zip(w, self.ref)]
        self.sig = [np.sqrt(vi + (u * u / 3 + DELTA ** 2) * g ** 2 + eta * eta / 3)
                    for vi, g in zip(var, self.ref)]  # + the output rounding


def check_grads(got, bounds, what, row_stat=True):
    """got: (dq, dk, dv) arrays [rows, D]; bounds: a GradBounds over the same rows."""
    stats = {}
    for name, g, r, w, sig, vt in zip(("dq", "dk", "dv"), got, bounds.ref, bounds.w, bounds.sig,
                                      bounds.var_t):
        gg = np.asarray(g, dtype=np.float64)
        assert np.all(np.isfinite(gg)), f"{what}: non-finite {name}"
        err = np.abs(gg - r)
        ratio = err / (W_FACTOR * w)
        worst = float(np.nanmax(np.where(w > 0, ratio, np.where(err > 0, np.inf, 0.0))))
        live = sig.max(axis=1) > 0
        R = np.sqrt(np.mean((err[live] / np.maximum(sig[live], 1e-300)) ** 2, axis=1))
        t = np.abs(((gg - r) * r).sum(axis=1))[live] / np.sqrt(np.maximum(vt[live], 1e-300))
        stats[name] = (round(worst, 3), round(float(R.max()) if R.size else 0.0, 2),
                       round(float(t.max()) if t.size else 0.0, 2))
        assert worst <= 1.0, f"{what}: {name} error above its bound: {stats}"
        if row_stat:
            assert R.size == 0 or R.max() <= R_MAX, f"{what}: {name} rows off the model: {stats}"
            assert t.size == 0 or t.max() <= T_MAX, f"{what}: {name} rows off the model: {stats}"
    print(what, stats)
    return stats


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkg.load_library()


def _case(seed, B, H, Sq, Sk, D, dt):
    g = torch.Generator().manual_seed(seed)
    mk = lambda S: torch.randn(B, S, H, D, generator=g).to(dt)  # noqa: E731
    return mk(Sq), mk(Sk), mk(Sk), mk(Sq)


def _given_forward_dense(q, k, v, scale, causal):
    """The forward's outputs as a caller hands them to the backward: the oracle's O
    rounded to the input dtype and its LSE in fp32 (host-side, no GPU value)."""
    o, lse = attention_dense(q, k, v, scale, causal)
    return torch.from_numpy(o).to(q.dtype), torch.from_numpy(lse).float()


def _run_given(q, k, v, do, o, lse, causal, scale, cu_q=None, cu_k=None):
    dev = [t.to(DEV) for t in (q, k, v, o, do, lse)]
    cq = None if cu_q is None else torch.as_tensor(cu_q).to(DEV)
    ck = None if cu_k is None else torch.as_tensor(cu_k).to(DEV)
    dq, dk, dv = pkg.attn_bwd(*dev, causal=causal, scale=scale, cu_seqlens_q=cq,
                              cu_seqlens_k=ck)
    st = pkg.attn_check()
    assert st == pkg.ATTN_OK, pkg.status_string(st)
    return [g.float().cpu().numpy() for g in (dq, dk, dv)]


def check_dense(got, q, k, v, do, o_in, scale, causal, what, heads=None):
    """Every (batch, head) of a dense problem against its bounds; returns the worst stats."""
    B, _, H, _ = q.shape
    worst = {}
    for b in range(B):
        for h in (range(H) if heads is None else heads):
            bd = GradBounds(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], scale, causal,
                            q.dtype, o_in=o_in[b, :, h])
            st = check_grads([g[b, :, h] for g in got], bd, f"{what} b{b} h{h}")
            worst = {n: tuple(max(a, c) for a, c in zip(worst.get(n, (0, 0)), st[n]))
                     for n in st}
    return worst


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
    o_in, lse_in = _given_forward_dense(q, k, v, scale, causal)
    got = _run_given(q, k, v, do, o_in, lse_in, causal, scale)
    check_dense(got, q, k, v, do, o_in, scale, causal, _id(case))
    if causal and Sk > Sq:  # keys no query sees get exactly zero gradient
        assert np.all(got[1][:, Sq:] == 0) and np.all(got[2][:, Sq:] == 0)


@pytest.mark.parametrize("dt", [BF, FP], ids=["bf16", "fp16"])
def test_bwd_peaked_scores(dt):
    """Q, K ~ N(0, 16): a peaked softmax stresses P = exp(S - LSE) recomputation, and in
    fp16 many P and dS values fall into the subnormal range."""
    g = torch.Generator().manual_seed(77)
    B, H, S, D = 1, 2, 512, 128
    q = (torch.randn(B, S, H, D, generator=g) * 4).to(dt)
    k = (torch.randn(B, S, H, D, generator=g) * 4).to(dt)
    v = torch.randn(B, S, H, D, generator=g).to(dt)
    do = torch.randn(B, S, H, D, generator=g).to(dt)
    scale = 1 / math.sqrt(D)
    o_in, lse_in = _given_forward_dense(q, k, v, scale, True)
    got = _run_given(q, k, v, do, o_in, lse_in, True, scale)
    check_dense(got, q, k, v, do, o_in, scale, True, "peaked")


@pytest.mark.parametrize("dt,frac", [(FP, 0.01), (BF, 0.03)], ids=["fp16_1pct", "bf16_3pct"])
def test_bwd_planted_row_error_is_caught(dt, frac):
    """The checks are sensitive: scaling one row of the GPU's dQ, dK or dV by 1 + frac on
    the host makes the check fail, while the unaltered result passes.  In fp16 a 1 %
    error is caught.  In bf16 a 1 % error along a dQ row lies within the kernel's own
    rounding noise along that direction (each row of dS sums to zero, so dQ is a small
    difference of terms each rounded to 8 bits, and that noise reaches about 0.5-1 % of
    |dQ|): no check can flag it without flagging correct results; 3 % is caught."""
    B, H, S, D = 1, 1, 512, 128
    q, k, v, do = _case(2024, B, H, S, S, D, dt)
    scale = 1 / math.sqrt(D)
    o_in, lse_in = _given_forward_dense(q, k, v, scale, True)
    got = _run_given(q, k, v, do, o_in, lse_in, True, scale)
    bd = GradBounds(q[0, :, 0], k[0, :, 0], v[0, :, 0], do[0, :, 0], scale, True, dt,
                    o_in=o_in[0, :, 0])
    clean = [g[0, :, 0] for g in got]
    check_grads(clean, bd, "unaltered")
    for which in range(3):
        ref = bd.ref[which]
        # a row that many terms contribute to (dQ: a late query; dK, dV: an early key)
        row = int(np.argmax(np.sqrt((ref[100:S - 100] ** 2).mean(axis=1)))) + 100
        bad = [x.copy() for x in clean]
        bad[which][row] *= 1 + frac
        with pytest.raises(AssertionError):
            check_grads(bad, bd, f"planted {('dq', 'dk', 'dv')[which]} row {row}")


def test_bwd_dk_dv_deterministic():
    q, k, v, do = _case(3, 1, 2, 600, 600, 128, BF)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = pkg.attn_fwd(qd, kd, vd, causal=True, scale=0.09)
    a = pkg.attn_bwd(qd, kd, vd, o, dod, lse, causal=True, scale=0.09)
    b = pkg.attn_bwd(qd, kd, vd, o, dod, lse, causal=True, scale=0.09)
    assert pkg.attn_check() == pkg.ATTN_OK
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


def _given_forward_packed(q, k, v, cq, ck, scale, causal):
    """As _given_forward_dense; rows of no sequence come out NaN (the backward never
    reads them)."""
    o, lse = attention_varlen(q, k, v, cq, ck, scale, causal)
    return torch.from_numpy(o).to(q.dtype), torch.from_numpy(lse).float()


def check_packed(got, q, k, v, do, o_in, cq, ck, scale, causal, what, heads=None):
    H = q.shape[1]
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        for h in (range(H) if heads is None else heads):
            if q1 == q0 or k1 == k0:  # no query or no key: exact zeros
                assert np.all(got[0][q0:q1, h] == 0)
                assert np.all(got[1][k0:k1, h] == 0) and np.all(got[2][k0:k1, h] == 0)
                continue
            bd = GradBounds(q[q0:q1, h], k[k0:k1, h], v[k0:k1, h], do[q0:q1, h], scale, causal,
                            q.dtype, o_in=o_in[q0:q1, h])
            check_grads([got[0][q0:q1, h], got[1][k0:k1, h], got[2][k0:k1, h]], bd,
                        f"{what} seq{b} h{h}")


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
    o_in, lse_in = _given_forward_packed(q, k, v, cq, ck, scale, causal)
    got = _run_given(q, k, v, do, o_in, lse_in, causal, scale, cq, ck)
    check_packed(got, q, k, v, do, o_in, cq, ck, scale, causal, _vid(case))
    assert np.all(got[0][:int(cq[0])] == 0) and np.all(got[0][int(cq[-1]):] == 0)
    for b in range(len(lens_q)):  # keys no query sees: exactly zero
        k0, k1 = int(ck[b]), int(ck[b + 1])
        unseen = k0 + (min(lens_q[b], lens_k[b]) if causal else (lens_k[b] if lens_q[b] else 0))
        if unseen < k1:
            assert np.all(got[1][unseen:k1] == 0) and np.all(got[2][unseen:k1] == 0)


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
    o_in, lse_in = _given_forward_dense(q, k, v, scale, True)
    got = _run_given(q, k, v, do, o_in, lse_in, True, scale)
    check_dense(got, q, k, v, do, o_in, scale, True, "dense 256 units", heads=[0, 7, 15])


def test_bwd_many_units_per_cta_packed():
    """A packed batch of 9000 tokens over 8 heads (about 600 units): the sequence walk,
    per-sequence tile offsets and dQ rows across sequences with several units per CTA."""
    lens = [3000, 17, 2500, 1, 3482]
    H, D = 8, 128
    q, k, v, do, cq, ck = _packed_case(77, lens, lens, H, D, BF, lead=3, tail=5)
    scale = 1.0 / math.sqrt(D)
    o_in, lse_in = _given_forward_packed(q, k, v, cq, ck, scale, True)
    got = _run_given(q, k, v, do, o_in, lse_in, True, scale, cq, ck)
    check_packed(got, q, k, v, do, o_in, cq, ck, scale, True, "packed 600 units", heads=[1, 6])


def test_bwd_full_size_sampled():
    """The benchmarked problem (B=1 H=32 S=16384 D=128 bf16 causal) in the bench's launch
    configuration, O and LSE from the GPU forward: dQ at seeded query rows and dK, dV at
    the last keys of two heads against the oracle's sampled backward, each element within
    its a-priori bound (the forward's O error bound included)."""
    from oracle.sdpa_oracle import attention_backward_sampled
    from scaled_dot_product_tcgen05_gb300 import workloads as W
    wl = W.standard_workloads()["bwd16k_causal"]
    inp = W.make_inputs(wl)
    q, k, v, do = inp["q"], inp["k"], inp["v"], inp["do"]
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = pkg.attn_fwd(qd, kd, vd, causal=True, scale=wl.scale)
    got = pkg.attn_bwd(qd, kd, vd, o, dod, lse, causal=True, scale=wl.scale)
    assert pkg.attn_check() == pkg.ATTN_OK
    S = wl.Sq
    u = U[BF]
    rng = np.random.default_rng(16384)
    q_rows = np.union1d(rng.choice(S, 24, replace=False), [0, 1, 127, 128, 8191, S - 1])
    k_rows = np.union1d(np.arange(S - 64, S), [S - 129, S - 1000])
    for h in (0, 17):
        qh, kh, vh, doh = (_f64(t[0, :, h]) for t in (q, k, v, do))
        dq, dk, dv, rows, p, ds, o_rows = attention_backward_sampled(
            qh, kh, vh, doh, wl.scale, True, q_rows, k_rows, return_terms=True)
        # per-element bounds over the sampled outputs, from the terms of the rows used
        gam = S * 2.0 ** -24
        vis = (p > 0).astype(np.float64)
        e_s = (u + gam + DELTA) * np.abs(ds)
        o_err = u * (p @ np.abs(vh) + 2 * np.abs(o_rows))
        d_err = (np.abs(doh[rows]) * o_err).sum(axis=1, keepdims=True)
        at = np.searchsorted(rows, q_rows)
        w_dq = wl.scale * (e_s[at] @ np.abs(kh) + d_err[at] * (p[at] @ np.abs(kh)))
        w_dk = wl.scale * ((e_s[:, k_rows] + d_err * p[:, k_rows]).T @ np.abs(qh[rows]))
        w_dv = ((u + gam + DELTA) * p[:, k_rows]).T @ np.abs(doh[rows])
        for name, g_all, idx, ref, w in (("dq", got[0], q_rows, dq, w_dq),
                                         ("dk", got[1], k_rows, dk, w_dk),
                                         ("dv", got[2], k_rows, dv, w_dv)):
            g = g_all[0, idx, h].float().cpu().numpy().astype(np.float64)
            bound = W_FACTOR * (w + u * np.abs(ref))
            worst = float((np.abs(g - ref) / bound).max())
            print(f"bwd16k head {h} {name}: worst err / bound {worst:.3f}")
            assert worst <= 1.0, f"bwd16k head {h} {name}: {worst}"
        assert vis.any()
