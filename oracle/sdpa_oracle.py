"""fp64 CPU oracle for the fused attention forward.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the CPU-baseline leg of the benchmark may
import this module.  The product path (the CUDA library and its Python binding)
never calls it; it shares no code, table or helper with the CUDA kernels.

What it computes is the plain definition of scaled dot-product attention,
written out step by step as an unfused pipeline:

  * scores S = scale * Q K^T, materialised in full (page "Multi-Head Attention
    的计算本质与性能瓶颈", §1, the three-op bmm / softmax / bmm example, and §2.1,
    the Attention(Q,K,V) = softmax(QK^T/sqrt(d_k)) V decomposition);
  * causal mask: key j is visible to query i only when j <= i, indices counted
    from the start of each sequence (same page, §3.1, the conditional
    assignment in the fused-kernel sketch);
  * packed variable-length batches: sequence b owns query rows
    cu_seqlens_q[b]:cu_seqlens_q[b+1] and key rows cu_seqlens_k[b]:cu_seqlens_k[b+1]
    and never sees another sequence (page "长文本处理性能断层真相", §1, the
    varlen call with int32 cu_seqlens);
  * sliding window + global rows (page "长文本处理性能断层真相", §2.5, the hybrid
    of a local-window attention for every query and full attention for the
    first global_tokens queries, spliced row-wise): query i >= global_q sees
    key j only when i - window_left <= j <= i + window_right (-1: that side
    unbounded); query i < global_q sees every key.  The causal rule applies on
    top of both;
  * a full-row softmax (row max, exp, sum, divide), then P V;
  * the per-row logsumexp LSE_i = max_j s_ij + ln sum_j exp(s_ij - max_j s_ij),
    natural log, over the scaled and masked scores.

It deliberately does NOT use the online (running max / running sum) form that
the GPU path uses (page "深度学习算子优化：从TFLOPS幻觉到FlashAttention实战", §3),
so the two share no algebra beyond the definition.

Readings where the pages are silent:
  * a row with no visible key (only possible for an empty key sequence) gives
    O = 0 and LSE = -inf;
  * causal alignment is top-left (the literal i >= j test), so it also holds
    when a sequence has Sq != Sk;
  * the page sizes its window by one number (window_size); here the two sides
    of the band are given separately and include their end points, so a causal
    window of W keys (the query and the W-1 keys before it) is window_left =
    W - 1, window_right = 0; the page's "full attention" for the global rows
    keeps the causal rule when the call is causal.

Parity status: every function here is pinned (tests/test_oracle.py,
tests/test_oracle_window.py, tests/test_oracle_decode.py: brute force, closed
forms, invariants, a library routine); none is "parity unpinned".
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np


def _as_f64(x) -> np.ndarray:
    """Exact conversion of an fp16/bf16/fp32 torch tensor or numpy array to fp64."""
    if hasattr(x, "detach"):  # torch tensor; bf16 has no numpy dtype, fp64 is exact
        import torch
        return x.detach().to(device="cpu", dtype=torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def visible_mask(row_idx: np.ndarray, Sk: int, causal: bool, window_left: int = -1,
                 window_right: int = -1, global_q: int = 0) -> np.ndarray:
    """visible[r, j]: may query row_idx[r] see key j (indices within the sequence)."""
    i = np.asarray(row_idx, dtype=np.int64)[:, None]
    j = np.arange(Sk, dtype=np.int64)[None, :]
    visible = np.ones((i.shape[0], Sk), dtype=bool)
    banded = i >= global_q          # global rows ignore the window
    if window_left >= 0:
        visible &= ~banded | (j >= i - window_left)
    if window_right >= 0:
        visible &= ~banded | (j <= i + window_right)
    if causal:
        visible &= j <= i
    return visible


def attention_one_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                       causal: bool, rows: Optional[Sequence[int]] = None,
                       return_p: bool = False, window_left: int = -1, window_right: int = -1,
                       global_q: int = 0):
    """Attention for one (sequence, head).

    q [Sq, D], k [Sk, D], v [Sk, Dv] in fp64.  ``rows`` restricts the output to
    those query indices (indices within the sequence).  ``window_left``,
    ``window_right`` and ``global_q`` add the sliding-window mask (defaults:
    none).  Returns (O [R, Dv], LSE [R]) and, when ``return_p``, the probability
    matrix P [R, Sk].
    """
    Sq = q.shape[0]
    Sk = k.shape[0]
    row_idx = np.arange(Sq) if rows is None else np.asarray(rows, dtype=np.int64)
    qs = q[row_idx]
    # step 1: all scores, materialised
    s = scale * (qs @ k.T)                                   # [R, Sk]
    # step 2: mask -> visible[i, j]
    visible = visible_mask(row_idx, Sk, causal, window_left, window_right, global_q)
    s_masked = np.where(visible, s, -np.inf)
    # step 3: full-row softmax
    has_key = visible.any(axis=1)
    m = np.where(has_key, s_masked.max(axis=1, initial=-np.inf), 0.0)
    e = np.where(visible, np.exp(s_masked - m[:, None]), 0.0)
    z = e.sum(axis=1)
    p = np.where(has_key[:, None], e / np.where(has_key, z, 1.0)[:, None], 0.0)
    # step 4: P V and the logsumexp
    o = p @ v
    with np.errstate(divide="ignore"):
        lse = np.where(has_key, m + np.log(np.where(has_key, z, 1.0)), -np.inf)
    if return_p:
        return o, lse, p
    return o, lse


def attention_dense(q, k, v, scale: float, causal: bool,
                    heads: Optional[Sequence[int]] = None,
                    rows: Optional[Sequence[int]] = None, window_left: int = -1,
                    window_right: int = -1, global_q: int = 0):
    """Dense batch: q [B,Sq,H,D], k/v [B,Sk,H,D] -> O [B,Sq,H,D], LSE [B,H,Sq].

    With ``heads``/``rows`` only those heads/query rows are computed; the others
    are returned as NaN so that they cannot be mistaken for checked values.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, Sq, H, D = q.shape
    Dv = v.shape[3]
    o = np.full((B, Sq, H, Dv), np.nan)
    lse = np.full((B, H, Sq), np.nan)
    row_sel = np.arange(Sq) if rows is None else np.asarray(rows, dtype=np.int64)
    for b in range(B):
        for h in (range(H) if heads is None else heads):
            ob, lb = attention_one_head(q[b, :, h, :], k[b, :, h, :], v[b, :, h, :],
                                        scale, causal, rows=row_sel, window_left=window_left,
                                        window_right=window_right, global_q=global_q)
            o[b, row_sel, h, :] = ob
            lse[b, h, row_sel] = lb
    return o, lse


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool,
                     heads: Optional[Sequence[int]] = None, window_left: int = -1,
                     window_right: int = -1, global_q: int = 0):
    """Packed varlen batch: q [Tq,H,D], k/v [Tk,H,D] -> O [Tq,H,D], LSE [H,Tq].

    Rows of q that belong to no sequence are returned as NaN.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    cq = [int(x) for x in np.asarray(cu_seqlens_q).tolist()]
    ck = [int(x) for x in np.asarray(cu_seqlens_k).tolist()]
    Tq, H, D = q.shape
    Dv = v.shape[2]
    o = np.full((Tq, H, Dv), np.nan)
    lse = np.full((H, Tq), np.nan)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 == q0:
            continue
        for h in (range(H) if heads is None else heads):
            ob, lb = attention_one_head(q[q0:q1, h, :], k[k0:k1, h, :], v[k0:k1, h, :],
                                        scale, causal, window_left=window_left,
                                        window_right=window_right, global_q=global_q)
            o[q0:q1, h, :] = ob
            lse[h, q0:q1] = lb
    return o, lse


def attention_decode(q, k_cache, v_cache, seqlens_k, scale: float, causal: bool,
                     heads: Optional[Sequence[int]] = None):
    """Decode against a KV cache: the Sq new queries are the LAST Sq positions.

    q [B,Sq,H,D], k_cache/v_cache [B,Sk,H,D], seqlens_k [B] (valid cache rows,
    None = Sk).  Query t of sequence b sits at position L_b - Sq + t, so with
    causal it sees keys 0 .. L_b - Sq + t (the KV-cache layout and decode step of
    page "长文本处理性能断层真相", §2.2); without causal it sees keys 0 .. L_b-1.
    Written as the top-left causal definition applied to a query array whose
    rows L_b-Sq .. L_b-1 hold the new queries.  A query at a negative position
    sees no key: O = 0, LSE = -inf.  Returns O [B,Sq,H,D], LSE [B,H,Sq].
    """
    q, kc, vc = _as_f64(q), _as_f64(k_cache), _as_f64(v_cache)
    B, Sq, H, D = q.shape
    Sk = kc.shape[1]
    Dv = vc.shape[3]
    lens = [Sk] * B if seqlens_k is None else [int(x) for x in np.asarray(seqlens_k).tolist()]
    o = np.full((B, Sq, H, Dv), np.nan)
    lse = np.full((B, H, Sq), np.nan)
    for b in range(B):
        L = lens[b]
        for h in (range(H) if heads is None else heads):
            o[b, :, h, :] = 0.0
            lse[b, h, :] = -np.inf
            if L == 0:
                continue
            if not causal:  # every new query sees the L cached keys
                ob, lb = attention_one_head(q[b, :, h, :], kc[b, :L, h, :], vc[b, :L, h, :],
                                            scale, False)
                o[b, :, h, :], lse[b, h, :] = ob, lb
                continue
            # causal: query t at row L - Sq + t of a length-L query array
            live = [t for t in range(Sq) if L - Sq + t >= 0]
            if not live:
                continue
            qpos = np.zeros((L, D))
            for t in live:
                qpos[L - Sq + t] = q[b, t, h, :]
            ob, lb = attention_one_head(qpos, kc[b, :L, h, :], vc[b, :L, h, :], scale, True,
                                        rows=[L - Sq + t for t in live])
            o[b, live, h, :] = ob
            lse[b, h, live] = lb
    return o, lse


def merge_partials(o_parts, lse_parts):
    """Combine attention results computed over disjoint key sets.

    o_parts [P, ..., D], lse_parts [P, ...] (natural log).  With w_p =
    exp(LSE_p - max_p LSE_p): O = sum_p w_p O_p / sum_p w_p and
    LSE = max_p LSE_p + ln sum_p w_p -- the softmax over the union of the key
    sets, rebuilt from per-set results (the combine step of the ring attention
    on page "长文本处理性能断层真相", §1, where each GPU holds a slice of the
    tokens).  Entries whose parts are all -inf give O = 0, LSE = -inf.
    """
    o = _as_f64(o_parts)
    lp = _as_f64(lse_parts)
    m = lp.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isneginf(lp), 0.0, np.exp(lp - m_safe[None]))
    z = w.sum(axis=0)
    out = (w[..., None] * o).sum(axis=0) / np.where(finite, z, 1.0)[..., None]
    out = np.where(finite[..., None], out, 0.0)
    with np.errstate(divide="ignore"):
        lse = np.where(finite, m_safe + np.log(np.where(finite, z, 1.0)), -np.inf)
    return out, lse


def attention_backward_one_head(q, k, v, do, scale: float, causal: bool, o=None,
                                return_terms: bool = False):
    """Gradients of attention for one (sequence, head): returns dQ, dK, dV.

    q [Sq, D], k [Sk, D], v [Sk, Dv], do = dL/dO [Sq, Dv], fp64.  The forward is
    the same definition as attention_one_head (scores S = scale Q K^T, masked,
    row softmax P, O = P V); the gradient is the chain rule through those three
    steps.  Page "Multi-Head Attention的计算本质与性能瓶颈", §3.3, reserves the
    backward interface (every operator implements backward(grad_output)) and
    states that masked connections carry no gradient ("gradient mask"); it
    gives no formulas, so this is plain calculus on the definition:
        dV = P^T dO
        dP = dO V^T
        dS = P * (dP - rowsum(dP * P))        (softmax Jacobian, row by row)
        dQ = scale * dS K,   dK = scale * dS^T Q
    Masked entries have P = 0 and so no gradient; a row with no visible key
    contributes nothing.

    A backward is handed the forward's output O as an input; since
    rowsum(dP * P) = rowsum(dO * O) for the exact O, the row term may be taken
    from it.  ``o`` (optional, [Sq, Dv]) is such a caller-provided O: the row
    term becomes rowsum(dO * o), i.e. the gradient a backward computes from
    the O it was given (with ``o`` equal to the exact O, the gradient above).
    ``return_terms`` also returns P and dS (the terms that error bounds of an
    implementation are built from).
    """
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    Sq, Sk = q.shape[0], k.shape[0]
    _, _, p = attention_one_head(q, k, v, scale, causal, return_p=True)
    dv = p.T @ do
    dp = do @ v.T
    if o is None:
        row = (dp * p).sum(axis=1, keepdims=True)
    else:
        row = (do * np.asarray(o, dtype=np.float64)).sum(axis=1, keepdims=True)
    ds = p * (dp - row)
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    if return_terms:
        return dq, dk, dv, p, ds
    return dq, dk, dv


def attention_backward_dense(q, k, v, do, scale: float, causal: bool,
                             heads: Optional[Sequence[int]] = None, o=None):
    """Dense batch: q/do [B,Sq,H,D], k/v [B,Sk,H,D] -> dQ, dK, dV in the same layouts.

    Heads not listed in ``heads`` are NaN.  ``o`` [B,Sq,H,Dv]: the caller's
    forward output for the row term (see attention_backward_one_head).
    """
    q, k, v, do = (_as_f64(x) for x in (q, k, v, do))
    o = None if o is None else _as_f64(o)
    B, Sq, H, D = q.shape
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    for b in range(B):
        for h in (range(H) if heads is None else heads):
            g = attention_backward_one_head(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h],
                                            scale, causal,
                                            o=None if o is None else o[b, :, h])
            dq[b, :, h], dk[b, :, h], dv[b, :, h] = g
    return dq, dk, dv


def attention_backward_sampled(q, k, v, do, scale: float, causal: bool, q_rows, k_rows,
                               return_terms: bool = False):
    """dQ at the query rows ``q_rows`` and dK, dV at the key rows ``k_rows`` of one
    (sequence, head), for sequences too long to form every score.

    The same definitions as attention_backward_one_head (page "Multi-Head
    Attention的计算本质与性能瓶颈", §3.3, the chain rule through the forward),
    evaluated on the score rows these outputs need: the rows ``q_rows`` and
    every query row that sees one of the keys ``k_rows`` (under causal masking,
    for keys near the end of the sequence, a few rows).  Returns dQ
    [len(q_rows), D], dK [len(k_rows), D], dV [len(k_rows), Dv] in fp64; with
    ``return_terms`` also the score rows used, their P and dS, and their O.
    """
    q, k, v, do = (_as_f64(x) for x in (q, k, v, do))
    Sq, Sk = q.shape[0], k.shape[0]
    q_rows = np.asarray(q_rows, dtype=np.int64)
    k_rows = np.asarray(k_rows, dtype=np.int64)
    sees = np.zeros(Sq, dtype=bool)
    for r0 in range(0, Sq, 1024):  # the query rows that see one of the keys
        rr = np.arange(r0, min(Sq, r0 + 1024))
        sees[rr] = visible_mask(rr, Sk, causal)[:, k_rows].any(axis=1)
    rows = np.union1d(q_rows, np.nonzero(sees)[0])
    _, _, p = attention_one_head(q, k, v, scale, causal, rows=rows, return_p=True)
    dp = do[rows] @ v.T
    ds = p * (dp - (dp * p).sum(axis=1, keepdims=True))
    at = np.searchsorted(rows, q_rows)
    dq = scale * (ds[at] @ k)
    dk = scale * (ds[:, k_rows].T @ q[rows])
    dv = p[:, k_rows].T @ do[rows]
    if return_terms:
        return dq, dk, dv, rows, p, ds, p @ v
    return dq, dk, dv

def attention_backward_varlen(q, k, v, do, cu_seqlens_q, cu_seqlens_k, scale: float,
                              causal: bool, heads: Optional[Sequence[int]] = None, o=None):
    """Packed varlen batch: q/do [Tq,H,D], k/v [Tk,H,D] -> dQ, dK, dV in the same layouts.

    Sequence b's queries cu_seqlens_q[b]:cu_seqlens_q[b+1] see only its keys
    cu_seqlens_k[b]:cu_seqlens_k[b+1] (page "长文本处理性能断层真相", §1), so its
    gradients are those of attention_backward_one_head on its slices.  A
    sequence without queries gives its keys zero dK and dV; one without keys
    gives its queries zero dQ.  Rows that belong to no sequence, and heads not
    listed in ``heads``, are NaN.  ``o`` [Tq,H,Dv]: the caller's forward output
    for the row term (see attention_backward_one_head).
    """
    q, k, v, do = (_as_f64(x) for x in (q, k, v, do))
    o = None if o is None else _as_f64(o)
    cq = [int(x) for x in np.asarray(cu_seqlens_q).tolist()]
    ck = [int(x) for x in np.asarray(cu_seqlens_k).tolist()]
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    H = q.shape[1]
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        for h in (range(H) if heads is None else heads):
            if q1 == q0 or k1 == k0:
                dq[q0:q1, h] = 0.0
                dk[k0:k1, h] = 0.0
                dv[k0:k1, h] = 0.0
                continue
            g = attention_backward_one_head(q[q0:q1, h], k[k0:k1, h], v[k0:k1, h],
                                            do[q0:q1, h], scale, causal,
                                            o=None if o is None else o[q0:q1, h])
            dq[q0:q1, h], dk[k0:k1, h], dv[k0:k1, h] = g
    return dq, dk, dv
