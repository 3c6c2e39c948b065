"""GPU parity of the sliding-window + global-rows mask against the fp64 oracle.

The mask is the 128K-context hybrid of page "长文本处理性能断层真相", §2.5: a band
of keys around each query (window_left keys before it, window_right after it)
and full attention for the first global_q queries of each sequence.  Cases
cover both kernels (head dim 128 on CTA pairs, head dim 64 and ATTN_PAIR=0 on
single CTAs), band edges on and off tile boundaries, one- and two-key windows,
global rows spanning several query tiles, unbounded sides, Sq != Sk (rows whose
band holds no key), varlen batches, and the full-size windowed workload on
sampled rows.
"""
import math

import pytest
import torch

from scaled_dot_product_tcgen05_gb300 import workloads as W
from oracle.sdpa_oracle import attention_dense, attention_varlen
from parity_helpers import compare, run_gpu

import scaled_dot_product_tcgen05_gb300 as pkg

pytestmark = pytest.mark.gpu

BF, FP = torch.bfloat16, torch.float16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkg.load_library()


def _dense_case(seed, B, H, Sq, Sk, D, dtype):
    g = torch.Generator().manual_seed(seed)
    mk = lambda S: torch.randn(B, S, H, D, generator=g).to(dtype)  # noqa: E731
    return mk(Sq), mk(Sk), mk(Sk)


CASES = [
    # (B, H, Sq, Sk, D, dtype, causal, window_left, window_right, global_q)
    (1, 2, 1000, 1000, 128, BF, True, 255, 0, 0),
    (1, 2, 1000, 1000, 64, FP, True, 255, 0, 0),
    (2, 2, 2050, 2050, 128, BF, True, 1000, -1, 64),
    (1, 2, 2050, 2050, 64, BF, True, 1000, 0, 300),
    (1, 2, 600, 600, 64, BF, True, 0, 0, 0),
    (1, 2, 700, 700, 128, FP, True, 1, 0, 0),
    (1, 3, 1500, 1500, 128, BF, False, 100, 300, 0),
    (1, 3, 1500, 1500, 64, FP, False, 300, 100, 200),
    (1, 2, 900, 900, 128, BF, False, -1, 50, 0),
    (1, 2, 900, 900, 128, BF, False, 50, -1, 0),
    (1, 2, 900, 900, 128, FP, False, -1, -1, 130),
    (2, 2, 300, 1000, 128, BF, False, 64, 64, 0),
    (2, 2, 1000, 300, 64, FP, False, 64, 64, 0),
    (2, 2, 1000, 300, 128, BF, False, 64, 64, 0),
    (1, 2, 1000, 1000, 128, BF, True, 127, 0, 0),
    (1, 2, 1000, 1000, 128, BF, True, 128, 0, 0),
    (1, 1, 4096, 4096, 128, BF, True, 4095, 0, 64),
]


def _id(c):
    return "B{}H{}q{}k{}D{}{}{}w{},{}g{}".format(c[0], c[1], c[2], c[3], c[4],
                                                 "bf" if c[5] == BF else "fp",
                                                 "c" if c[6] else "", c[7], c[8], c[9])


def _check(case, what):
    B, H, Sq, Sk, D, dt, causal, wl, wr, g = case
    q, k, v = _dense_case(Sq * 3 + Sk + wl + 7 * g, B, H, Sq, Sk, D, dt)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_gpu(q, k, v, causal, scale, window=(wl, wr), global_q=g)
    o_ref, l_ref = attention_dense(q, k, v, scale, causal, window_left=wl, window_right=wr,
                                   global_q=g)
    compare(o, lse, o_ref, l_ref, what=f"{what} {_id(case)}")
    # rows whose band holds no key: O = 0 exactly and LSE = -inf
    empty = torch.isneginf(torch.from_numpy(l_ref))
    if empty.any():
        lse_c = lse.cpu()
        assert torch.isneginf(lse_c[empty]).all()
        rows = empty[0, 0].nonzero().flatten()
        assert torch.all(o[:, rows.to(o.device)] == 0)


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_window_dense(case):
    _check(case, "window")


@pytest.mark.parametrize("case", [c for c in CASES if c[4] == 128][:6], ids=_id)
def test_window_single_cta_head_dim_128(case, monkeypatch):
    monkeypatch.setenv("ATTN_PAIR", "0")
    _check(case, "window 1sm")


@pytest.mark.parametrize("D,dt", [(64, FP), (128, BF)])
@pytest.mark.parametrize("causal,wl,wr,g", [(True, 200, 0, 10), (False, 50, 80, 0),
                                            (False, 0, 0, 300)])
def test_window_varlen(D, dt, causal, wl, wr, g):
    lens_q = [1, 0, 300, 129, 5, 256, 1000]
    lens_k = [1, 7, 300, 129, 0, 100, 1000]
    gen = torch.Generator().manual_seed(21 + wl)
    cq = W.cu_seqlens_from_lengths(lens_q)
    ck = W.cu_seqlens_from_lengths(lens_k)
    q = torch.randn(int(cq[-1]), 3, D, generator=gen).to(dt)
    k = torch.randn(int(ck[-1]), 3, D, generator=gen).to(dt)
    v = torch.randn(int(ck[-1]), 3, D, generator=gen).to(dt)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_gpu(q, k, v, causal, scale, cq, ck, window=(wl, wr), global_q=g)
    o_ref, l_ref = attention_varlen(q, k, v, cq, ck, scale, causal, window_left=wl,
                                    window_right=wr, global_q=g)
    compare(o, lse, o_ref, l_ref, what=f"varlen window {causal} {wl} {wr} {g} D={D}")


def test_window_full_size_sampled_rows():
    """The 128K windowed workload: full GPU run, oracle on 256 rows of 4 heads."""
    wl = W.standard_workloads()["window128k_causal"]
    heads, rows = W.sampled_heads_rows(wl)
    rows = sorted(set(rows) | {1, 63, 64, 65, 4095, 4096, 4097})  # global / band edges
    inp = W.make_inputs(wl)
    o, lse = run_gpu(inp["q"], inp["k"], inp["v"], True, wl.scale, window=wl.window,
                     global_q=wl.global_q)
    o_ref, l_ref = attention_dense(inp["q"], inp["k"], inp["v"], wl.scale, True, heads=heads,
                                   rows=rows, window_left=wl.window[0],
                                   window_right=wl.window[1], global_q=wl.global_q)
    o_s = o[:, rows][:, :, heads].float().cpu().numpy()
    l_s = lse[:, heads][:, :, rows].cpu().numpy()
    compare(o_s, l_s, o_ref[:, rows][:, :, heads], l_ref[:, heads][:, :, rows], what=wl.name)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_window_default_equals_attn_fwd():
    """window=(-1,-1), global_q=0 through attn_fwd_window gives attn_fwd's bits."""
    q, k, v = _dense_case(3, 1, 2, 700, 700, 128, BF)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o1, l1 = pkg.attn_fwd(qd, kd, vd, causal=True)
    o2 = torch.empty_like(o1)
    l2 = torch.empty_like(l1)
    st = pkg.attn_fwd_window_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o2.data_ptr(),
                                 l2.data_ptr(), 1, 2, 700, 700, 128, 1 / math.sqrt(128), True,
                                 -1, -1, 0, 0, 0, 1, torch.cuda.current_stream().cuda_stream)
    assert st == pkg.ATTN_OK and pkg.attn_check() == pkg.ATTN_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
