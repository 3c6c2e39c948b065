"""GPU parity of the KV-cache decode and of the partial-result merge.

Decode (page "长文本处理性能断层真相", §2.2): Sq <= 16 new queries per sequence are
the last Sq positions of a sequence whose cache holds L_b rows.  Cases cover
Sq = 1, 2, 4, 5, 16 (the three kernel widths), head dims 64/128, fp16/bf16,
causal and not, per-sequence cache lengths (empty, shorter than Sq, not a
multiple of the 64-key tile), the unsplit and the split-and-merge paths, the
two full-size decode workloads on sampled heads, and device-side errors.
Merge (ring-attention combine, same page, §1): attn_fwd on key shards plus
attn_merge against the oracle over all keys.
"""
import math

import numpy as np
import pytest
import torch

import scaled_dot_product_tcgen05_gb300 as pkg
from scaled_dot_product_tcgen05_gb300 import workloads as W
from oracle.sdpa_oracle import attention_decode, attention_dense, merge_partials
from parity_helpers import compare

pytestmark = pytest.mark.gpu

BF, FP = torch.bfloat16, torch.float16
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkg.load_library()


def _case(seed, B, Sq, Sk, H, D, dt):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(B, Sq, H, D, generator=g).to(dt),
            torch.randn(B, Sk, H, D, generator=g).to(dt),
            torch.randn(B, Sk, H, D, generator=g).to(dt))


def _run(q, k, v, lens, causal, scale):
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV) if lens is not None else None
    o, lse = pkg.attn_decode(q.to(DEV), k.to(DEV), v.to(DEV), seqlens_k=sl, causal=causal,
                             scale=scale)
    st = pkg.attn_check()
    assert st == pkg.ATTN_OK, pkg.status_string(st)
    return o, lse


CASES = [
    # (B, Sq, Sk, H, D, dtype, causal, lens)
    (2, 1, 300, 4, 128, BF, True, None),
    (3, 1, 1000, 2, 64, FP, True, [1000, 17, 0]),
    (2, 2, 777, 3, 128, FP, False, [5, 777]),
    (2, 4, 4100, 2, 128, BF, True, [4100, 63]),
    (3, 5, 2000, 2, 64, BF, True, [2, 1999, 64]),
    (1, 16, 5000, 2, 128, BF, True, None),
    (2, 16, 900, 2, 64, FP, False, [900, 16]),
    (1, 1, 20000, 1, 128, BF, False, None),
    (40, 1, 200, 32, 128, BF, True, None),     # B*H >= 8 per SM: no split, no merge
    (40, 3, 150, 32, 64, FP, False, None),
]


def _id(c):
    return "B{}q{}k{}H{}D{}{}{}{}".format(c[0], c[1], c[2], c[3], c[4],
                                          "bf" if c[5] == BF else "fp", "c" if c[6] else "",
                                          "" if c[7] is None else "L" + "-".join(map(str, c[7])))


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_decode_parity(case):
    B, Sq, Sk, H, D, dt, causal, lens = case
    q, k, v = _case(B * 131 + Sq * 7 + Sk, B, Sq, Sk, H, D, dt)
    scale = 1.0 / math.sqrt(D)
    o, lse = _run(q, k, v, lens, causal, scale)
    o_ref, l_ref = attention_decode(q, k, v, None if lens is None else np.array(lens), scale,
                                    causal)
    compare(o, lse, o_ref, l_ref, what=_id(case))
    empty = np.isneginf(l_ref)
    if empty.any():  # queries that see no key: O = 0 exactly, LSE = -inf
        lc = lse.cpu().numpy()
        assert np.isneginf(lc[empty]).all()
        oc = o.float().cpu().numpy()
        for b, h, t in zip(*np.nonzero(empty)):
            assert np.all(oc[b, t, h] == 0)


@pytest.mark.parametrize("name", ["decode128k_q1", "decode32k_b16_q4"])
def test_decode_full_size_sampled_heads(name):
    wl = W.standard_workloads()[name]
    heads, _ = W.sampled_heads_rows(wl)
    inp = W.make_inputs(wl)
    o, lse = _run(inp["q"], inp["k"], inp["v"], None, True, wl.scale)
    bsel = sorted({0, wl.B - 1})
    sub = [inp[n][bsel][:, :, heads] for n in ("q", "k", "v")]
    o_ref, l_ref = attention_decode(*sub, None, wl.scale, True)
    o_s = o[bsel][:, :, heads].float().cpu().numpy()
    l_s = lse[bsel][:, heads].cpu().numpy()
    compare(o_s, l_s, o_ref, l_ref, what=name)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_decode_bad_seqlens_reported_and_context_survives():
    q, k, v = _case(5, 2, 1, 256, 2, 64, FP)
    sl = torch.tensor([10, 257], dtype=torch.int32, device=DEV)
    pkg.attn_decode(q.to(DEV), k.to(DEV), v.to(DEV), seqlens_k=sl)
    assert pkg.attn_check() == pkg.ATTN_ERR_BAD_SEQLENS
    sl = torch.tensor([-1, 3], dtype=torch.int32, device=DEV)
    pkg.attn_decode(q.to(DEV), k.to(DEV), v.to(DEV), seqlens_k=sl)
    assert pkg.attn_check() == pkg.ATTN_ERR_BAD_SEQLENS
    o, lse = _run(q, k, v, [256, 3], True, 0.125)
    o_ref, l_ref = attention_decode(q, k, v, np.array([256, 3]), 0.125, True)
    compare(o, lse, o_ref, l_ref, what="after bad seqlens")


def test_decode_workspace_too_small_rejected():
    B, Sq, Sk, H, D = 1, 1, 8192, 2, 128
    need = pkg.decode_workspace_bytes(B, H, Sq, Sk, D)
    assert need > 0
    q, k, v = (t.to(DEV) for t in _case(6, B, Sq, Sk, H, D, BF))
    ws = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(pkg.AttnError) as e:
        pkg.attn_decode(q, k, v, workspace=ws)
    assert e.value.status == pkg.ATTN_ERR_INVALID_ARG
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    pkg.attn_decode(q, k, v, workspace=ws)
    assert pkg.attn_check() == pkg.ATTN_OK


@pytest.mark.parametrize("D,dt", [(64, FP), (128, BF)])
def test_merge_of_key_shards_equals_attention_over_all_keys(D, dt):
    """Ring-attention combine: attn_fwd on 3 key shards, then attn_merge."""
    B, S, Sk, H = 2, 300, 1000, 3
    g = torch.Generator().manual_seed(7 + D)
    q = torch.randn(B, S, H, D, generator=g).to(dt)
    k = torch.randn(B, Sk, H, D, generator=g).to(dt)
    v = torch.randn(B, Sk, H, D, generator=g).to(dt)
    scale = 1 / math.sqrt(D)
    cuts = [0, 128, 700, 1000]
    parts_o, parts_l = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o, l = pkg.attn_fwd(q.to(DEV), k[:, a:b].contiguous().to(DEV),
                            v[:, a:b].contiguous().to(DEV), scale=scale)
        parts_o.append(o)
        parts_l.append(l)
    o, lse = pkg.attn_merge(torch.stack(parts_o), torch.stack(parts_l))
    assert pkg.attn_check() == pkg.ATTN_OK
    o_ref, l_ref = attention_dense(q, k, v, scale, False)
    compare(o, lse, o_ref, l_ref, what=f"merge D={D}")


def test_merge_against_the_oracle_merge_with_empty_parts():
    P, B, S, H, D = 4, 2, 50, 3, 40
    g = torch.Generator().manual_seed(9)
    op = torch.randn(P, B, S, H, D, generator=g).to(BF)
    lp = torch.randn(P, B, H, S, generator=g) * 3
    lp[1] = -math.inf                  # an empty shard
    lp[:, 0, 0, :5] = -math.inf        # rows no shard sees
    o, lse = pkg.attn_merge(op.to(DEV), lp.to(DEV))
    assert pkg.attn_check() == pkg.ATTN_OK
    # the oracle takes matching leading dims: LSE as [P, B, S, H]
    o_ref, l_ref = merge_partials(op.float().numpy(), lp.permute(0, 1, 3, 2).numpy())
    compare(o, lse, o_ref, l_ref.transpose(0, 2, 1), what="merge vs oracle")
    assert torch.all(o[0, :5, 0] == 0) and torch.isneginf(lse[0, 0, :5]).all()
