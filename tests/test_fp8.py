"""FP8 (e4m3) forward: the input decoding on the CPU and GPU parity.

The oracle is the same fp64 definition applied to the dequantised inputs
(code * per-tensor scale); the decoding itself is torch's float8_e4m3fn
conversion, pinned here against e4m3 bit patterns with known values.

Tolerance (from the arithmetic): Q, K, V reach both sides as the same e4m3
values, S is accumulated exactly enough in fp32, and the one extra rounding is
the probabilities to e4m3 (3 mantissa bits: relative half-ulp 2^-4) before
P V.  The row sum adds the same rounded values, so for a row dominated by one
key the error cancels; the worst case is two comparable weights, where O
moves by up to 2^-4 * 1/4 * |v_1 - v_2| (about 0.1 for unit-variance V).
Bounds: O max-abs <= 0.15, mean-abs <= 1e-2 (random-sign rounding errors
average out over many keys); LSE uses the unrounded sum: 1e-3 relative as the
16-bit path.
"""
import math

import numpy as np
import pytest
import torch

import scaled_dot_product_tcgen05_gb300 as pkg
from scaled_dot_product_tcgen05_gb300 import workloads as W
from oracle.sdpa_oracle import attention_dense

DEV = "cuda:0"
O_MAX, O_MEAN, LSE_REL = 0.15, 1e-2, 1e-3


def test_e4m3_decoding_matches_known_codes():
    """OCP e4m3 (1-4-3, bias 7): 0x38 = 1, 0x40 = 2, 0x7e = 448, 0x01 = 2^-9,
    0x08 = 2^-6 (smallest normal), 0xb8 = -1, 0x3c = 1.5."""
    codes = torch.tensor([0x38, 0x40, 0x7E, 0x01, 0x08, 0xB8, 0x3C], dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64).tolist()
    assert vals == [1.0, 2.0, 448.0, 2.0 ** -9, 2.0 ** -6, -1.0, 1.5]


def test_quantize_round_trip_is_within_half_ulp():
    g = torch.Generator().manual_seed(1)
    x = torch.randn(4096, generator=g)
    codes, s = W.quantize_e4m3(x)
    back = codes.to(torch.float64) * s
    rel = (back - x.double()).abs() / x.double().abs().clamp_min(2.0 ** -6 * s)
    assert float(rel.max()) <= 2.0 ** -4 + 1e-9


def _case(seed, B, H, Sq, Sk):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Sq, H, 128, generator=g)
    k = torch.randn(B, Sk, H, 128, generator=g)
    v = torch.randn(B, Sk, H, 128, generator=g)
    return [W.quantize_e4m3(t) for t in (q, k, v)]


def _compare(o, lse, o_ref, l_ref, what):
    og = o.float().cpu().numpy().astype(np.float64)
    lg = lse.cpu().numpy().astype(np.float64)
    d = np.abs(og - o_ref)
    dl = np.abs(lg - l_ref) / np.maximum(1.0, np.abs(l_ref))
    stats = dict(o_max=float(d.max()), o_mean=float(d.mean()), lse=float(dl.max()))
    print(f"{what}: {stats}")
    assert stats["o_max"] <= O_MAX and stats["o_mean"] <= O_MEAN and stats["lse"] <= LSE_REL, \
        f"{what}: {stats}"
    return stats


CASES = [(1, 2, 256, 256, True), (1, 2, 300, 300, False), (2, 3, 1000, 1000, True),
         (1, 2, 130, 517, False), (1, 1, 1, 1, True), (1, 4, 2048, 2048, True)]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}q{}k{}{}".format(*c[:4], "c" if c[4] else ""))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
def test_fp8_parity(case, out_dtype):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B, H, Sq, Sk, causal = case
    (q8, qs), (k8, ks), (v8, vs) = _case(Sq * 3 + Sk, B, H, Sq, Sk)
    scale = 1.0 / math.sqrt(128)
    o, lse = pkg.attn_fwd_fp8(q8.to(DEV), k8.to(DEV), v8.to(DEV), q_scale=qs, k_scale=ks,
                              v_scale=vs, causal=causal, scale=scale, out_dtype=out_dtype)
    assert pkg.attn_check() == pkg.ATTN_OK
    deq = [t.to(torch.float64) * s for t, s in ((q8, qs), (k8, ks), (v8, vs))]
    o_ref, l_ref = attention_dense(*deq, scale, causal)
    _compare(o, lse, o_ref, l_ref, f"{case} {out_dtype}")


@pytest.mark.gpu
def test_fp8_full_size_sampled_rows():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = W.standard_workloads()["fp8_long64k_causal"]
    heads, rows = W.sampled_heads_rows(wl)
    inp = W.make_inputs(wl)
    (q8, qs), (k8, ks), (v8, vs) = (W.quantize_e4m3(inp[n]) for n in ("q", "k", "v"))
    o, lse = pkg.attn_fwd_fp8(q8.to(DEV), k8.to(DEV), v8.to(DEV), q_scale=qs, k_scale=ks,
                              v_scale=vs, causal=True, scale=wl.scale)
    assert pkg.attn_check() == pkg.ATTN_OK
    sub = [t.view(torch.uint8)[:, :, heads].view(torch.float8_e4m3fn).to(torch.float64) * s
           for t, s in ((q8, qs), (k8, ks), (v8, vs))]
    o_ref, l_ref = attention_dense(*sub, wl.scale, True, rows=rows)
    o_s = o[:, rows][:, :, heads].cpu()
    l_s = lse[:, heads][:, :, rows].cpu()
    _compare(o_s, l_s, o_ref[:, rows], l_ref[:, :, rows], wl.name)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


@pytest.mark.gpu
def test_fp8_paired_row_blocks_ragged_causal():
    """Many units per CTA: row blocks are scheduled in pairs and aligned to the end of
    the sequence; S = 16000 leaves a partial first block.  Sampled rows of two heads."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B, H, S = 2, 32, 16000
    (q8, qs), (k8, ks), (v8, vs) = _case(16001, B, H, S, S)
    scale = 1.0 / math.sqrt(128)
    o, lse = pkg.attn_fwd_fp8(q8.to(DEV), k8.to(DEV), v8.to(DEV), q_scale=qs, k_scale=ks,
                              v_scale=vs, causal=True, scale=scale)
    assert pkg.attn_check() == pkg.ATTN_OK
    heads = [3, 30]
    rows = sorted({0, 1, 127, 128, 129, 255, 256, 383, 384, 7000, S - 257, S - 256, S - 129,
                   S - 128, S - 2, S - 1})
    sub = [t.view(torch.uint8)[:, :, heads].view(torch.float8_e4m3fn).to(torch.float64) * s
           for t, s in ((q8, qs), (k8, ks), (v8, vs))]
    o_ref, l_ref = attention_dense(*sub, scale, True, rows=rows)
    o_s = o[:, rows][:, :, heads].cpu()
    l_s = lse[:, heads][:, :, rows].cpu()
    _compare(o_s, l_s, o_ref[:, rows], l_ref[:, :, rows], "fp8 paired blocks")
