"""GPU parity: the CUDA path against the fp64 CPU oracle on the same seeded inputs.

All calls go through the C ABI (ctypes binding).  Workloads follow the five
families of the attention-forward study (tiny, 512, 2K with a peaked draw,
packed varlen, long context) plus edge cases: ragged tails, Sq != Sk, empty
and single-token sequences, zero and negative scale, poisoned output buffers.
"""
import math

import numpy as np
import pytest
import torch

import scaled_dot_product_tcgen05_gb300 as pkg
from scaled_dot_product_tcgen05_gb300 import workloads as W
from oracle.sdpa_oracle import attention_dense, attention_varlen
from parity_helpers import compare, run_gpu

pytestmark = pytest.mark.gpu

WL = W.standard_workloads()
# workloads the oracle checks in full (the long-context ones are sampled below)
SMALL = [n for n, w in WL.items()
         if w.Sq <= 4096 and not w.windowed and not w.decode and not w.backward and not w.fp8]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkg.load_library()


@pytest.mark.parametrize("name", SMALL)
def test_workload_parity(name):
    wl = WL[name]
    inp = W.make_inputs(wl)
    o, lse = run_gpu(inp["q"], inp["k"], inp["v"], wl.causal, wl.scale, inp["cu_seqlens_q"],
                     inp["cu_seqlens_k"])
    if wl.varlen:
        o_ref, l_ref = attention_varlen(inp["q"], inp["k"], inp["v"], inp["cu_seqlens_q"],
                                        inp["cu_seqlens_k"], wl.scale, wl.causal)
    else:
        o_ref, l_ref = attention_dense(inp["q"], inp["k"], inp["v"], wl.scale, wl.causal)
    compare(o, lse, o_ref, l_ref, what=name)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [True, False])
def test_peaked_head_dim_128(dtype, causal):
    """The peaked draw (Q, K ~ N(0, 16)) at head dim 128, the CTA-pair kernel's case.

    Nearly one-hot rows are where the rounding of P to 16 bits shows in O unless
    the softmax denominator accounts for it; 24 heads of 2048 x 2048.
    """
    wl = W.Workload(name="peaked_d128", wid=3, B=2, H=12, Sq=2048, Sk=2048, D=128, dtype=dtype,
                    causal=causal, std=(4.0, 4.0, 1.0), draw=3)
    inp = W.make_inputs(wl)
    o, lse = run_gpu(inp["q"], inp["k"], inp["v"], causal, wl.scale)
    o_ref, l_ref = attention_dense(inp["q"], inp["k"], inp["v"], wl.scale, causal)
    compare(o, lse, o_ref, l_ref, what=f"peaked_d128_{dtype}_{causal}")


@pytest.mark.parametrize("name", ["long64k_causal", "long128k_causal"])
def test_long_context_sampled_rows(name):
    """Full GPU run; the oracle checks 256 seeded rows on 4 seeded heads."""
    wl = WL[name]
    heads, rows = W.sampled_heads_rows(wl)
    inp = W.make_inputs(wl)
    o, lse = run_gpu(inp["q"], inp["k"], inp["v"], True, wl.scale)
    o_ref, l_ref = attention_dense(inp["q"], inp["k"], inp["v"], wl.scale, True, heads=heads,
                                   rows=rows)
    o_s = o[:, rows][:, :, heads].float().cpu().numpy()
    l_s = lse[:, heads][:, :, rows].cpu().numpy()
    compare(o_s, l_s, o_ref[:, rows][:, :, heads], l_ref[:, heads][:, :, rows], what=name)
    # every output is finite, and rows of the unsampled heads are plausible
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def _dense_case(seed, B, H, Sq, Sk, D, dtype, std=1.0):
    g = torch.Generator().manual_seed(seed)
    mk = lambda S: (torch.randn(B, S, H, D, generator=g) * std).to(dtype)  # noqa: E731
    return mk(Sq), mk(Sk), mk(Sk)


EDGE = [
    # (B, H, Sq, Sk, D, dtype, causal)
    (1, 1, 1, 1, 64, torch.float16, False),
    (1, 1, 1, 1, 128, torch.bfloat16, True),
    (2, 3, 127, 127, 64, torch.bfloat16, True),
    (2, 3, 129, 129, 128, torch.float16, True),
    (1, 2, 2050, 2050, 64, torch.float16, True),
    (1, 2, 2050, 2050, 128, torch.bfloat16, False),
    (2, 2, 300, 77, 128, torch.bfloat16, False),
    (2, 2, 77, 300, 64, torch.float16, False),
    (2, 2, 300, 77, 64, torch.bfloat16, True),
    (2, 2, 77, 300, 128, torch.float16, True),
    (3, 5, 256, 256, 128, torch.float16, False),
    (1, 4, 385, 1000, 128, torch.bfloat16, False),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: "B{}H{}q{}k{}D{}{}{}".format(
    c[0], c[1], c[2], c[3], c[4], "bf" if c[5] == torch.bfloat16 else "fp", "c" if c[6] else ""))
def test_edge_shapes(case):
    B, H, Sq, Sk, D, dt, causal = case
    q, k, v = _dense_case(Sq * 7 + Sk, B, H, Sq, Sk, D, dt)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_gpu(q, k, v, causal, scale)
    o_ref, l_ref = attention_dense(q, k, v, scale, causal)
    compare(o, lse, o_ref, l_ref, what=str(case))


@pytest.mark.parametrize("scale", [0.0, -0.2, 0.9])
def test_scale_values(scale):
    q, k, v = _dense_case(3, 1, 2, 200, 200, 64, torch.float16)
    for causal in (False, True):
        o, lse = run_gpu(q, k, v, causal, scale)
        o_ref, l_ref = attention_dense(q, k, v, scale, causal)
        compare(o, lse, o_ref, l_ref, what=f"scale={scale} causal={causal}")


def _varlen(seed, lens_q, lens_k, H, D, dtype):
    g = torch.Generator().manual_seed(seed)
    cq = W.cu_seqlens_from_lengths(lens_q)
    ck = W.cu_seqlens_from_lengths(lens_k)
    q = torch.randn(int(cq[-1]), H, D, generator=g).to(dtype)
    k = torch.randn(max(int(ck[-1]), 1), H, D, generator=g).to(dtype)
    v = torch.randn(max(int(ck[-1]), 1), H, D, generator=g).to(dtype)
    return q, k, v, cq, ck


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dt", [(64, torch.float16), (128, torch.bfloat16)])
def test_varlen_edges(causal, D, dt):
    lens_q = [1, 0, 300, 129, 5, 256, 1000]
    lens_k = [1, 7, 300, 129, 0, 100, 1000]
    q, k, v, cq, ck = _varlen(11, lens_q, lens_k, 3, D, dt)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_gpu(q, k, v, causal, scale, cq, ck)
    o_ref, l_ref = attention_varlen(q, k, v, cq, ck, scale, causal)
    compare(o, lse, o_ref, l_ref, what=f"varlen causal={causal} D={D}")
    # the sequence with no keys: O = 0 exactly, LSE = -inf
    a, b = int(cq[4]), int(cq[5])
    assert torch.all(o[a:b] == 0) and torch.all(torch.isneginf(lse[:, a:b]))


@pytest.mark.parametrize("D,causal,guard", [(128, True, 4096), (128, True, 4104),
                                             (64, False, 4104), (64, True, 4104)],
                         ids=["pair_o32", "pair_o16", "pair_d64_o16", "single_d64_o16"])
def test_poisoned_outputs_and_guard_bands(D, causal, guard):
    """Writes land only on valid rows: guards and rows outside every sequence keep NaN.
    A guard of 4104 elements puts O 16 bytes off a 32-byte boundary, so the rows are
    written with 16-byte stores instead of 32-byte ones."""
    H, dt = 2, torch.bfloat16
    lens = [130, 3, 250]
    q, k, v, cq, ck = _varlen(12, lens, lens, H, D, dt)
    Tq = int(cq[-1])
    pad_rows = 40                      # rows after the last sequence: not owned by anyone
    dev = torch.device("cuda:0")
    qd = torch.cat([q, torch.randn(pad_rows, H, D).to(dt)]).to(dev)
    kd, vd = k.to(dev), v.to(dev)
    o_buf = torch.full(((Tq + pad_rows) * H * D + 2 * guard,), float("nan"), dtype=dt, device=dev)
    l_buf = torch.full((H * (Tq + pad_rows) + 2 * guard,), float("nan"), device=dev)
    o = o_buf[guard:guard + (Tq + pad_rows) * H * D].view(Tq + pad_rows, H, D)
    lse = l_buf[guard:guard + H * (Tq + pad_rows)].view(H, Tq + pad_rows)
    pkg.attn_fwd(qd, kd, vd, causal=causal, cu_seqlens_q=cq.to(dev), cu_seqlens_k=ck.to(dev),
                 out=o, lse=lse)
    assert pkg.attn_check() == pkg.ATTN_OK
    assert torch.isnan(o_buf[:guard]).all() and torch.isnan(o_buf[-guard:]).all()
    assert torch.isnan(l_buf[:guard]).all() and torch.isnan(l_buf[-guard:]).all()
    assert torch.isnan(o[Tq:]).all() and torch.isnan(lse[:, Tq:]).all()
    o_ref, l_ref = attention_varlen(q, k, v, cq, ck, 1 / math.sqrt(D), causal)
    compare(o[:Tq], lse[:, :Tq], o_ref, l_ref, what="poisoned")


def test_bad_cu_seqlens_reported():
    H, D, dt = 2, 64, torch.float16
    dev = torch.device("cuda:0")
    q = torch.randn(300, H, D).to(dt).to(dev)
    cu = torch.tensor([0, 200, 100, 300], dtype=torch.int32, device=dev)  # decreasing
    o, lse = pkg.attn_fwd(q, q, q, cu_seqlens_q=cu, cu_seqlens_k=cu)
    assert pkg.attn_check() == pkg.ATTN_ERR_BAD_SEQLENS
    cu2 = torch.tensor([0, 100, 400], dtype=torch.int32, device=dev)  # past the end
    pkg.attn_fwd(q, q, q, cu_seqlens_q=cu2, cu_seqlens_k=cu2)
    assert pkg.attn_check() == pkg.ATTN_ERR_BAD_SEQLENS
    # the context stays usable and the next call is clean
    qc, kc, vc = _dense_case(1, 1, 2, 128, 128, 64, torch.float16)
    o, lse = run_gpu(qc, kc, vc, False, 0.125)
    o_ref, l_ref = attention_dense(qc, kc, vc, 0.125, False)
    compare(o, lse, o_ref, l_ref)


def test_deterministic_and_stream_ordered():
    q, k, v = _dense_case(5, 2, 4, 1024, 1024, 128, torch.bfloat16)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1 = run_gpu(q, k, v, True, 0.088, stream=s)
        o2, l2 = run_gpu(q, k, v, True, 0.088, stream=s)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_host_and_misplaced_pointers_rejected():
    q = torch.randn(1, 128, 2, 64).half()  # host memory
    st = pkg.attn_fwd_raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(),
                          1, 2, 128, 128, 64, 0.125, False, 0, 0, 0, 0)
    assert st == pkg.ATTN_ERR_INVALID_ARG


def test_grid_is_persistent(monkeypatch):
    # CTA pairs (head dim 128; head dim 64 without a causal mask): one pair per two SMs
    for D, seed, causal in ((128, 6, True), (64, 7, False)):
        q, k, v = _dense_case(seed, 1, 32, 4096, 4096, D, torch.bfloat16)
        run_gpu(q, k, v, causal, 1 / math.sqrt(D))
        grid, smem = pkg.last_launch()
        assert grid == 2 * (pkg.num_sms() // 2) and smem <= 232448
    run_gpu(q, k, v, True, 0.125)  # head dim 64, causal: single CTAs, one per SM
    grid, smem = pkg.last_launch()
    assert grid == pkg.num_sms() and smem <= 232448


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("case", [
    (2, 3, 700, 700, torch.bfloat16, True),
    (1, 2, 300, 520, torch.float16, False),
], ids=["dense_bf16_causal", "dense_fp16_q300_k520"])
def test_single_cta_kernel(case, D, monkeypatch):
    """Both head dims run on CTA pairs; ATTN_PAIR=0 keeps the single-CTA kernel covered."""
    monkeypatch.setenv("ATTN_PAIR", "0")
    B, H, Sq, Sk, dt, causal = case
    q, k, v = _dense_case(Sq + 3 * Sk + D, B, H, Sq, Sk, D, dt)
    o, lse = run_gpu(q, k, v, causal, 1 / math.sqrt(D))
    grid, _ = pkg.last_launch()
    assert grid <= pkg.num_sms()
    o_ref, l_ref = attention_dense(q, k, v, 1 / math.sqrt(D), causal)
    compare(o, lse, o_ref, l_ref, what=f"1sm D={D} {case}")
    lens = [300, 1, 129, 0, 900]
    qv, kv, vv, cq, ck = _varlen(13, lens, lens, 2, D, torch.bfloat16)
    o, lse = run_gpu(qv, kv, vv, True, 0.1, cq, ck)
    o_ref, l_ref = attention_varlen(qv, kv, vv, cq, ck, 0.1, True)
    compare(o, lse, o_ref, l_ref, what=f"1sm D={D} varlen")


PAIR_CASES = [
    (2, 3, 700, 700, torch.bfloat16, True),
    (1, 2, 300, 520, torch.float16, False),
    (1, 4, 2050, 2050, torch.bfloat16, True),
    (2, 2, 77, 300, torch.float16, True),
]


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: "B{}H{}q{}k{}{}{}".format(
    c[0], c[1], c[2], c[3], "bf" if c[4] == torch.bfloat16 else "fp", "c" if c[5] else ""))
def test_cta_pair_kernel(case, D, monkeypatch):
    """Both head dims on CTA pairs (2-SM MMAs)."""
    monkeypatch.setenv("ATTN_PAIR", "1")
    B, H, Sq, Sk, dt, causal = case
    q, k, v = _dense_case(Sq + 5 * Sk + D, B, H, Sq, Sk, D, dt)
    o, lse = run_gpu(q, k, v, causal, 1 / math.sqrt(D))
    grid, _ = pkg.last_launch()
    assert grid % 2 == 0
    o_ref, l_ref = attention_dense(q, k, v, 1 / math.sqrt(D), causal)
    compare(o, lse, o_ref, l_ref, what=f"pair D={D} {case}")


@pytest.mark.parametrize("D", [128, 64])
def test_cta_pair_kernel_varlen(D, monkeypatch):
    monkeypatch.setenv("ATTN_PAIR", "1")
    for causal in (False, True):
        lens_q = [1, 0, 300, 129, 5, 256, 1000]
        lens_k = [1, 7, 300, 129, 0, 100, 1000]
        q, k, v, cq, ck = _varlen(14, lens_q, lens_k, 3, D, torch.bfloat16)
        o, lse = run_gpu(q, k, v, causal, 0.09, cq, ck)
        o_ref, l_ref = attention_varlen(q, k, v, cq, ck, 0.09, causal)
        compare(o, lse, o_ref, l_ref, what=f"pair varlen causal={causal}")
        a, b = int(cq[4]), int(cq[5])
        assert torch.all(o[a:b] == 0) and torch.all(torch.isneginf(lse[:, a:b]))


def _boundary_rows(S, n_random, seed):
    """Rows 0, S-1, both sides of every 128-row tile edge near the start and end of the
    sequence (end-aligned causal blocks put the partial block first), plus seeded rows."""
    edge = set()
    for base in (0, S % 128, S % 256):
        for t in range(4):
            for d in (-1, 0, 1):
                for r in (base + 128 * t + d, S - 1 - (base + 128 * t + d)):
                    if 0 <= r < S:
                        edge.add(r)
    g = torch.Generator().manual_seed(seed)
    edge.update((torch.randperm(S - 2, generator=g)[:n_random] + 1).tolist())
    return sorted(edge | {0, S - 1})


@pytest.mark.parametrize("D,dt", [(128, torch.bfloat16), (64, torch.float16)],
                         ids=["cta_pair_d128", "single_cta_d64"])
def test_paired_row_blocks_ragged_causal(D, dt):
    """A causal problem with many units per worker: row blocks are scheduled in pairs
    (heaviest with lightest of one head) and aligned to the end of the sequence, so
    S = 16000 leaves a partial first block whose rows before 0 do not exist.  The oracle
    checks rows at every tile edge near both ends and seeded rows of three heads."""
    B, H, S = 2, 32, 16000
    q, k, v = _dense_case(16000 + D, B, H, S, S, D, dt)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_gpu(q, k, v, True, scale)
    heads = [0, 17, 31]
    rows = _boundary_rows(S, 60, seed=D)
    o_ref, l_ref = attention_dense(q[:, :, heads], k[:, :, heads], v[:, :, heads], scale, True,
                                   rows=rows)
    o_s = o[:, rows][:, :, heads].float().cpu().numpy()
    l_s = lse[:, heads][:, :, rows].cpu().numpy()
    compare(o_s, l_s, o_ref[:, rows], l_ref[:, :, rows], what=f"paired blocks D={D}")
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


# Unit roundoff of the 16-bit P and O: 2^-8 (bf16, 8 significant bits), 2^-11 (fp16).
_U16 = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}


def _equal_scores_case(pattern, S, D, dt):
    """Q = e_0 in every row, K[j, 0] in {0, 1} by ``pattern``, V constant per head.

    Every score is 0 or scale, so a row's probabilities take two values, each shared by
    hundreds of keys.  ``scale`` is chosen so that the smaller (A, C2) or the larger
    (C1) of the two exponentials lies 0.45 of a unit in the last place above a 16-bit
    value: its rounding to 16 bits, made once per key, is as large as it gets short of
    a tie, and every one of those keys carries it.
      A  : key j scores high iff j % 64 == 0 (a high key in every half tile, so the
           row max is known from the first tile on and the low keys are below it);
      C1 : the first half of the keys low, the second half high by a factor 2^4 in
           probability (within the kernels' 2^8 rescale threshold, so a row that meets
           the low keys first keeps its stale max and the high keys' values exceed 1);
      C2 : the first half high, the second half low.
    """
    u_bits = 8 if dt == torch.bfloat16 else 11  # significant bits
    q = torch.zeros(1, S, 2, D)
    q[..., 0] = 1.0
    k = torch.zeros(1, S, 2, D)
    j = torch.arange(S)
    if pattern == "A":
        k[0, j % 64 == 0, :, 0] = 1.0
        small = 0.5 * (1.0 + 0.45 * 2.0 ** (1 - u_bits))  # in [1/2, 1): ulp = 2^-u_bits
        scale = -math.log(small)
    else:
        high = (j >= S // 2) if pattern == "C1" else (j < S // 2)
        k[0, high, :, 0] = 1.0
        big = 16.0 * (1.0 + 0.45 * 2.0 ** (1 - u_bits))  # in [16, 32): ulp = 16·2^(1-u_bits)
        scale = math.log(big)
    v = torch.empty(1, S, 2, D)
    v[:, :, 0] = 100.0  # exact in both 16-bit formats
    v[:, :, 1] = -37.25
    return q.to(dt), k.to(dt), v.to(dt), scale


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("pattern", ["A", "C1", "C2"])
def test_many_equal_rounded_probabilities(pattern, D, dt, causal):
    """The one-sum denominator with constant V of large magnitude.

    The kernels normalise O by the exact row sum plus, once per tile and thread, the
    16-bit rounding error of the thread's largest probability, while P.V uses every
    rounded probability.  When hundreds of keys share one probability value whose
    rounding is close to half a unit, the numerator carries that rounding hundreds of
    times and the denominator once per tile.  With V = c in every row the exact O is c,
    and the kernel's O is c·(Σ p̃)/(Σ p + corrections): its relative error is at most
    the unit roundoff u of the rounded probabilities, plus u for the 16-bit output,
    plus fp32 summation error (≤ 1e-4 at these lengths).  So |O - c| ≤ (2u + 1e-4)·|c|.
    That bound scales with |V|; the parity tolerance of 2e-2 is for V of unit size.
    The LSE uses the exact sum and meets the usual relative bound.
    """
    S = 1000  # several 128-key tiles and 256-row units, ragged tail
    q, k, v, scale = _equal_scores_case(pattern, S, D, dt)
    o, lse = run_gpu(q, k, v, causal, scale)
    o_ref, l_ref = attention_dense(q, k, v, scale, causal)
    u = _U16[dt]
    c = v.double()[0, 0, :, 0].numpy()  # per head
    bound = (2 * u + 1e-4) * np.abs(c)
    og = o.double().cpu().numpy()
    err = np.abs(og - o_ref)  # [1, S, H, D]
    worst = err.max(axis=(0, 1, 3))
    assert np.all(worst <= bound), f"{pattern} D={D} {dt}: |O - c| {worst} > bound {bound}"
    assert np.allclose(o_ref, c[None, None, :, None], rtol=1e-12, atol=0)
    lg = lse.double().cpu().numpy()
    rel = np.abs(lg - l_ref) / np.maximum(1.0, np.abs(l_ref))
    assert rel.max() <= 1e-3, f"LSE {rel.max()}"
