"""Seeded synthetic inputs for the attention forward workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it without sharing any of the method.

Layouts (all contiguous, head dim innermost):
  dense  : q [B, Sq, H, D], k/v [B, Sk, H, D]
  varlen : q [total_q, H, D], k/v [total_k, H, D] with int32 cu_seqlens [B+1]

Every tensor is drawn head by head: the values of head ``h`` of tensor ``x``
(0 = Q, 1 = K, 2 = V) come from a CPU ``torch.Generator`` seeded with
``base_seed * 100_000 + x * 1000 + h``, as fp32 ``randn * std`` cast to the
storage dtype with round-to-nearest-even.  A subset of heads can therefore be
regenerated on its own, which keeps the long-context checks within host memory.
``base_seed = 1000 * workload_id + draw``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic attention problem (shapes, dtype, value distribution)."""

    name: str
    wid: int                  # workload id, part of the seed
    B: int                    # batch (dense) or number of sequences (varlen)
    H: int
    Sq: int                   # dense: per-batch length; varlen: 0 (taken from lengths)
    Sk: int
    D: int
    dtype: str                # "fp16" | "bf16"
    causal: bool
    std: tuple = (1.0, 1.0, 1.0)   # std of Q, K, V
    draw: int = 0
    varlen: bool = False
    len_range: tuple = (128, 4096)  # inclusive, varlen only
    window: tuple = (-1, -1)        # (left, right) band of keys per query; -1 = unbounded
    global_q: int = 0               # leading query rows that ignore the window
    decode: bool = False            # Sq new queries against a full KV cache of Sk rows
    backward: bool = False          # gradients dQ, dK, dV from a seeded dO
    fp8: bool = False               # Q, K, V quantised per tensor to e4m3 (dtype = output)

    @property
    def windowed(self) -> bool:
        return tuple(self.window) != (-1, -1) or self.global_q != 0

    @property
    def base_seed(self) -> int:
        return 1000 * self.wid + self.draw

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


def _wl(name, wid, B, H, S, D, dtype, causal, **kw):
    return Workload(name=name, wid=wid, B=B, H=H, Sq=S, Sk=S, D=D, dtype=dtype,
                    causal=causal, **kw)


def standard_workloads() -> dict:
    """The five workload families of the attention-forward study.

    1 tiny      B=1  H=2  S=128   D=64  fp16, causal and non-causal
    2 mha512    B=4  H=8  S=512   D=128 fp16, causal and non-causal
    3 mha2k     B=8  H=12 S=2048  D=64  fp16 and bf16, causal and non-causal,
                draw 0: N(0,1) everywhere; draw 1: Q,K ~ N(0,16), V ~ N(0,1)
    4 varlen    16 sequences, lengths uniform in [128, 4096], H=32 D=128 bf16 causal
    5 long      B=1 H=32 S=65536 (and 131072) D=128 bf16 causal
    6 window    B=1 H=32 S=131072 D=128 bf16 causal, sliding window of 4096 keys
                (the query and the 4095 before it) with 64 global query rows: the
                128K-context hybrid of page "长文本处理性能断层真相", §2.5
    8 backward  B=1 H=32 S=16384 D=128 bf16 causal: dQ, dK, dV from a seeded dO
    9 fp8       the long 64K causal problem with Q, K, V quantised to e4m3 (bf16 output)
    7 decode    KV-cache decode (page "长文本处理性能断层真相", §2.2): one new token
                per sequence against a 128K-token cache (B=1 H=32 D=128 bf16), and
                a batch of 16 sequences with 32K-token caches and 4 new tokens each
    """
    w = {}
    for c in (False, True):
        tag = "causal" if c else "full"
        w[f"tiny_{tag}"] = _wl(f"tiny_{tag}", 1, 1, 2, 128, 64, "fp16", c)
        w[f"mha512_{tag}"] = _wl(f"mha512_{tag}", 2, 4, 8, 512, 128, "fp16", c)
        for dt in ("fp16", "bf16"):
            w[f"mha2k_{dt}_{tag}"] = _wl(f"mha2k_{dt}_{tag}", 3, 8, 12, 2048, 64, dt, c)
            w[f"mha2k_{dt}_{tag}_peaked"] = _wl(f"mha2k_{dt}_{tag}_peaked", 3, 8, 12, 2048, 64,
                                                dt, c, std=(4.0, 4.0, 1.0), draw=1)
    w["varlen_causal"] = Workload(name="varlen_causal", wid=4, B=16, H=32, Sq=0, Sk=0, D=128,
                                  dtype="bf16", causal=True, varlen=True)
    w["long64k_causal"] = _wl("long64k_causal", 5, 1, 32, 65536, 128, "bf16", True)
    w["long128k_causal"] = _wl("long128k_causal", 5, 1, 32, 131072, 128, "bf16", True, draw=2)
    w["window128k_causal"] = _wl("window128k_causal", 6, 1, 32, 131072, 128, "bf16", True,
                                 window=(4095, 0), global_q=64)
    w["fp8_long64k_causal"] = _wl("fp8_long64k_causal", 9, 1, 32, 65536, 128, "bf16", True,
                                  fp8=True)
    w["bwd16k_causal"] = _wl("bwd16k_causal", 8, 1, 32, 16384, 128, "bf16", True, backward=True)
    w["decode128k_q1"] = Workload(name="decode128k_q1", wid=7, B=1, H=32, Sq=1, Sk=131072,
                                  D=128, dtype="bf16", causal=True, decode=True)
    w["decode32k_b16_q4"] = Workload(name="decode32k_b16_q4", wid=7, B=16, H=32, Sq=4,
                                     Sk=32768, D=128, dtype="bf16", causal=True, decode=True,
                                     draw=1)
    return w


def varlen_lengths(wl: Workload) -> torch.Tensor:
    """Sequence lengths of a varlen workload (int64, on the CPU)."""
    g = torch.Generator().manual_seed(wl.base_seed)
    lo, hi = wl.len_range
    return torch.randint(lo, hi + 1, (wl.B,), generator=g)


def cu_seqlens_from_lengths(lengths: Sequence[int]) -> torch.Tensor:
    """int32 prefix offsets [0, L0, L0+L1, ...]."""
    out = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    if len(lengths):
        out[1:] = torch.cumsum(torch.as_tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return out


def _draw_head(seed: int, rows: int, D: int, std: float, dtype) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, D, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def make_tensor(base_seed: int, which: int, shape_rows: Sequence[int], H: int, D: int,
                std: float, dtype, heads: Optional[Sequence[int]] = None,
                pin: bool = False) -> torch.Tensor:
    """Draw one [*shape_rows, H, D] tensor head by head (see module docstring).

    Heads not listed in ``heads`` are left as zeros (used to bound host time when
    only a few heads are checked); ``heads=None`` draws all of them.
    """
    rows = 1
    for r in shape_rows:
        rows *= r
    out = torch.zeros(rows, H, D, dtype=dtype, pin_memory=pin)
    for h in (range(H) if heads is None else heads):
        out[:, h, :] = _draw_head(base_seed * 100_000 + which * 1000 + h, rows, D, std, dtype)
    return out.view(*shape_rows, H, D)


def make_inputs(wl: Workload, heads: Optional[Sequence[int]] = None, pin: bool = False):
    """Return dict(q, k, v, cu_seqlens_q, cu_seqlens_k, lengths) on the CPU."""
    dt = DTYPES[wl.dtype]
    if wl.varlen:
        lengths = varlen_lengths(wl)
        cu = cu_seqlens_from_lengths(lengths.tolist())
        total = int(cu[-1])
        q_rows = k_rows = (total,)
    else:
        lengths = None
        cu = None
        q_rows, k_rows = (wl.B, wl.Sq), (wl.B, wl.Sk)
    q = make_tensor(wl.base_seed, 0, q_rows, wl.H, wl.D, wl.std[0], dt, heads, pin)
    k = make_tensor(wl.base_seed, 1, k_rows, wl.H, wl.D, wl.std[1], dt, heads, pin)
    v = make_tensor(wl.base_seed, 2, k_rows, wl.H, wl.D, wl.std[2], dt, heads, pin)
    out = dict(q=q, k=k, v=v, cu_seqlens_q=cu, cu_seqlens_k=cu, lengths=lengths)
    if wl.backward:  # the output gradient dO, tensor index 3, N(0, 1)
        out["do"] = make_tensor(wl.base_seed, 3, q_rows, wl.H, wl.D, 1.0, dt, heads, pin)
    return out


def sampled_heads_rows(wl: Workload, n_heads: int = 4, n_rows: int = 256):
    """Seeded sample of (heads, query rows) for checks the oracle cannot do in full.

    Rows always include 0 and Sq-1 plus ``n_rows - 2`` further distinct rows.
    """
    g = torch.Generator().manual_seed(1000 * wl.wid + 99)
    heads = sorted(torch.randperm(wl.H, generator=g)[:n_heads].tolist())
    S = wl.Sq
    n_rows = min(n_rows, S)
    inner = torch.randperm(max(S - 2, 0), generator=g)[: max(n_rows - 2, 0)] + 1
    rows = sorted(set([0, S - 1] + inner.tolist()))
    return heads, rows


def attention_flops(B: int, H: int, Sq: int, Sk: int, D: int, causal: bool) -> float:
    """FLOP count used for every TFLOP/s figure: 4*B*H*Sq*Sk*D, halved for causal.

    Two matmuls (Q K^T and P V) of 2*Sq*Sk*D flops each per (batch, head), as in
    the roofline worked example of the page "深度学习算子优化：从TFLOPS幻觉到
    FlashAttention实战", §2 (seq_len 2048, head_dim 64 -> about 1.07e9 per head).
    """
    f = 4.0 * B * H * Sq * Sk * D
    return f / 2.0 if causal else f


def varlen_flops(lengths: Sequence[int], H: int, D: int, causal: bool) -> float:
    """Sum over sequences of attention_flops(1, H, L, L, D, causal)."""
    return sum(attention_flops(1, H, int(L), int(L), D, causal) for L in lengths)


def visible_key_counts(Sq: int, Sk: int, causal: bool, window=(-1, -1), global_q: int = 0):
    """Number of keys each query row 0..Sq-1 of one sequence may see (int64 array).

    Used only to count the work of windowed problems (FLOPs = 4*D per visible
    (query, key) pair); row i >= global_q sees keys max(0, i-left) ..
    min(Sk-1, i+right), rows below global_q see all keys, causal caps at i.
    """
    import numpy as np
    i = np.arange(Sq, dtype=np.int64)
    wl, wr = window
    lo = np.zeros(Sq, dtype=np.int64)
    hi = np.full(Sq, Sk, dtype=np.int64)
    band = i >= global_q
    if wl >= 0:
        lo = np.where(band, np.maximum(0, i - wl), lo)
    if wr >= 0:
        hi = np.where(band, np.minimum(Sk, i + wr + 1), hi)
    if causal:
        hi = np.minimum(hi, i + 1)
    return np.maximum(0, hi - lo)


def window_flops(B: int, H: int, Sq: int, Sk: int, D: int, causal: bool, window=(-1, -1),
                 global_q: int = 0) -> float:
    """4 * D FLOPs per visible (query, key) pair, summed over rows, heads and batch."""
    return 4.0 * D * B * H * float(visible_key_counts(Sq, Sk, causal, window, global_q).sum())


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor e4m3 codes of a tensor and their scale (x ~ code * scale).

    The scale maps the largest magnitude to 448 (the e4m3 maximum); codes are
    torch's float8_e4m3fn rounding (nearest even).  Input generation only: the
    attention math sees the codes and the scale.
    """
    amax = float(x.abs().max()) if x.numel() else 1.0
    scale = (amax / 448.0) if amax > 0 else 1.0
    codes = (x.float() / scale).to(torch.float8_e4m3fn)
    return codes, scale
