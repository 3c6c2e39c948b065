"""Failure detection without faulting a GPU.

Every device-side wait is bounded (ATTN_WAIT_TIMEOUT_MS); when one runs out the
kernel writes the error word, its roles drain and the CTA exits, so the
context stays usable and attn_check reports ATTN_ERR_DEVICE_TIMEOUT.  The
injected faults (ATTN_INJECT_FAULT) are a tile fill that is never issued (1:
block 0 of the forward kernels -- the CTA-pair kernel, and the single-CTA
kernel that ATTN_PAIR=0 selects -- skips its first K tile, block 0 of the
decode kernel its first fill, so a wait runs out) and an empty launch grid that
the launch itself rejects (2, decode only: ATTN_ERR_CUDA).  Neither traps,
faults or hangs the GPU.  The forward cases run units with more K/V tiles than
the loaders have stages, so a loader gives up in the middle of a unit and must
drain exactly the copies it issued; in the CTA-pair kernel the two softmax
warps of a row may give up at different points and must still meet at their
shared barrier.  Host-side failures (no device, bad arguments) are covered
without a GPU.
"""
import ctypes
import math
import os

import numpy as np
import pytest
import torch

import scaled_dot_product_tcgen05_gb300 as pkg
from oracle.sdpa_oracle import attention_decode, attention_dense
from parity_helpers import compare, run_gpu


class _env:
    """Set environment variables for the duration of a block."""

    def __init__(self, **kv):
        self.kv = kv

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in self.kv}
        os.environ.update({k: str(v) for k, v in self.kv.items()})

    def __exit__(self, *exc):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


# ------------------------------------------------------------------ host side
def test_host_failures_are_reported_without_a_device():
    """No CUDA device here: a well-formed call fails with ATTN_ERR_CUDA, argument errors
    are found before any CUDA call."""
    if torch.cuda.is_available():
        pytest.skip("needs a host without a CUDA device")
    lib = pkg.load_library()
    A = 0x10000
    def call(**kw):
        a = dict(q=A, k=A + 0x100, v=A + 0x200, o=A + 0x300, lse=A + 0x400, B=1, H=2, Sq=1,
                 Sk=128, D=128)
        a.update(kw)
        return lib.attn_fwd_decode(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"],
                                   a["Sq"], a["Sk"], a["D"], ctypes.c_float(0.1), 1, None,
                                   None, 0, 0, None)
    with _env(ATTN_INJECT_FAULT=2):
        assert call() == pkg.ATTN_ERR_CUDA        # cudaGetDevice fails: no device
        assert call(D=96) == pkg.ATTN_ERR_UNSUPPORTED  # checked before any CUDA call
    assert pkg.status_string(pkg.ATTN_ERR_DEVICE_TIMEOUT) != pkg.status_string(pkg.ATTN_OK)


# ------------------------------------------------------------------ device side
def _decode_case():
    g = torch.Generator().manual_seed(44)
    B, Sq, Sk, H, D = 2, 1, 1000, 4, 128
    q = torch.randn(B, Sq, H, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Sk, H, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Sk, H, D, generator=g).to(torch.bfloat16)
    return q, k, v


def _long_decode_case():
    """One query against a 65536-row cache: block 0 streams 8 fills through 4 stages."""
    g = torch.Generator().manual_seed(46)
    B, Sq, Sk, H, D = 1, 1, 65536, 1, 128
    q = torch.randn(B, Sq, H, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Sk, H, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Sk, H, D, generator=g).to(torch.bfloat16)
    return q, k, v


def _run_decode(q, k, v):
    dev = "cuda:0"
    o, lse = pkg.attn_decode(q.to(dev), k.to(dev), v.to(dev), causal=True,
                             scale=1 / math.sqrt(q.shape[-1]))
    return o, lse, pkg.attn_check()


@pytest.mark.gpu
@pytest.mark.parametrize("case", [_decode_case, _long_decode_case],
                         ids=["one_fill_per_block", "more_fills_than_stages"])
def test_bounded_wait_runs_out_and_the_context_stays_usable(case):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    q, k, v = case()
    with _env(ATTN_INJECT_FAULT=1, ATTN_WAIT_TIMEOUT_MS=200):
        _, _, st = _run_decode(q, k, v)
    assert st == pkg.ATTN_ERR_DEVICE_TIMEOUT, pkg.status_string(st)
    # the same call without the fault: correct results on the same context
    o, lse, st = _run_decode(q, k, v)
    assert st == pkg.ATTN_OK, pkg.status_string(st)
    o_ref, l_ref = attention_decode(q, k, v, None, 1 / math.sqrt(q.shape[-1]), True)
    compare(o, lse, o_ref, l_ref, what="decode after an injected timeout")


@pytest.mark.gpu
def test_rejected_launch_returns_cuda_error_and_clears_it():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    q, k, v = _decode_case()
    with _env(ATTN_INJECT_FAULT=2):
        with pytest.raises(pkg.AttnError) as e:
            _run_decode(q, k, v)
        assert e.value.status == pkg.ATTN_ERR_CUDA
    assert pkg.attn_check() == pkg.ATTN_OK  # nothing sticky left behind
    o, lse, st = _run_decode(q, k, v)
    assert st == pkg.ATTN_OK, pkg.status_string(st)
    o_ref, l_ref = attention_decode(q, k, v, None, 1 / math.sqrt(q.shape[-1]), True)
    compare(o, lse, o_ref, l_ref, what="decode after a rejected launch")


@pytest.mark.gpu
def test_debug_log_names_each_launch(capfd):
    """ATTN_DEBUG=1: one stderr line per launch; silent otherwise."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    q, k, v = _decode_case()
    _run_decode(q, k, v)
    assert "attn:" not in capfd.readouterr().err
    with _env(ATTN_DEBUG=1):
        _run_decode(q, k, v)
    err = capfd.readouterr().err
    grid, smem = pkg.last_launch()
    assert f"attn: attn_fwd_decode grid={grid} smem={smem}" in err, err


@pytest.mark.gpu
@pytest.mark.parametrize("D,pair", [(128, "1"), (64, "1"), (64, "0")],
                         ids=["cta_pair_d128", "cta_pair_d64", "single_cta_d64"])
def test_forward_bounded_wait_runs_out_and_the_context_stays_usable(D, pair, monkeypatch):
    """attn_fwd with a K tile that never arrives: every role of the affected CTAs winds
    down within the time limit, the call reports ATTN_ERR_DEVICE_TIMEOUT, and the same
    call without the fault then matches the oracle on the same context.  S = 1000 gives
    the first unit of pair / block 0 eight K/V tiles, more than either ring holds."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    monkeypatch.setenv("ATTN_PAIR", pair)
    g = torch.Generator().manual_seed(47 + D)
    B, S, H = 1, 1000, 4
    q, k, v = (torch.randn(B, S, H, D, generator=g).to(torch.bfloat16) for _ in range(3))
    scale = 1 / math.sqrt(D)
    dev = "cuda:0"
    with _env(ATTN_INJECT_FAULT=1, ATTN_WAIT_TIMEOUT_MS=200):
        pkg.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True, scale=scale)
        st = pkg.attn_check()
    assert st == pkg.ATTN_ERR_DEVICE_TIMEOUT, pkg.status_string(st)
    o, lse = run_gpu(q, k, v, True, scale)  # asserts ATTN_OK
    o_ref, l_ref = attention_dense(q, k, v, scale, True)
    compare(o, lse, o_ref, l_ref, what=f"forward D={D} after an injected timeout")
