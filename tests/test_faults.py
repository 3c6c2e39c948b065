"""Failure detection without faulting a GPU.

Every device-side wait is bounded (ATTN_WAIT_TIMEOUT_MS); when one runs out the
kernel writes the error word, its roles drain and the CTA exits, so the
context stays usable and attn_check reports ATTN_ERR_DEVICE_TIMEOUT.  The
injected faults (ATTN_INJECT_FAULT, honoured by attn_fwd_decode only) are a
tile fill that is never issued (1: a wait runs out) and an empty launch grid
that the launch itself rejects (2: ATTN_ERR_CUDA).  Neither traps, faults or
hangs the GPU.  Host-side failures (no device, bad arguments) are covered
without a GPU.
"""
import ctypes
import math
import os

import numpy as np
import pytest
import torch

import scaled_dot_product_tcgen05_gb300 as pkg
from oracle.sdpa_oracle import attention_decode
from parity_helpers import compare


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


def _run_decode(q, k, v):
    dev = "cuda:0"
    o, lse = pkg.attn_decode(q.to(dev), k.to(dev), v.to(dev), causal=True,
                             scale=1 / math.sqrt(q.shape[-1]))
    return o, lse, pkg.attn_check()


@pytest.mark.gpu
def test_bounded_wait_runs_out_and_the_context_stays_usable():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    q, k, v = _decode_case()
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
