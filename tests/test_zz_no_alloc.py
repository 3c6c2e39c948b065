"""attn_fwd_noalloc: the entry point for callers that cannot allocate device memory.

Such callers (a framework whose own allocator owns the GPU's memory, or a loop
that cannot accept cudaMalloc's implicit synchronisation) get the same kernel
with its scratch (the device error word) in a static device array.  This test
calls it through the C ABI twice in a row and checks each output against the
fp64 oracle and against the existing attn_fwd entry point, within the parity
tolerance.  The file name makes pytest collect it last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import scaled_dot_product_tcgen05_gb300 as pkg
from oracle.sdpa_oracle import attention_dense, attention_varlen
from parity_helpers import compare

pytestmark = pytest.mark.gpu


def _noalloc(lib):
    f = lib.attn_fwd_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, vp, vp, i, vp,
                  ctypes.POINTER(ctypes.c_int)]
    f.restype = i
    return f


CASES = [
    # (dense B, S, H, D, dtype, causal, varlen lengths or None)
    (2, 700, 4, 128, torch.bfloat16, True, None),
    (0, 0, 3, 64, torch.float16, False, [5, 300, 0, 129]),
]


@pytest.mark.parametrize("case", CASES, ids=["dense_bf16_causal", "varlen_fp16"])
def test_noalloc_matches_attn_fwd_on_two_calls(case):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B, S, H, D, dt, causal, lens = case
    lib = pkg.load_library()
    fn = _noalloc(lib)
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(77)
    if lens is None:
        shape = (B, S, H, D)
        cu = None
        Sq = Sk = S
    else:
        cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lens), 0)
        shape = (int(cu[-1]), H, D)
        B, Sq, Sk = len(lens), int(cu[-1]), int(cu[-1])
        cu = cu.to(dev)
    q_h, k_h, v_h = (torch.randn(shape, generator=g).to(dt) for _ in range(3))
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    scale = 1.0 / math.sqrt(D)
    if lens is None:
        o_or, l_or = attention_dense(q_h, k_h, v_h, scale, causal)
    else:
        cu_h = cu.cpu()
        o_or, l_or = attention_varlen(q_h, k_h, v_h, cu_h, cu_h, scale, causal)
    o_ref, lse_ref = pkg.attn_fwd(q, k, v, causal=causal, scale=scale, cu_seqlens_q=cu,
                                  cu_seqlens_k=cu)
    assert pkg.attn_check() == pkg.ATTN_OK
    o_ref64 = o_ref.double().cpu().numpy()
    l_ref64 = lse_ref.double().cpu().numpy()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        status = ctypes.c_int(-99)
        rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H,
                Sq, Sk, D, ctypes.c_float(scale), 1 if causal else 0,
                cu.data_ptr() if cu is not None else None,
                cu.data_ptr() if cu is not None else None,
                1 if dt == torch.bfloat16 else 0, stream, ctypes.byref(status))
        assert rc == pkg.ATTN_OK, pkg.status_string(rc)
        assert status.value == pkg.ATTN_OK, pkg.status_string(status.value)
        torch.cuda.synchronize()
        sel = ~np.isnan(o_ref64)
        if lens is not None:  # rows of the sequence without keys: O = 0, LSE = -inf in both
            sel_rows = torch.isneginf(lse_ref)
            assert torch.equal(torch.isneginf(lse), sel_rows)
        compare(o, lse, o_or, l_or, what=f"noalloc call {call} vs the oracle")
        compare(o, lse, np.where(sel, o_ref64, np.nan), l_ref64,
                what=f"noalloc call {call} vs attn_fwd")


def test_noalloc_rejects_bad_arguments_without_launching():
    lib = pkg.load_library()
    fn = _noalloc(lib)
    status = ctypes.c_int(-99)
    A = 0x10000
    assert fn(A, A, A, A, A, 1, 2, 128, 128, 96, ctypes.c_float(0.1), 0, None, None, 0, None,
              ctypes.byref(status)) == pkg.ATTN_ERR_UNSUPPORTED
    assert fn(A + 8, A, A, A, A, 1, 2, 128, 128, 64, ctypes.c_float(0.1), 0, None, None, 0,
              None, None) == pkg.ATTN_ERR_MISALIGNED
