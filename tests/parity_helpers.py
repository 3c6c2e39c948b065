"""Shared helpers of the GPU parity tests: run the CUDA path, run the oracle, compare.

Tolerances (stated for fp16/bf16 inputs, fp32 accumulation):
  O   : max |O_gpu - O_ref| <= 2e-2 and mean |O_gpu - O_ref| <= 2e-3
  LSE : |LSE_gpu - LSE_ref| <= 1e-3 * max(1, |LSE_ref|)
The LSE bound is relative except near zero, where a relative error is
ill-conditioned (a causal row 0 has LSE = s_00, which may be ~0).
"""
from __future__ import annotations

import numpy as np
import torch

import scaled_dot_product_tcgen05_gb300 as pkg

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_REL = 1e-3


def compare(o_gpu, lse_gpu, o_ref, lse_ref, row_mask=None, what=""):
    """Element-wise comparison over the entries where the reference is not NaN."""
    o = o_gpu.float().cpu().numpy().astype(np.float64) if hasattr(o_gpu, "cpu") else o_gpu
    l = lse_gpu.cpu().numpy().astype(np.float64) if hasattr(lse_gpu, "cpu") else lse_gpu
    sel_o = ~np.isnan(o_ref)
    sel_l = ~np.isnan(lse_ref)
    assert sel_o.any() and sel_l.any(), "nothing to compare"
    d = np.abs(o[sel_o] - o_ref[sel_o])
    assert np.all(np.isfinite(o[sel_o])), f"{what}: non-finite O"
    lr, lg = lse_ref[sel_l], l[sel_l]
    both_inf = np.isneginf(lr) & np.isneginf(lg)
    with np.errstate(invalid="ignore"):  # -inf - -inf, masked by both_inf
        dl = np.where(both_inf, 0.0, np.abs(lg - lr) / np.maximum(1.0, np.abs(lr)))
    stats = dict(o_max=float(d.max()), o_mean=float(d.mean()), lse_rel=float(np.nanmax(dl)),
                 n_o=int(d.size), n_lse=int(dl.size))
    assert stats["o_max"] <= O_MAX_ABS, f"{what}: O max-abs {stats}"
    assert stats["o_mean"] <= O_MEAN_ABS, f"{what}: O mean-abs {stats}"
    assert stats["lse_rel"] <= LSE_REL, f"{what}: LSE {stats}"
    return stats


def run_gpu(q, k, v, causal, scale, cu_q=None, cu_k=None, stream=None, window=(-1, -1),
            global_q=0):
    """Copies host inputs to cuda:0, runs attn_fwd, checks the device status."""
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    cq = cu_q.to(dev) if cu_q is not None else None
    ck = cu_k.to(dev) if cu_k is not None else None
    o, lse = pkg.attn_fwd(qd, kd, vd, causal=causal, scale=scale, cu_seqlens_q=cq,
                          cu_seqlens_k=ck, stream=stream, window=window, global_q=global_q)
    st = pkg.attn_check(stream)
    assert st == pkg.ATTN_OK, pkg.status_string(st)
    return o, lse
