"""ctypes binding of the C ABI in include/attn.h (argument marshalling only).

Every step of the attention forward runs in the CUDA library; this module only
checks shapes and dtypes, allocates outputs with torch, and passes raw device
pointers and the current CUDA stream.  If the library is missing the calls
raise: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Tuple

import torch

from .build_lib import LIB_PATH

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_MISALIGNED = -3
ATTN_ERR_CUDA = -4
ATTN_ERR_DEVICE_TIMEOUT = -5
ATTN_ERR_BAD_SEQLENS = -6

DTYPE_CODES = {torch.float16: 0, torch.bfloat16: 1}

EXPORTED = ("attn_fwd", "attn_check", "attn_status_string", "attn_num_sms",
            "attn_last_launch", "attn_release", "attn_fwd_noalloc", "attn_fwd_window",
            "attn_fwd_decode", "attn_decode_workspace", "attn_merge", "attn_bwd",
            "attn_bwd_workspace", "attn_fwd_fp8", "attn_fwd_fp8_workspace")

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class AttnError(RuntimeError):
    """A non-zero status returned by the CUDA library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (once) and return the CUDA library; raises if it was never built."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library {p} not built; run __graft_entry__.build() "
                               "(there is no CPU fallback)")
        lib = ctypes.CDLL(p)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp, i, vp]
        lib.attn_fwd.restype = i
        lib.attn_fwd_window.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, i, i, vp, vp,
                                        i, vp]
        lib.attn_fwd_window.restype = i
        lib.attn_fwd_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp,
                                        ctypes.c_size_t, i, vp]
        lib.attn_fwd_decode.restype = i
        lib.attn_decode_workspace.argtypes = [i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        lib.attn_decode_workspace.restype = i
        lib.attn_merge.argtypes = [vp, vp, i, i, i, i, i, vp, vp, i, vp]
        lib.attn_merge.restype = i
        lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp,
                                 vp, ctypes.c_size_t, i, vp]
        lib.attn_bwd.restype = i
        lib.attn_bwd_workspace.argtypes = [i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        lib.attn_bwd_workspace.restype = i
        lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, f, f, f, i, vp,
                                     ctypes.c_size_t, i, vp]
        lib.attn_fwd_fp8.restype = i
        lib.attn_fwd_fp8_workspace.argtypes = [i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        lib.attn_fwd_fp8_workspace.restype = i
        lib.attn_check.argtypes = [vp]
        lib.attn_check.restype = i
        lib.attn_status_string.argtypes = [i]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_num_sms.argtypes = []
        lib.attn_num_sms.restype = i
        lib.attn_last_launch.argtypes = [ctypes.POINTER(i), ctypes.POINTER(i)]
        lib.attn_last_launch.restype = i
        lib.attn_release.argtypes = []
        lib.attn_release.restype = i
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load_library().attn_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def attn_fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int,
                 Sq: int, Sk: int, D: int, scale: float, causal: bool, cu_q_ptr: int,
                 cu_k_ptr: int, dtype_code: int, stream: int) -> int:
    """Direct call of the C entry point with integer device pointers; returns the status."""
    return load_library().attn_fwd(q_ptr or None, k_ptr or None, v_ptr or None, o_ptr or None,
                                   lse_ptr or None, B, H, Sq, Sk, D, ctypes.c_float(scale),
                                   1 if causal else 0, cu_q_ptr or None, cu_k_ptr or None,
                                   dtype_code, stream or None)


def attn_fwd_window_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int,
                        H: int, Sq: int, Sk: int, D: int, scale: float, causal: bool,
                        window_left: int, window_right: int, global_q: int, cu_q_ptr: int,
                        cu_k_ptr: int, dtype_code: int, stream: int) -> int:
    """Direct call of the windowed C entry point; returns the status."""
    return load_library().attn_fwd_window(
        q_ptr or None, k_ptr or None, v_ptr or None, o_ptr or None, lse_ptr or None, B, H, Sq, Sk,
        D, ctypes.c_float(scale), 1 if causal else 0, int(window_left), int(window_right),
        int(global_q), cu_q_ptr or None, cu_k_ptr or None, dtype_code, stream or None)


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, causal: bool = False,
             scale: Optional[float] = None, cu_seqlens_q: Optional[torch.Tensor] = None,
             cu_seqlens_k: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
             lse: Optional[torch.Tensor] = None, window: Tuple[int, int] = (-1, -1),
             global_q: int = 0, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Fused attention forward on the GPU.  Returns (O, LSE).

    dense : q [B,Sq,H,D], k/v [B,Sk,H,D] -> O like q, LSE fp32 [B,H,Sq]
    varlen: q [Tq,H,D], k/v [Tk,H,D], int32 cu_seqlens [B+1] -> O like q, LSE [H,Tq]
    ``scale`` defaults to 1/sqrt(D).  ``causal`` keeps key j for query i iff j <= i
    (indices inside each sequence).  ``window = (left, right)`` keeps only keys
    i - left <= j <= i + right (-1: that side unbounded; causal needs right <= 0)
    for the query rows i >= ``global_q``; the first ``global_q`` rows of each
    sequence attend to every key (up to the diagonal when causal).  The default
    runs the ``attn_fwd`` entry point, any window or global rows
    ``attn_fwd_window``.  The launch is asynchronous on ``stream`` (default:
    torch's current stream); device-side errors are reported by
    :func:`attn_check`.
    """
    varlen = cu_seqlens_q is not None or cu_seqlens_k is not None
    if varlen and (cu_seqlens_q is None or cu_seqlens_k is None):
        raise ValueError("cu_seqlens_q and cu_seqlens_k must be given together")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype not in DTYPE_CODES:
            raise ValueError(f"{name} must be fp16 or bf16, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share one dtype")
    if varlen:
        if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
            raise ValueError("varlen q/k/v must be [total, H, D]")
        Tq, H, D = q.shape
        Tk = k.shape[0]
        if k.shape != (Tk, H, D) or v.shape != (Tk, H, D):
            raise ValueError("k/v shape mismatch")
        for name, c in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
            if c.dtype != torch.int32 or not c.is_cuda or c.dim() != 1 or not c.is_contiguous():
                raise ValueError(f"{name} must be a contiguous int32 CUDA vector")
        if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 1:
            raise ValueError("cu_seqlens_q/k must both have B+1 entries")
        B, Sq, Sk = cu_seqlens_q.numel() - 1, Tq, Tk
        lse_shape = (H, Tq)
    else:
        if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
            raise ValueError("dense q/k/v must be [B, S, H, D]")
        B, Sq, H, D = q.shape
        Sk = k.shape[1]
        if k.shape != (B, Sk, H, D) or v.shape != (B, Sk, H, D):
            raise ValueError("k/v shape mismatch")
        lse_shape = (B, H, Sq)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must match q")
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    elif tuple(lse.shape) != lse_shape or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError(f"lse must be a contiguous fp32 tensor of shape {lse_shape}")
    wl, wr = (int(x) for x in window)
    windowed = (wl, wr) != (-1, -1) or int(global_q) != 0
    with torch.cuda.device(q.device):
        cq = cu_seqlens_q.data_ptr() if varlen else 0
        ck = cu_seqlens_k.data_ptr() if varlen else 0
        if windowed:
            st = attn_fwd_window_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                     lse.data_ptr(), B, H, Sq, Sk, D, float(scale), causal, wl,
                                     wr, int(global_q), cq, ck, DTYPE_CODES[q.dtype],
                                     _stream_handle(stream))
        else:
            st = attn_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              lse.data_ptr(), B, H, Sq, Sk, D, float(scale), causal, cq, ck,
                              DTYPE_CODES[q.dtype], _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_window" if windowed else "attn_fwd")
    return out, lse


def _check_16bit(name, t):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in DTYPE_CODES:
        raise ValueError(f"{name} must be fp16 or bf16, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def decode_workspace_bytes(B: int, H: int, Sq: int, Sk: int, D: int) -> int:
    """Workspace bytes attn_fwd_decode needs for these sizes on the current device."""
    n = ctypes.c_size_t(0)
    st = load_library().attn_decode_workspace(B, H, Sq, Sk, D, ctypes.byref(n))
    if st != ATTN_OK:
        raise AttnError(st, "attn_decode_workspace")
    return int(n.value)


def attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, *,
                seqlens_k: Optional[torch.Tensor] = None, causal: bool = True,
                scale: Optional[float] = None, workspace: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention of Sq <= 16 new queries per sequence against a KV cache.

    q [B,Sq,H,D], k_cache/v_cache [B,Sk,H,D], optional int32 seqlens_k [B] (valid
    cache rows, default Sk).  The new queries are the last Sq positions of each
    sequence; with ``causal`` query t sees cache rows 0 .. L_b - Sq + t.  Returns
    (O [B,Sq,H,D], LSE fp32 [B,H,Sq]).  ``workspace`` (a CUDA uint8 tensor of at
    least :func:`decode_workspace_bytes`) is allocated when not given.
    """
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _check_16bit(name, t)
    if not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise ValueError("q, k_cache, v_cache must share one dtype")
    if q.dim() != 4 or k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("q must be [B,Sq,H,D] and k_cache/v_cache [B,Sk,H,D]")
    B, Sq, H, D = q.shape
    Sk = k_cache.shape[1]
    if k_cache.shape != (B, Sk, H, D):
        raise ValueError("k_cache/v_cache shape mismatch")
    if seqlens_k is not None and (seqlens_k.dtype != torch.int32 or not seqlens_k.is_cuda or
                                  seqlens_k.shape != (B,) or not seqlens_k.is_contiguous()):
        raise ValueError("seqlens_k must be a contiguous int32 CUDA vector of B entries")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        need = decode_workspace_bytes(B, H, Sq, Sk, D)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
        st = load_library().attn_fwd_decode(
            q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
            lse.data_ptr(), B, H, Sq, Sk, D, ctypes.c_float(scale), 1 if causal else 0,
            seqlens_k.data_ptr() if seqlens_k is not None else None,
            workspace.data_ptr() if need > 0 else None, workspace.numel(),
            DTYPE_CODES[q.dtype], _stream_handle(stream) or None)
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_decode")
    return out, lse


def attn_merge(o_parts: torch.Tensor, lse_parts: torch.Tensor, *,
               out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
               stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention over the union of disjoint key sets from per-set results.

    o_parts [P,B,S,H,D] (fp16/bf16), lse_parts fp32 [P,B,H,S] (stacked attn_fwd
    outputs; a varlen result is B = 1) -> (O [B,S,H,D], LSE [B,H,S]).
    """
    _check_16bit("o_parts", o_parts)
    if o_parts.dim() != 5:
        raise ValueError("o_parts must be [P, B, S, H, D]")
    P, B, S, H, D = o_parts.shape
    if (lse_parts.shape != (P, B, H, S) or lse_parts.dtype != torch.float32 or
            not lse_parts.is_cuda or not lse_parts.is_contiguous()):
        raise ValueError("lse_parts must be a contiguous fp32 CUDA tensor [P, B, H, S]")
    if out is None:
        out = torch.empty(o_parts.shape[1:], dtype=o_parts.dtype, device=o_parts.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=o_parts.device)
    with torch.cuda.device(o_parts.device):
        st = load_library().attn_merge(o_parts.data_ptr(), lse_parts.data_ptr(), P, B, S, H, D,
                                       out.data_ptr(), lse.data_ptr(),
                                       DTYPE_CODES[o_parts.dtype], _stream_handle(stream) or None)
    if st != ATTN_OK:
        raise AttnError(st, "attn_merge")
    return out, lse


def bwd_workspace_bytes(B: int, H: int, Sq: int, D: int, packed: bool = False) -> int:
    """Workspace bytes attn_bwd needs (packed: B sequences, Sq total query rows)."""
    n = ctypes.c_size_t(0)
    st = load_library().attn_bwd_workspace(B, H, Sq, D, 1 if packed else 0, ctypes.byref(n))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_workspace")
    return int(n.value)


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
             dout: torch.Tensor, lse: torch.Tensor, *, causal: bool = False,
             scale: Optional[float] = None, cu_seqlens_q: Optional[torch.Tensor] = None,
             cu_seqlens_k: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, dq: Optional[torch.Tensor] = None,
             dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None, stream=None):
    """Gradients (dQ, dK, dV) of :func:`attn_fwd` from dO, in the forward's layouts.

    dense : q, o, dout [B,Sq,H,D]; k, v [B,Sk,H,D]; lse fp32 [B,H,Sq]
    varlen: q, o, dout [Tq,H,D]; k, v [Tk,H,D]; int32 cu_seqlens [B+1]; lse [H,Tq]
    ``lse`` is what attn_fwd returned for the same inputs.  ``workspace`` (uint8
    CUDA tensor of at least :func:`bwd_workspace_bytes`) is allocated when not
    given.
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_16bit(name, t)
    if not (q.dtype == k.dtype == v.dtype == o.dtype == dout.dtype):
        raise ValueError("q, k, v, o, dout must share one dtype")
    varlen = cu_seqlens_q is not None or cu_seqlens_k is not None
    if varlen:
        if cu_seqlens_q is None or cu_seqlens_k is None:
            raise ValueError("cu_seqlens_q and cu_seqlens_k must be given together")
        if q.dim() != 3 or k.dim() != 3:
            raise ValueError("varlen q/o/dout must be [Tq,H,D], k/v [Tk,H,D]")
        Tq, H, D = q.shape
        Tk = k.shape[0]
        if k.shape != (Tk, H, D) or v.shape != k.shape or o.shape != q.shape or \
                dout.shape != q.shape:
            raise ValueError("shape mismatch")
        for name, c in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
            if c.dtype != torch.int32 or not c.is_cuda or c.dim() != 1 or not c.is_contiguous():
                raise ValueError(f"{name} must be a contiguous int32 CUDA vector")
        if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 1:
            raise ValueError("cu_seqlens_q/k must both have B+1 entries")
        B, Sq, Sk = cu_seqlens_q.numel() - 1, Tq, Tk
        lse_shape, ws_args = (H, Tq), (B, H, Tq, D, True)
    else:
        if q.dim() != 4 or k.dim() != 4:
            raise ValueError("dense layouts: q [B,Sq,H,D], k/v [B,Sk,H,D]")
        B, Sq, H, D = q.shape
        Sk = k.shape[1]
        if k.shape != (B, Sk, H, D) or v.shape != k.shape or o.shape != q.shape or \
                dout.shape != q.shape:
            raise ValueError("shape mismatch")
        lse_shape, ws_args = (B, H, Sq), (B, H, Sq, D)
    if tuple(lse.shape) != lse_shape or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError(f"lse must be a contiguous fp32 tensor of shape {lse_shape}")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        need = bwd_workspace_bytes(*ws_args)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(k) if dk is None else dk
        dv = torch.empty_like(v) if dv is None else dv
        st = load_library().attn_bwd(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Sq, Sk, D,
            ctypes.c_float(scale), 1 if causal else 0,
            cu_seqlens_q.data_ptr() if varlen else None,
            cu_seqlens_k.data_ptr() if varlen else None, workspace.data_ptr(),
            workspace.numel(), DTYPE_CODES[q.dtype], _stream_handle(stream) or None)
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


def fp8_workspace_bytes(B: int, H: int, Sk: int, D: int = 128) -> int:
    """Workspace bytes attn_fwd_fp8 needs for these sizes."""
    n = ctypes.c_size_t(0)
    st = load_library().attn_fwd_fp8_workspace(B, H, Sk, D, ctypes.byref(n))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_fp8_workspace")
    return int(n.value)


def attn_fwd_fp8(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, q_scale: float = 1.0,
                 k_scale: float = 1.0, v_scale: float = 1.0, causal: bool = False,
                 scale: Optional[float] = None, out_dtype=torch.bfloat16,
                 workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                 lse: Optional[torch.Tensor] = None, stream=None):
    """Attention forward on e4m3 inputs (dense, head dim 128).  Returns (O, LSE).

    q [B,Sq,H,128], k/v [B,Sk,H,128] as torch.float8_e4m3fn (or uint8 codes); the
    real values are code * scale per tensor.  O is ``out_dtype`` (bf16/fp16).
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.element_size() != 1:
            raise ValueError(f"{name} must be a contiguous 1-byte (e4m3) CUDA tensor")
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape:
        raise ValueError("q [B,Sq,H,D], k/v [B,Sk,H,D]")
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    if k.shape != (B, Sk, H, D):
        raise ValueError("k/v shape mismatch")
    if out_dtype not in DTYPE_CODES:
        raise ValueError("out_dtype must be fp16 or bf16")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        need = fp8_workspace_bytes(B, H, Sk, D)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        if out is None:
            out = torch.empty((B, Sq, H, D), dtype=out_dtype, device=q.device)
        if lse is None:
            lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
        st = load_library().attn_fwd_fp8(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, Sq,
            Sk, D, ctypes.c_float(scale), ctypes.c_float(q_scale), ctypes.c_float(k_scale),
            ctypes.c_float(v_scale), 1 if causal else 0, workspace.data_ptr(), workspace.numel(),
            DTYPE_CODES[out_dtype], _stream_handle(stream) or None)
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_fp8")
    return out, lse


def attn_check(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return load_library().attn_check(_stream_handle(stream))


def num_sms() -> int:
    return load_library().attn_num_sms()


def last_launch() -> Tuple[int, int]:
    g, s = ctypes.c_int(0), ctypes.c_int(0)
    st = load_library().attn_last_launch(ctypes.byref(g), ctypes.byref(s))
    if st != ATTN_OK:
        raise AttnError(st, "attn_last_launch")
    return g.value, s.value
