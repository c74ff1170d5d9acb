"""Exact attention (FlashAttention-2 formulation) for GB300 / sm_103a.

The computation lives in ``libfa.so`` (hand-written CUDA: TMA, tcgen05 MMA
with tensor-memory accumulators, warp-specialised softmax), reached through
its C ABI (``include/fa.h``).  This package is the thin Python side: the
ctypes binding (``_lib``), convenience wrappers that allocate outputs with
PyTorch, the seeded input generators (``inputs``) and the build script.

PyTorch is used for device memory and streams only.  There is no CPU or
eager fallback: if the library is missing the calls raise.
"""
from __future__ import annotations

import math

from . import _lib

__all__ = ["attention_fwd", "attention_bwd", "attention_fwd_varlen", "attention_bwd_varlen",
           "hadamard_quant_fp8", "attention_fwd_fp8"]


def _default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def attention_fwd(q, k, v, causal: bool = False, scale: float | None = None, stream=None,
                  window: int | None = None):
    """Returns (O, LSE).  q [B,Hq,N,d], k/v [B,Hkv,N,d]: contiguous CUDA
    bf16/fp16 tensors; LSE is fp32 [B,Hq,N] (natural log).  ``window`` (with
    causal=True) limits row r to keys r - window + 1 .. r."""
    import torch
    B, Hq, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    sc = _default_scale(d) if scale is None else scale
    if window is None:
        _lib.fa_fwd(q, k, v, o, lse, causal, sc, stream)
    else:
        if not causal:
            raise ValueError("a sliding window is defined on top of the causal mask")
        _lib.fa_fwd_local(q, k, v, o, lse, window, sc, stream)
    return o, lse


def attention_bwd(q, k, v, o, lse, dO, causal: bool = False, scale: float | None = None,
                  workspace=None, stream=None, deterministic: bool = False, window: int | None = None):
    """Returns (dQ, dK, dV) from the forward's O and LSE and the incoming dO.

    ``deterministic=True`` forms dQ in a second pass over Q tiles instead of
    by atomic addition (bit-identical results from run to run)."""
    import torch
    B, Hq, N, d = q.shape
    if workspace is None:
        size_fn = _lib.fa_bwd_two_pass_workspace_bytes if deterministic else _lib.fa_bwd_workspace_bytes
        workspace = torch.empty(size_fn(B, Hq, N, d), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    sc = _default_scale(d) if scale is None else scale
    if window is not None:
        if not causal:
            raise ValueError("a sliding window is defined on top of the causal mask")
        _lib.fa_bwd_local(q, k, v, o, lse, dO, dq, dk, dv, window, sc, deterministic, workspace, stream)
    else:
        fn = _lib.fa_bwd_two_pass if deterministic else _lib.fa_bwd
        fn(q, k, v, o, lse, dO, dq, dk, dv, causal, sc, workspace, stream)
    return dq, dk, dv


def attention_fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int | None = None, causal: bool = False,
                         scale: float | None = None, window: int | None = None, stream=None):
    """Packed batch: sequence b is rows cu_seqlens[b] .. cu_seqlens[b+1]-1 of
    q [total,Hq,d] and k/v [total,Hkv,d] and attends only within itself.
    ``cu_seqlens`` is an int32 tensor [B+1] on the device.  Returns
    (O [total,Hq,d], LSE [Hq,total] fp32).  ``max_seqlen`` defaults to the
    longest sequence (read back from the device once)."""
    import torch
    total, Hq, d = q.shape
    if max_seqlen is None:
        max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item())
    if window is not None and not causal:
        raise ValueError("a sliding window is defined on top of the causal mask")
    o = torch.empty_like(q)
    lse = torch.empty((Hq, total), dtype=torch.float32, device=q.device)
    sc = _default_scale(d) if scale is None else scale
    _lib.fa_fwd_varlen(q, k, v, o, lse, cu_seqlens, max_seqlen, causal, sc, window or 0, stream)
    return o, lse


def attention_bwd_varlen(q, k, v, o, lse, dO, cu_seqlens, max_seqlen: int | None = None, causal: bool = False,
                         scale: float | None = None, window: int | None = None, deterministic: bool = False,
                         workspace=None, stream=None):
    """Gradients (dQ [total,Hq,d], dK, dV [total,Hkv,d]) of a packed batch
    from the forward's O and LSE and the incoming dO; arguments as
    ``attention_fwd_varlen``.  ``deterministic=True`` forms dQ in a second
    pass instead of by atomic addition."""
    import torch
    total, Hq, d = q.shape
    if max_seqlen is None:
        max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item())
    if window is not None and not causal:
        raise ValueError("a sliding window is defined on top of the causal mask")
    if workspace is None:
        workspace = torch.empty(_lib.fa_bwd_varlen_workspace_bytes(total, Hq, d, deterministic),
                                dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    sc = _default_scale(d) if scale is None else scale
    _lib.fa_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens, max_seqlen, causal, sc, deterministic,
                       workspace, window or 0, stream)
    return dq, dk, dv


def hadamard_quant_fp8(x, signs=None, stream=None):
    """Random-sign Hadamard rotation (if ``signs`` is given) and per-tensor
    e4m3 quantisation of a bf16 tensor [..., d].  Returns (x8, descale)."""
    import torch
    d = x.shape[-1]
    x8 = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device=x.device)
    descale = torch.empty(1, dtype=torch.float32, device=x.device)
    ws = torch.empty(_lib.fa_hadamard_quant_workspace_bytes(x.numel() // d, d), dtype=torch.uint8,
                     device=x.device)
    _lib.fa_hadamard_quant_fp8(x, signs, x8, descale, ws, stream)
    return x8, descale


def attention_fwd_fp8(q8, k8, v8, q_descale, k_descale, v_descale, causal: bool = False,
                      scale: float | None = None, stream=None):
    """FP8 forward: bf16 O and fp32 LSE from e4m3 Q, K, V and their descales."""
    import torch
    B, Hq, N, d = q8.shape
    o = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, device=q8.device)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q8.device)
    _lib.fa_fwd_fp8(q8, k8, v8, q_descale, k_descale, v_descale, o, lse, causal,
                    _default_scale(d) if scale is None else scale, stream)
    return o, lse
