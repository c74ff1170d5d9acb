"""ctypes binding of libfa.so: the C ABI of include/fa.h, same names.

Argument marshalling only -- every step of the computation runs in the CUDA
kernels.  There is no fallback: if the library has not been built, or a call
returns an error status, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libfa.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_WORKSPACE, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(6)
FA_FP16, FA_BF16 = 0, 1

EXPORTS = (
    "fa_fwd", "fa_fwd_local", "fa_bwd_local", "fa_fwd_varlen", "fa_bwd_varlen", "fa_bwd_varlen_workspace_bytes",
    "fa_bwd", "fa_bwd_workspace_bytes", "fa_bwd_two_pass", "fa_bwd_two_pass_workspace_bytes",
    "fa_bwd_noalloc", "fa_hadamard_quant_fp8",
    "fa_hadamard_quant_workspace_bytes", "fa_fwd_fp8", "fa_get_device_status",
    "fa_selftest_bounded_wait", "fa_status_string", "fa_fwd_f32_out", "fa_probe_exp2", "fa_fwd_persistent",
)

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} ({status})")
        self.status = status


def load():
    """Load libfa.so (it must already be built: ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run __graft_entry__.build()); there is no fallback path")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, F, Z, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_long
        lib.fa_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, P]
        lib.fa_fwd_local.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, P]
        lib.fa_fwd_f32_out.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, P]
        lib.fa_fwd_persistent.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, P]
        lib.fa_bwd_local.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, P, Z, P]
        lib.fa_fwd_varlen.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, P]
        lib.fa_bwd_varlen.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, I, P, Z, P]
        lib.fa_bwd_varlen_workspace_bytes.argtypes = [I, I, I, I]
        lib.fa_bwd_varlen_workspace_bytes.restype = Z
        lib.fa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, P, Z, P]
        lib.fa_bwd_two_pass.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, P, Z, P]
        lib.fa_bwd_two_pass_workspace_bytes.argtypes = [I, I, I, I]
        lib.fa_bwd_two_pass_workspace_bytes.restype = Z
        lib.fa_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, P]
        lib.fa_bwd_workspace_bytes.argtypes = [I, I, I, I]
        lib.fa_bwd_workspace_bytes.restype = Z
        lib.fa_hadamard_quant_fp8.argtypes = [P, P, P, P, L, I, P, Z, P]
        lib.fa_hadamard_quant_workspace_bytes.argtypes = [L, I]
        lib.fa_hadamard_quant_workspace_bytes.restype = Z
        lib.fa_fwd_fp8.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P]
        lib.fa_get_device_status.argtypes = [P]
        lib.fa_selftest_bounded_wait.argtypes = [I, P]
        lib.fa_probe_exp2.argtypes = [P, I, I, P]
        lib.fa_probe_exp2.restype = ctypes.c_longlong
        lib.fa_status_string.argtypes = [I]
        lib.fa_status_string.restype = ctypes.c_char_p
        for name in ("fa_fwd", "fa_fwd_local", "fa_fwd_f32_out", "fa_fwd_persistent", "fa_bwd_local", "fa_fwd_varlen", "fa_bwd_varlen",
                     "fa_bwd", "fa_bwd_two_pass", "fa_bwd_noalloc", "fa_hadamard_quant_fp8", "fa_fwd_fp8",
                     "fa_get_device_status", "fa_selftest_bounded_wait"):
            getattr(lib, name).restype = I
        _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != FA_OK:
        msg = load().fa_status_string(status).decode()
        raise FAError(fn, status, msg)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float16:
        return FA_FP16
    raise TypeError(f"unsupported element type {t.dtype}")


def _need(name, t, dtypes=()):
    """Refuses a tensor the C call cannot take: the library receives bare
    pointers, so a wrong element type or a strided view would be read as
    something else without any error."""
    if t is None:
        return
    if dtypes and t.dtype not in dtypes:
        raise TypeError(f"{name}: element type {t.dtype}, expected {' or '.join(str(x) for x in dtypes)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: tensor must be contiguous")


def _io16(q, lse=None, f32=(), **same):
    """Checks a 16-bit call's tensors (q's element type for `same`, fp32
    for lse and `f32`) and returns q's type code."""
    import torch
    code = _dtype_code(q)
    _need("q", q)
    for name, t in same.items():
        _need(name, t, (q.dtype,))
    for name, t in (("lse", lse),) + tuple(f32):
        _need(name, t, (torch.float32,))
    return code


def _dims(q, k):
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    return B, Hq, Hkv, N, d


def fa_fwd(q, k, v, o, lse, causal: bool, scale: float, stream=None):
    """O and LSE for q [B,Hq,N,d], k/v [B,Hkv,N,d] (contiguous CUDA tensors)."""
    B, Hq, Hkv, N, d = _dims(q, k)
    code = _io16(q, lse, k=k, v=v, o=o)
    _check("fa_fwd", load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d,
                                   int(causal), float(scale), code, _stream(stream)))


def fa_fwd_persistent(q, k, v, o, lse, causal: bool, scale: float, stream=None):
    """fa_fwd as the persistent kernel (dynamic block schedule); same results."""
    B, Hq, Hkv, N, d = _dims(q, k)
    code = _io16(q, lse, k=k, v=v, o=o)
    _check("fa_fwd_persistent", load().fa_fwd_persistent(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq,
                                                         Hkv, N, d, int(causal), float(scale), code,
                                                         _stream(stream)))


def fa_fwd_f32_out(q, k, v, o_f32, lse, causal: bool, scale: float, stream=None):
    """fa_fwd with O written in fp32 (o_f32 [B,Hq,N,d] float32): the
    normalised accumulator before rounding to the input type."""
    B, Hq, Hkv, N, d = _dims(q, k)
    code = _io16(q, lse, f32=(("o_f32", o_f32),), k=k, v=v)
    _check("fa_fwd_f32_out", load().fa_fwd_f32_out(_ptr(q), _ptr(k), _ptr(v), _ptr(o_f32), _ptr(lse), B, Hq, Hkv,
                                                   N, d, int(causal), float(scale), code, _stream(stream)))


def fa_fwd_local(q, k, v, o, lse, window: int, scale: float, stream=None):
    """Causal sliding-window forward: row r sees keys r - window + 1 .. r."""
    B, Hq, Hkv, N, d = _dims(q, k)
    code = _io16(q, lse, k=k, v=v, o=o)
    _check("fa_fwd_local", load().fa_fwd_local(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d,
                                               int(window), float(scale), code, _stream(stream)))


def fa_bwd_local(q, k, v, o, lse, dO, dq, dk, dv, window: int, scale: float, deterministic: bool, workspace,
                 stream=None):
    B, Hq, Hkv, N, d = _dims(q, k)
    code = _io16(q, lse, k=k, v=v, o=o, dO=dO, dq=dq, dk=dk, dv=dv)
    _need("workspace", workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("fa_bwd_local", load().fa_bwd_local(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d,
        int(window), float(scale), code, int(bool(deterministic)), _ptr(workspace), ws_bytes,
        _stream(stream)))


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens, max_seqlen: int, causal: bool, scale: float, window: int = 0,
                  stream=None):
    """Packed sequences: q/o [total,Hq,d], k/v [total,Hkv,d], lse [Hq,total],
    cu_seqlens int32 [B+1] on the device."""
    import torch
    total, Hq, d = q.shape
    Hkv = k.shape[1]
    B = cu_seqlens.numel() - 1
    code = _io16(q, lse, k=k, v=v, o=o)
    _need("cu_seqlens", cu_seqlens, (torch.int32,))
    _check("fa_fwd_varlen", load().fa_fwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens), B, int(max_seqlen), total, Hq, Hkv, d,
        int(causal), int(window), float(scale), code, _stream(stream)))


def fa_bwd_varlen_workspace_bytes(total: int, Hq: int, d: int, deterministic: bool) -> int:
    return int(load().fa_bwd_varlen_workspace_bytes(total, Hq, d, int(bool(deterministic))))


def fa_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens, max_seqlen: int, causal: bool, scale: float,
                  deterministic: bool, workspace, window: int = 0, stream=None):
    import torch
    total, Hq, d = q.shape
    Hkv = k.shape[1]
    B = cu_seqlens.numel() - 1
    code = _io16(q, lse, k=k, v=v, o=o, dO=dO, dq=dq, dk=dk, dv=dv)
    _need("cu_seqlens", cu_seqlens, (torch.int32,))
    _need("workspace", workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("fa_bwd_varlen", load().fa_bwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_seqlens),
        B, int(max_seqlen), total, Hq, Hkv, d, int(causal), int(window), float(scale), code,
        int(bool(deterministic)), _ptr(workspace), ws_bytes, _stream(stream)))


def fa_bwd_workspace_bytes(B: int, Hq: int, N: int, d: int) -> int:
    return int(load().fa_bwd_workspace_bytes(B, Hq, N, d))


def fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, causal: bool, scale: float, workspace, stream=None):
    B, Hq, Hkv, N, d = _dims(q, k)
    code = _io16(q, lse, k=k, v=v, o=o, dO=dO, dq=dq, dk=dk, dv=dv)
    _need("workspace", workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("fa_bwd", load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                                   _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, int(causal), float(scale),
                                   code, _ptr(workspace), ws_bytes, _stream(stream)))


def fa_bwd_two_pass_workspace_bytes(B: int, Hq: int, N: int, d: int) -> int:
    return int(load().fa_bwd_two_pass_workspace_bytes(B, Hq, N, d))


def fa_bwd_two_pass(q, k, v, o, lse, dO, dq, dk, dv, causal: bool, scale: float, workspace, stream=None):
    """Deterministic backward: dQ from a second pass over Q tiles, no atomics."""
    B, Hq, Hkv, N, d = _dims(q, k)
    code = _io16(q, lse, k=k, v=v, o=o, dO=dO, dq=dq, dk=dk, dv=dv)
    _need("workspace", workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("fa_bwd_two_pass", load().fa_bwd_two_pass(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv,
        N, d, int(causal), float(scale), code, _ptr(workspace), ws_bytes, _stream(stream)))


def fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, causal: bool, scale: float, stream=None):
    """fa_bwd using the library's built-in scratch buffer instead of a
    caller workspace: for callers that cannot allocate device memory.  Calls
    that may overlap on the GPU race on that buffer."""
    B, Hq, Hkv, N, d = _dims(q, k)
    code = _io16(q, lse, k=k, v=v, o=o, dO=dO, dq=dq, dk=dk, dv=dv)
    _check("fa_bwd_noalloc", load().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO),
                                                   _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, int(causal),
                                                   float(scale), code, _stream(stream)))


def fa_hadamard_quant_workspace_bytes(rows: int, d: int) -> int:
    return int(load().fa_hadamard_quant_workspace_bytes(rows, d))


def _byte_types():
    import torch
    return (torch.float8_e4m3fn, torch.uint8)


def fa_hadamard_quant_fp8(x, signs, x8, descale, workspace, stream=None):
    """x bf16 (the only input type of the C call), x8 e4m3 bytes, signs and
    descale fp32."""
    import torch
    _need("x", x, (torch.bfloat16,))
    _need("signs", signs, (torch.float32,))
    _need("x8", x8, _byte_types())
    _need("descale", descale, (torch.float32,))
    _need("workspace", workspace)
    d = x.shape[-1]
    rows = x.numel() // d
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("fa_hadamard_quant_fp8", load().fa_hadamard_quant_fp8(
        _ptr(x), _ptr(signs), _ptr(x8), _ptr(descale), rows, d, _ptr(workspace), ws_bytes,
        _stream(stream)))


def fa_fwd_fp8(q8, k8, v8, q_descale, k_descale, v_descale, o, lse, causal: bool, scale: float,
               stream=None):
    import torch
    B, Hq, Hkv, N, d = _dims(q8, k8)
    for name, t in (("q8", q8), ("k8", k8), ("v8", v8)):
        _need(name, t, _byte_types())
    for name, t in (("q_descale", q_descale), ("k_descale", k_descale), ("v_descale", v_descale), ("lse", lse)):
        _need(name, t, (torch.float32,))
    _need("o", o, (torch.bfloat16,))
    _check("fa_fwd_fp8", load().fa_fwd_fp8(
        _ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_descale), _ptr(k_descale), _ptr(v_descale), _ptr(o),
        _ptr(lse), B, Hq, Hkv, N, d, int(causal), float(scale), _stream(stream)))


def fa_get_device_status(stream=None) -> int:
    """FA_OK, or FA_ERR_TIMEOUT if a bounded device wait ran out (clears it)."""
    return int(load().fa_get_device_status(_stream(stream)))


def fa_selftest_bounded_wait(timeout_us: int, stream=None):
    _check("fa_selftest_bounded_wait", load().fa_selftest_bounded_wait(int(timeout_us), _stream(stream)))


def fa_probe_exp2(sink, blocks: int, iters: int, stream=None) -> int:
    """Launches the exp2 throughput probe; returns the exp2 evaluations it
    performs.  sink: float32 CUDA tensor of at least blocks * 256 elements."""
    if sink.numel() < blocks * 256:
        raise ValueError("sink too small")
    n = load().fa_probe_exp2(_ptr(sink), int(blocks), int(iters), _stream(stream))
    if n < 0:
        raise FAError("fa_probe_exp2", FA_ERR_INVALID_ARG, "invalid arguments or launch failure")
    return int(n)
