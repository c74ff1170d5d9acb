"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and the oracle shares no
code with that path: inputs reach both sides from the seeded generators only.

The arithmetic lives in ``fa_oracle.c`` (plain C, fp64, OpenMP over rows);
this module compiles it with gcc on first use and marshals numpy arrays.

Functions and the passages they follow:

* ``attention_fwd`` -- O = softmax(scale Q K^T [+causal mask]) V and the
  row log-sum-exp L ("6.2 FlashAttention V2 chi tiet", section 6.1 pseudocode;
  blog.csdn.net FlashAttention-2 page, 3.1.1 forward formula analysis).
* ``attention_fwd_rows`` -- the same, for selected (b, h, r) rows.
* ``attention_bwd`` / ``attention_bwd_group`` -- analytic gradients with
  D = rowsum(dO o O) (blog.csdn.net page, 3.1.2 backward formula analysis;
  Vietnamese page section 7.3), dK/dV summed over grouped query heads (the
  blog's MQA/GQA paragraph).
* ``hadamard`` / ``e4m3_round`` -- random-sign Hadamard rotation and the OCP
  e4m3 grid used by the FP8 path (FlashAttention-3 summary page, FP8 and
  incoherent processing section).
* ``mx_e4m3`` / ``fp8_bwd_model`` -- block-scaled e4m3 quantisation (one
  power-of-two scale per 32 entries along a product's reduction axis) and a
  model of the backward with its five products on quantised operands: the
  numerical basis of an FP8 backward (the pages report the FP8 forward only).

Every function is pinned by the CPU tests in ``tests/test_oracle.py`` against
closed forms, finite differences, library routines and the page's two-block
worked recurrence.  The FP8 *error level* is parity unpinned by the pages (they
give only a ratio); see ``fp8_reference``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into oracle/_build/liboracle.so (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            L = ctypes.c_long
            lib.oracle_fwd.argtypes = [P, P, P, P, P, L, L, L, L, L, ctypes.c_int, L, ctypes.c_double]
            lib.oracle_fwd_rows.argtypes = [P, P, P, P, L, P, P, L, L, L, L, L, ctypes.c_int, L, ctypes.c_double]
            lib.oracle_bwd_group.argtypes = [P, P, P, P, L, L, P, P, P, L, L, L, L, L, ctypes.c_int, L, ctypes.c_double]
            lib.oracle_bwd.argtypes = [P, P, P, P, P, P, P, L, L, L, L, L, ctypes.c_int, L, ctypes.c_double]
            lib.oracle_hadamard.argtypes = [P, P, P, L, L]
            lib.oracle_e4m3_round.argtypes = [P, P, L]
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            lib.oracle_set_threads.restype = None
            lib.oracle_get_threads.restype = ctypes.c_int
            for name in ("oracle_fwd", "oracle_fwd_rows", "oracle_bwd_group",
                         "oracle_bwd", "oracle_hadamard", "oracle_e4m3_round"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def set_threads(n: int) -> int:
    """Threads the oracle's loops use from now on (n < 1: all host
    processors); returns the count in effect.  Results do not depend on it."""
    lib = _load()
    lib.oracle_set_threads(int(n))
    return int(lib.oracle_get_threads())


def _f64(x) -> np.ndarray:
    """Widen to a C-contiguous float64 array (torch tensors are accepted)."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").float().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, name: str):
    if rc != 0:
        raise ValueError(f"{name}: invalid arguments (code {rc})")


def _shapes(q, k):
    B, Hq, N, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if (Bk, Nk, dk) != (B, N, d) or Hq % Hkv:
        raise ValueError("q/k shapes disagree")
    return B, Hq, Hkv, N, d


def attention_fwd(q, k, v, causal: bool, scale: float, window: int = 0):
    """Return (O, L) in fp64; q [B,Hq,N,d], k/v [B,Hkv,N,d].  ``window`` > 0
    additionally hides key c from query r unless r - c < window."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, N, d = _shapes(q, k)
    o = np.empty_like(q)
    lse = np.empty((B, Hq, N), dtype=np.float64)
    _check(_load().oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                              B, Hq, Hkv, N, d, int(causal), int(window), float(scale)), "oracle_fwd")
    return o, lse


def attention_fwd_rows(q, k, v, rows, causal: bool, scale: float, window: int = 0):
    """O and L for the listed (b, h, r) rows only; returns ([n,d], [n])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, N, d = _shapes(q, k)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = rows.shape[0]
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    _check(_load().oracle_fwd_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(rows), n,
                                   _ptr(o), _ptr(lse), B, Hq, Hkv, N, d,
                                   int(causal), int(window), float(scale)), "oracle_fwd_rows")
    return o, lse


def attention_bwd(q, k, v, dO, causal: bool, scale: float, window: int = 0):
    """Return (dQ, dK, dV) in fp64 for loss = sum(dO o O)."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, Hq, Hkv, N, d = _shapes(q, k)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    _check(_load().oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq),
                              _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d,
                              int(causal), int(window), float(scale)), "oracle_bwd")
    return dq, dk, dv


def attention_bwd_group(q, k, v, dO, b: int, g: int, causal: bool, scale: float, window: int = 0):
    """Gradients of one (batch b, key/value head g) group.

    Returns dq [G,N,d] for query heads g*G..g*G+G-1 and dk, dv [N,d].
    """
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, Hq, Hkv, N, d = _shapes(q, k)
    G = Hq // Hkv
    dq = np.empty((G, N, d), dtype=np.float64)
    dk = np.empty((N, d), dtype=np.float64)
    dv = np.empty((N, d), dtype=np.float64)
    _check(_load().oracle_bwd_group(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), int(b),
                                    int(g), _ptr(dq), _ptr(dk), _ptr(dv), B, Hq,
                                    Hkv, N, d, int(causal), int(window), float(scale)),
           "oracle_bwd_group")
    return dq, dk, dv


def hadamard(x, signs=None):
    """(x o s) H_d / sqrt(d) along the last axis (dense Sylvester product)."""
    x = _f64(x)
    d = x.shape[-1]
    rows = x.size // d
    out = np.empty_like(x)
    s = None if signs is None else _f64(signs).reshape(d)
    _check(_load().oracle_hadamard(_ptr(x), None if s is None else _ptr(s),
                                   _ptr(out), rows, d), "oracle_hadamard")
    return out


def e4m3_round(x):
    """Round to the e4m3fn grid (ties to even), saturating at +-448."""
    x = _f64(x)
    out = np.empty_like(x)
    _check(_load().oracle_e4m3_round(_ptr(x), _ptr(out), x.size), "oracle_e4m3_round")
    return out


def fp8_dequantized(q, k, v, signs):
    """Q, K, V as the FP8 path sees them: Q and K rotated by the random-sign
    Hadamard (if ``signs`` is not None), each tensor quantised per tensor to
    e4m3 with sigma = amax / 448 and dequantised (fp64).

    The e4m3 code of a value is an integer decided by floating point, so it
    is decided in the precision the FP8 path uses, fp32 (the pages fix
    none): with c = 1/sqrt(d) for a rotated tensor (1 otherwise) and x' the
    value before that factor (the unnormalised transform, or the input),
    amax = fl32(max |x'| * c), and the code is the nearest e4m3 value (ties
    to even, saturating) of fl32(fl32(x' * c) * fl32(448 / amax)); sigma =
    fl32(amax / 448).  Rounding x / sigma in fp64 instead splits exact ties
    the other way: for 16-bit inputs without the rotation x * 448 / amax
    often lies exactly on an e4m3 midpoint, which the fp64 quotient by the
    rounded sigma misses by an ulp.

    Each tensor is handled one leading slice at a time, in two passes (the
    amax over all slices, then the rounding of each slice; the rotation and
    the rounding are per row), so the host memory needed is the fp64 output
    plus one slice."""
    f32 = np.float32

    def qdq(x, rotate: bool):
        d = x.shape[-1]
        c = f32(1.0 / np.sqrt(d)) if rotate else f32(1.0)

        def part(i):  # x' in fp32
            if rotate:
                return (hadamard(x[i], signs) * np.sqrt(d)).astype(f32)
            return _f64(x[i]).astype(f32)

        amax = f32(max(f32(np.abs(part(i)).max()) for i in range(x.shape[0])) * c)
        out = np.empty(tuple(x.shape), dtype=np.float64)
        if amax == 0.0:
            out[...] = 0.0
            return out
        inv = f32(448.0) / amax
        sigma = float(amax / f32(448.0))
        for i in range(x.shape[0]):
            t = (part(i) * c) * inv  # two fp32 products, each rounded to nearest
            out[i] = e4m3_round(t.astype(np.float64)) * sigma
        return out

    rot = signs is not None
    return qdq(q, rot), qdq(k, rot), qdq(v, False)


def fp8_reference(q, k, v, signs, causal: bool, scale: float):
    """Diagnostic model of the FP8 path's input quantisation.

    Q and K are rotated by the random-sign Hadamard (if ``signs`` is not
    None), then Q, K and V are each quantised per tensor to e4m3 with
    sigma = amax / 448, dequantised, and fed to the exact fp64 attention.
    The rotation is orthogonal, so without quantisation this returns exactly
    ``attention_fwd(q, k, v)``.  It separates the error of input
    quantisation from that of a kernel; the error level itself is parity
    unpinned by the pages, which report only a 2.6x ratio.
    """
    return attention_fwd(*fp8_dequantized(q, k, v, signs), causal, scale)


def mx_e4m3(x, axis: int, block: int = 32):
    """Block-scaled e4m3 quantisation along ``axis``: every run of ``block``
    consecutive entries along that axis (the last run may be shorter) shares
    one power-of-two scale 2^e, the smallest with max|x| <= 448 * 2^e, so no
    entry saturates; each entry becomes 2^e * e4m3(x / 2^e).  A block of
    zeros keeps scale 1.  Exponents are limited to the 8-bit exponent-only
    scale range [-127, 127].

    This is the operand format of a block-scaled FP8 product: one scale per
    32 entries along the product's reduction axis (the blocked counterpart of
    the per-tensor scaling in the FlashAttention-3 summary page, FP8 and
    incoherent processing section).  Returns (dequantised x, exponents), the
    exponents with ``axis`` shortened to ceil(n / block)."""
    x = _f64(x)
    xm = np.moveaxis(x, axis, -1)
    n = xm.shape[-1]
    nb = -(-n // block)
    out = np.empty_like(xm)
    exps = np.zeros(xm.shape[:-1] + (nb,), dtype=np.int64)
    for j in range(nb):
        blk = xm[..., j * block:(j + 1) * block]
        amax = np.abs(blk).max(axis=-1)
        e = np.zeros(amax.shape, dtype=np.int64)
        nz = amax > 0
        if nz.any():
            _, ex = np.frexp(amax[nz] / 448.0)   # first guess, then exact fix-up
            ev = ex.astype(np.int64)
            ev = np.where(amax[nz] > np.ldexp(448.0, ev), ev + 1, ev)
            ev = np.where(amax[nz] <= np.ldexp(448.0, ev - 1), ev - 1, ev)
            e[nz] = np.clip(ev, -127, 127)
        sc = np.ldexp(1.0, e)[..., None]
        out[..., j * block:(j + 1) * block] = e4m3_round(blk / sc) * sc
        exps[..., j] = e
    return np.moveaxis(out, -1, axis), np.moveaxis(exps, -1, axis)


def fp8_bwd_model(q, k, v, dO, causal: bool, scale: float, mode="mx32", signs=None,
                  products=("S", "dP", "dV", "dK", "dQ")):
    """Model of an FP8 backward: the gradients of ``attention_bwd`` with the
    operands of all five products of the backward step list (blog.csdn.net
    FlashAttention-2 page, 3.1.2: S = Q K^T, dP = dO V^T, dV = P^T dO,
    dK = dS^T Q, dQ = dS K) quantised to e4m3 before an exact fp64 product.

    mode: None -- no quantisation (equals ``attention_bwd``);
          "mx32" -- ``mx_e4m3`` along each product's reduction axis (d for S
          and dP, queries for dV and dK, keys for dQ);
          "tensor" -- one scale per operand matrix, sigma = amax / 448 of that
          matrix (the most favourable per-tensor choice: a kernel knows the
          amax of P or dS only after forming them).
    P = exp(S - L) uses L of the same quantised S, D = rowsum(dO o O) with
    O = P V; ``signs`` rotates Q and K by the random-sign Hadamard first and
    rotates dQ, dK back (the rotation is orthogonal, so mode None stays
    exact).  ``products`` names the products that take quantised operands
    (the others stay exact), to attribute the error.  Returns (dQ, dK, dV)
    in fp64."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, Hq, Hkv, N, d = _shapes(q, k)
    G = Hq // Hkv

    unknown = set(products) - {"S", "dP", "dV", "dK", "dQ"}
    if unknown:
        raise ValueError(f"unknown products {sorted(unknown)}")

    def qz(x, axis, product):
        if mode is None or product not in products:
            return x
        if mode == "mx32":
            return mx_e4m3(x, axis)[0]
        if mode == "tensor":
            sigma = np.abs(x).max() / 448.0
            return x if sigma == 0.0 else e4m3_round(x / sigma) * sigma
        raise ValueError(f"unknown mode {mode!r}")

    if signs is not None:
        q, k = hadamard(q, signs), hadamard(k, signs)
    keep = np.tril(np.ones((N, N), dtype=bool)) if causal else np.ones((N, N), dtype=bool)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            Q, K, V, dOh = q[b, h], k[b, g], v[b, g], dO[b, h]
            S = scale * (qz(Q, 1, "S") @ qz(K, 1, "S").T)
            S = np.where(keep, S, -np.inf)
            m = S.max(axis=1, keepdims=True)
            L = m + np.log(np.exp(S - m).sum(axis=1, keepdims=True))
            P = np.exp(S - L)
            D = (dOh * (P @ V)).sum(axis=1, keepdims=True)
            dP = qz(dOh, 1, "dP") @ qz(V, 1, "dP").T
            dS = P * (dP - D)
            dv[b, g] += qz(P, 0, "dV").T @ qz(dOh, 0, "dV")
            dk[b, g] += scale * (qz(dS, 0, "dK").T @ qz(Q, 0, "dK"))
            dq[b, h] = scale * (qz(dS, 1, "dQ") @ qz(K, 0, "dQ"))
    if signs is not None:
        s = _f64(signs).reshape(d)
        dq, dk = hadamard(dq) * s, hadamard(dk) * s
    return dq, dk, dv


def _segments(cu):
    cu = [int(x) for x in (cu.tolist() if hasattr(cu, "tolist") else cu)]
    return [(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]


def attention_fwd_varlen(q, k, v, cu_seqlens, causal: bool, scale: float, window: int = 0):
    """Packed sequences (token-major q [total,Hq,d], k/v [total,Hkv,d]):
    every sequence attends only within itself, so this is attention_fwd on
    each sequence in turn.  Returns O [total,Hq,d] and L [Hq,total]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    total, Hq, d = q.shape
    o = np.zeros_like(q)
    lse = np.zeros((Hq, total), dtype=np.float64)
    for a, b in _segments(cu_seqlens):
        if b == a:
            continue
        ob, lb = attention_fwd(q[a:b].transpose(1, 0, 2)[None], k[a:b].transpose(1, 0, 2)[None],
                               v[a:b].transpose(1, 0, 2)[None], causal, scale, window)
        o[a:b] = ob[0].transpose(1, 0, 2)
        lse[:, a:b] = lb[0]
    return o, lse


def attention_bwd_varlen(q, k, v, dO, cu_seqlens, causal: bool, scale: float, window: int = 0):
    """Gradients for packed sequences: attention_bwd on each sequence in turn.
    Returns dQ [total,Hq,d], dK, dV [total,Hkv,d]."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for a, b in _segments(cu_seqlens):
        if b == a:
            continue
        t = lambda x: x[a:b].transpose(1, 0, 2)[None]  # noqa: E731
        gq, gk, gv = attention_bwd(t(q), t(k), t(v), t(dO), causal, scale, window)
        dq[a:b], dk[a:b], dv[a:b] = (g[0].transpose(1, 0, 2) for g in (gq, gk, gv))
    return dq, dk, dv
