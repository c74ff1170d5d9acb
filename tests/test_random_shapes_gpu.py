"""Seeded random shapes for fa_fwd and fa_bwd against the fp64 oracle.

The draws cross every dispatch boundary of the two entry points: sequence
lengths on both sides of the persistent forward's (N <= 2048) and the
persistent backward's (N <= 1024) ranges, ragged tails, GQA ratios 1-4, both
head dimensions and both 16-bit element types, causal or not.  Tolerances are
those of every parity test: O element-wise within 4e-3 plus half an ulp of
the output type, LSE max-abs 1e-3, gradients relative Frobenius <= 1e-2."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_85_gb300 import _lib
from exact_attention_85_gb300.inputs import make_custom

from _tol import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


def _draw(seed):
    g = np.random.default_rng(seed)
    G = int(g.choice([1, 2, 4]))
    Hkv = int(g.integers(1, 3))
    N = int(g.choice([int(g.integers(1, 700)), int(g.integers(700, 1100)), int(g.integers(1900, 2200)),
                      int(g.integers(2200, 2700))]))
    d = int(g.choice([64, 128]))
    dtype = torch.bfloat16 if g.integers(2) else torch.float16
    causal = bool(g.integers(2))
    B = 1 if N > 1500 else int(g.integers(1, 3))
    return B, G * Hkv, Hkv, N, d, dtype, causal


@pytest.mark.parametrize("seed", range(12))
def test_random_shape_forward_backward(cuda_lib, seed):
    B, Hq, Hkv, N, d, dtype, causal = _draw(1000 + seed)
    x = make_custom(B, Hq, Hkv, N, d, dtype, seed=seed)
    q, k, v, dO = (x[n].cuda().contiguous() for n in ("q", "k", "v", "dO"))
    scale = d ** -0.5
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    _lib.fa_fwd(q, k, v, o, lse, causal, scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(_lib.fa_bwd_workspace_bytes(B, Hq, N, d), dtype=torch.uint8, device="cuda")
    _lib.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, causal, scale, ws)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    what = f"B{B} Hq{Hq} Hkv{Hkv} N{N} d{d} {str(dtype)[6:]} causal={causal}"
    o_ref, lse_ref = oracle.attention_fwd(x["q"], x["k"], x["v"], causal, scale)
    check_o(o, o_ref, f"{what} O")
    check_lse(lse, lse_ref, f"{what} LSE")
    rq, rk, rv = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dO"], causal, scale)
    check_grad(dq, rq, f"{what} dQ")
    check_grad(dk, rk, f"{what} dK")
    check_grad(dv, rv, f"{what} dV")
