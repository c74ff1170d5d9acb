"""Backward parity: fa_bwd (through the C ABI) against the fp64 oracle's
analytic gradients.  Tolerance: relative Frobenius error <= 1e-2 per tensor."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_85_gb300 import _lib
from exact_attention_85_gb300.inputs import HEADLINE, WORKLOADS, make_custom, make_inputs

from _tol import check_grad

pytestmark = pytest.mark.gpu


def _run(x, causal, scale):
    q, k, v, dO = (x[n].cuda().contiguous() for n in ("q", "k", "v", "dO"))
    B, Hq, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    _lib.fa_fwd(q, k, v, o, lse, causal, scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(_lib.fa_bwd_workspace_bytes(B, Hq, N, d), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)  # contents on entry must not matter
    _lib.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, causal, scale, ws)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    return dq, dk, dv


SHAPES = [
    # B, Hq, Hkv, N, d, dtype, causal
    (1, 1, 1, 1, 128, torch.bfloat16, True),
    (1, 1, 1, 1, 64, torch.float16, False),
    (1, 2, 2, 64, 128, torch.bfloat16, True),
    (1, 2, 1, 127, 128, torch.bfloat16, False),
    (1, 2, 2, 129, 64, torch.float16, True),
    (2, 4, 2, 300, 128, torch.bfloat16, True),
    (2, 4, 4, 300, 64, torch.bfloat16, False),
    (1, 4, 1, 500, 128, torch.bfloat16, True),
    (1, 6, 2, 384, 64, torch.float16, True),
    (2, 2, 2, 256, 128, torch.float16, False),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,dtype,causal", SHAPES)
def test_bwd_small_full_compare(cuda_lib, B, Hq, Hkv, N, d, dtype, causal):
    x = make_custom(B, Hq, Hkv, N, d, dtype, seed=N * 3 + d + Hq)
    scale = d ** -0.5
    dq, dk, dv = _run(x, causal, scale)
    rq, rk, rv = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dO"], causal, scale)
    check_grad(dq, rq, "dQ")
    check_grad(dk, rk, "dK")
    check_grad(dv, rv, "dV")


def test_bwd_tiny_workload_full(cuda_lib):
    w = WORKLOADS["tiny_fp16_d64_n256"]
    x = make_inputs(w)
    dq, dk, dv = _run(x, w.causal, w.scale)
    rq, rk, rv = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dO"], w.causal, w.scale)
    check_grad(dq, rq, "dQ")
    check_grad(dk, rk, "dK")
    check_grad(dv, rv, "dV")


def test_bwd_repeatable_within_tolerance(cuda_lib):
    """dK and dV are owned by one CTA each (bit-identical across runs); dQ is
    summed with fp32 atomics, so only its order of additions may differ."""
    x = make_custom(2, 4, 2, 700, 128, torch.bfloat16, seed=5)
    a = _run(x, True, 0.09)
    b = _run(x, True, 0.09)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    rel = float((a[0].float() - b[0].float()).norm() / a[0].float().norm())
    assert rel < 1e-3


def test_bwd_full_size_whole_tensor(cuda_lib):
    """Training shape B8 H16 N2048 d128 causal: the whole dQ, dK and dV of the
    full-size launch against the oracle, per tensor and per (batch, head)
    plane (a plane computed wrong shows even where the tensor-wide norm would
    dilute it)."""
    w = WORKLOADS["train_bf16_b8_h16_n2k_causal"]
    x = make_inputs(w)
    dq, dk, dv = _run(x, w.causal, w.scale)
    rq, rk, rv = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dO"], w.causal, w.scale)
    errs = [check_grad(got, ref, f"{nm}") for nm, got, ref in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv))]
    worst = 0.0
    for nm, got, ref in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        g = got.float().cpu().numpy()
        for b in range(ref.shape[0]):
            for h in range(ref.shape[1]):
                worst = max(worst, check_grad(g[b, h], ref[b, h], f"{nm} plane ({b}, {h})"))
    print(f"training shape: dQ/dK/dV rel {errs[0]:.2e} {errs[1]:.2e} {errs[2]:.2e}; worst plane {worst:.2e}")


@pytest.mark.parametrize("name", ["long_bf16_b1_h16_n16k_causal", "gqa_bf16_b4_hq32_hkv8_n4k_causal", HEADLINE])
def test_bwd_full_size_groups(cuda_lib, name):
    """Full-size launch; the oracle checks the first, a middle and the last
    (batch, kv-head) group entirely (its query heads' dQ and the group's dK,
    dV) and the rest is checked for finiteness."""
    w = WORKLOADS[name]
    x = make_inputs(w)
    dq, dk, dv = _run(x, w.causal, w.scale)
    G = w.Hq // w.Hkv
    for b, g in ((0, 0), (w.B // 2, w.Hkv // 2), (w.B - 1, w.Hkv - 1)):
        rq, rk, rv = oracle.attention_bwd_group(x["q"], x["k"], x["v"], x["dO"], b, g, w.causal, w.scale)
        check_grad(dq[b, g * G:(g + 1) * G], rq, f"{name} ({b}, {g}) dQ")
        check_grad(dk[b, g], rk, f"{name} ({b}, {g}) dK")
        check_grad(dv[b, g], rv, f"{name} ({b}, {g}) dV")
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
