"""Persistent backward main kernel (fa_bwd at N <= 1024, dense layout): work
items (one K/V tile of one key/value head) handed out dynamically by cluster
launch control, per-item set-up and epilogue overlapped.  Checked against the
fp64 oracle (relative Frobenius error <= 1e-2 per tensor), and dK / dV bit
for bit against the deterministic two-pass backward, whose first pass runs
the same per-tile arithmetic with one CTA per work item (dQ is summed by
atomics in a scheduling-dependent order, so it is compared within the
tolerance only)."""
import pytest
import torch

import oracle
from exact_attention_85_gb300 import _lib
from exact_attention_85_gb300.inputs import make_custom

from _tol import check_grad

pytestmark = pytest.mark.gpu


def _fwd_bwd(x, causal, scale, two_pass=False, align16=False):
    q, k, v, dO = (x[n].cuda().contiguous() for n in ("q", "k", "v", "dO"))
    B, Hq, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    _lib.fa_fwd(q, k, v, o, lse, causal, scale)
    dq = torch.empty_like(q)
    if align16:  # dK and dV 16 bytes past a 32-byte boundary
        bk = torch.empty(k.numel() + 8, dtype=k.dtype, device="cuda")
        bv = torch.empty(v.numel() + 8, dtype=v.dtype, device="cuda")
        dk, dv = bk[8:].view(k.shape), bv[8:].view(v.shape)
        assert dk.data_ptr() % 32 == 16 and dv.data_ptr() % 32 == 16
    else:
        dk, dv = torch.empty_like(k), torch.empty_like(v)
    if two_pass:
        ws = torch.empty(_lib.fa_bwd_two_pass_workspace_bytes(B, Hq, N, d), dtype=torch.uint8, device="cuda")
        _lib.fa_bwd_two_pass(q, k, v, o, lse, dO, dq, dk, dv, causal, scale, ws)
    else:
        ws = torch.empty(_lib.fa_bwd_workspace_bytes(B, Hq, N, d), dtype=torch.uint8, device="cuda")
        ws.fill_(0xFF)
        _lib.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, causal, scale, ws)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    return dq, dk, dv


@pytest.mark.parametrize("B,Hq,Hkv,N,d,dtype,causal", [
    (48, 8, 8, 384, 128, torch.bfloat16, True),    # many short items, ragged-free
    (24, 8, 2, 300, 128, torch.bfloat16, True),    # GQA, ragged tail
    (16, 4, 4, 1000, 64, torch.float16, False),    # d = 64, no mask, ragged tail
    (64, 16, 16, 256, 128, torch.bfloat16, False),
])
def test_persistent_bwd_vs_oracle_and_two_pass(cuda_lib, B, Hq, Hkv, N, d, dtype, causal):
    x = make_custom(B, Hq, Hkv, N, d, dtype, seed=B + N + d)
    scale = d ** -0.5
    dq, dk, dv = _fwd_bwd(x, causal, scale)
    rq, rk, rv = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dO"], causal, scale)
    check_grad(dq, rq, "dQ")
    check_grad(dk, rk, "dK")
    check_grad(dv, rv, "dV")
    _, dk2, dv2 = _fwd_bwd(x, causal, scale, two_pass=True)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_bwd_with_16_byte_aligned_dk_dv_falls_back(cuda_lib):
    """The persistent main kernel stores dK / dV rows 32 bytes at a time; with
    them only 16-byte aligned fa_bwd runs one CTA per work item instead, with
    the same results."""
    x = make_custom(8, 4, 2, 512, 128, torch.bfloat16, seed=77)
    scale = 128 ** -0.5
    dq, dk, dv = _fwd_bwd(x, True, scale, align16=True)
    rq, rk, rv = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dO"], True, scale)
    check_grad(dq, rq, "dQ")
    check_grad(dk, rk, "dK")
    check_grad(dv, rv, "dV")
    _, dk2, dv2 = _fwd_bwd(x, True, scale)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_persistent_bwd_concurrent_streams(cuda_lib):
    """Two persistent backward passes with different inputs running at the
    same time on two streams: each grid takes only its own not-yet-launched
    CTAs' work items, so dK and dV equal the one-stream results bit for bit
    (dQ up to the order of its atomic additions) and match the oracle."""
    B, H, N, d = 16, 8, 512, 128
    scale = d ** -0.5
    xs = [make_custom(B, H, H, N, d, torch.bfloat16, seed=s) for s in (51, 52)]
    dev = [{n: x[n].cuda().contiguous() for n in ("q", "k", "v", "dO")} for x in xs]
    fw = []
    for t in dev:
        o = torch.empty_like(t["q"])
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        _lib.fa_fwd(t["q"], t["k"], t["v"], o, lse, True, scale)
        fw.append((o, lse))
    outs = [tuple(torch.empty_like(t[n]) for n in ("q", "k", "v")) for t in dev]
    wss = [torch.empty(_lib.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda") for _ in dev]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(3):
        for t, (o, lse), g, ws, st in zip(dev, fw, outs, wss, streams):
            _lib.fa_bwd(t["q"], t["k"], t["v"], o, lse, t["dO"], *g, True, scale, ws, st)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    for x, g in zip(xs, outs):
        dq, dk, dv = _fwd_bwd(x, True, scale)
        assert torch.equal(g[1], dk) and torch.equal(g[2], dv)
        rq, rk, rv = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dO"], True, scale)
        check_grad(g[0], rq, "dQ")
        check_grad(g[1], rk, "dK")
        check_grad(g[2], rv, "dV")
