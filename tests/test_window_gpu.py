"""Causal sliding-window attention (fa_fwd_local / fa_bwd_local) against the
fp64 oracle with the same mask.  Tolerances as for the full forward and
backward (O: max |err| <= 4e-3 plus half an output ulp, LSE: 1e-3, grads:
relative Frobenius error <= 1e-2)."""
import pytest
import torch

import oracle
from exact_attention_85_gb300 import _lib
from exact_attention_85_gb300.inputs import make_custom

from _tol import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


def _fwd(x, window, scale):
    q, k, v = (x[n].cuda().contiguous() for n in ("q", "k", "v"))
    B, Hq, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    _lib.fa_fwd_local(q, k, v, o, lse, window, scale)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    return q, k, v, o, lse


def _bwd(t, dO, window, scale, deterministic):
    q, k, v, o, lse = t
    B, Hq, N, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    size = (_lib.fa_bwd_two_pass_workspace_bytes if deterministic else _lib.fa_bwd_workspace_bytes)(B, Hq, N, d)
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)
    _lib.fa_bwd_local(q, k, v, o, lse, dO.cuda().contiguous(), dq, dk, dv, window, scale, deterministic, ws)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    return dq, dk, dv


CASES = [
    # B, Hq, Hkv, N, d, dtype, window
    (1, 2, 2, 300, 128, torch.bfloat16, 1),
    (1, 2, 1, 300, 128, torch.bfloat16, 2),
    (1, 2, 2, 517, 64, torch.float16, 100),
    (2, 2, 2, 640, 128, torch.bfloat16, 128),
    (1, 4, 2, 640, 128, torch.bfloat16, 129),
    (1, 2, 2, 1000, 128, torch.bfloat16, 256),
    (1, 2, 2, 777, 64, torch.bfloat16, 300),
    (1, 2, 2, 384, 128, torch.float16, 5000),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,dtype,window", CASES)
def test_window_forward_and_backward(cuda_lib, B, Hq, Hkv, N, d, dtype, window):
    x = make_custom(B, Hq, Hkv, N, d, dtype, seed=N + window)
    scale = d ** -0.5
    t = _fwd(x, window, scale)
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], True, scale, window=window)
    check_o(t[3], ro)
    check_lse(t[4], rl)
    rq, rk, rv = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dO"], True, scale, window=window)
    for det in (False, True):
        dq, dk, dv = _bwd(t, x["dO"], window, scale, det)
        check_grad(dq, rq, f"dQ det={det}")
        check_grad(dk, rk, f"dK det={det}")
        check_grad(dv, rv, f"dV det={det}")


def test_window_at_least_n_equals_causal(cuda_lib):
    """With W >= N every causal key is inside the window: same kernels, same
    tiles, so the results equal the plain causal ones bit for bit."""
    x = make_custom(1, 2, 2, 500, 128, torch.bfloat16, seed=3)
    scale = 0.08
    t = _fwd(x, 500, scale)
    q, k, v = t[:3]
    o = torch.empty_like(q)
    lse = torch.empty_like(t[4])
    _lib.fa_fwd(q, k, v, o, lse, True, scale)
    torch.cuda.synchronize()
    assert torch.equal(o, t[3]) and torch.equal(lse, t[4])


def test_window_rejects_zero(cuda_lib):
    x = make_custom(1, 1, 1, 64, 64, torch.bfloat16, seed=1)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(_lib.FAError) as e:
        _lib.fa_fwd_local(q, k, v, o, lse, 0, 0.125)
    assert e.value.status == _lib.FA_ERR_INVALID_ARG


def _o16(q):
    """An output buffer only 16-byte aligned: fa_fwd_local then runs the
    one-CTA-per-block kernel instead of the persistent one (32-byte stores)."""
    buf = torch.empty(q.numel() + 8, dtype=q.dtype, device=q.device)
    o = buf[8:].view(q.shape)
    assert o.data_ptr() % 32 == 16
    return o


@pytest.mark.parametrize("B,Hq,Hkv,N,d,dtype,window", [
    (1, 4, 2, 1500, 128, torch.bfloat16, 1),
    (2, 4, 1, 1100, 128, torch.float16, 200),
    (1, 2, 2, 3000, 64, torch.bfloat16, 1000),
    (1, 2, 2, 2600, 128, torch.bfloat16, 2048),  # the largest window routed to the persistent kernel
    (1, 2, 2, 2600, 128, torch.bfloat16, 2049),  # the smallest one that is not
])
def test_window_persistent_and_plain_kernels_agree(cuda_lib, B, Hq, Hkv, N, d, dtype, window):
    """The two forward kernels fa_fwd_local chooses between (persistent for
    windows up to 2048 keys with a 32-byte-aligned O, else one CTA per
    block) compute every block the same way: the same bits, and both within
    the tolerance of the oracle."""
    x = make_custom(B, Hq, Hkv, N, d, dtype, seed=N + 3 * window, with_grad=False)
    scale = d ** -0.5
    q, k, v, o, lse = _fwd(x, window, scale)
    o2 = _o16(q)
    lse2 = torch.empty_like(lse)
    _lib.fa_fwd_local(q, k, v, o2, lse2, window, scale)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], True, scale, window=window)
    check_o(o, ro)
    check_lse(lse, rl)
