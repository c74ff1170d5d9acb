"""Packed variable-length batches (fa_fwd_varlen / fa_bwd_varlen) against the
fp64 oracle applied sequence by sequence.  Tolerances as for the dense path
(O: 4e-3 plus half an output ulp, LSE: 1e-3, grads: relative Frobenius
error <= 1e-2 per tensor)."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_85_gb300 import _lib
from exact_attention_85_gb300.inputs import make_custom, make_varlen, varlen_lengths

from _tol import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


def _run(x, max_len, causal, scale, window=0, deterministic=False):
    q, k, v, dO = (x[n].cuda().contiguous() for n in ("q", "k", "v", "dO"))
    cu = x["cu_seqlens"].cuda()
    total, Hq, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((Hq, total), dtype=torch.float32, device="cuda")
    _lib.fa_fwd_varlen(q, k, v, o, lse, cu, max_len, causal, scale, window)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(_lib.fa_bwd_varlen_workspace_bytes(total, Hq, d, deterministic), dtype=torch.uint8,
                     device="cuda")
    ws.fill_(0xFF)
    _lib.fa_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, cu, max_len, causal, scale, deterministic, ws, window)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    return o, lse, dq, dk, dv


CASES = [
    # lengths, Hq, Hkv, d, dtype, causal, window
    ([1, 127, 128, 129, 255, 256, 257, 600], 2, 2, 128, torch.bfloat16, True, 0),
    ([300, 1, 64, 513], 4, 2, 128, torch.bfloat16, False, 0),
    ([129, 0, 700, 2], 2, 1, 64, torch.float16, True, 0),
    ([640, 333, 17], 2, 2, 128, torch.bfloat16, True, 100),
    (varlen_lengths(6, 900, seed=5), 2, 2, 64, torch.bfloat16, True, 0),
]


@pytest.mark.parametrize("lengths,Hq,Hkv,d,dtype,causal,window", CASES)
@pytest.mark.parametrize("deterministic", [False, True])
def test_varlen_matches_oracle(cuda_lib, lengths, Hq, Hkv, d, dtype, causal, window, deterministic):
    x = make_varlen(lengths, Hq, Hkv, d, dtype, seed=sum(lengths) + d)
    scale = d ** -0.5
    max_len = max(lengths)
    o, lse, dq, dk, dv = _run(x, max_len, causal, scale, window, deterministic)
    ro, rl = oracle.attention_fwd_varlen(x["q"], x["k"], x["v"], x["cu_seqlens"], causal, scale, window)
    check_o(o, ro)
    check_lse(lse, rl)
    rq, rk, rv = oracle.attention_bwd_varlen(x["q"], x["k"], x["v"], x["dO"], x["cu_seqlens"], causal, scale,
                                             window)
    check_grad(dq, rq, "dQ")
    check_grad(dk, rk, "dK")
    check_grad(dv, rv, "dV")


def test_equal_lengths_equal_dense_bit_for_bit(cuda_lib):
    """B sequences of one length N packed token-major run the same kernels on
    the same tiles as the dense [B][H][N][d] call: identical bits."""
    B, Hq, Hkv, N, d = 2, 4, 2, 300, 128
    x = make_custom(B, Hq, Hkv, N, d, torch.bfloat16, seed=9)
    scale = d ** -0.5
    q, k, v, dO = (x[n].cuda().contiguous() for n in ("q", "k", "v", "dO"))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    _lib.fa_fwd(q, k, v, o, lse, True, scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(_lib.fa_bwd_two_pass_workspace_bytes(B, Hq, N, d), dtype=torch.uint8, device="cuda")
    _lib.fa_bwd_two_pass(q, k, v, o, lse, dO, dq, dk, dv, True, scale, ws)
    pack = lambda t: t.transpose(1, 2).reshape(B * N, t.shape[1], d).contiguous()  # noqa: E731
    xp = {"q": pack(q).cpu(), "k": pack(k).cpu(), "v": pack(v).cpu(), "dO": pack(dO).cpu(),
          "cu_seqlens": torch.arange(0, (B + 1) * N, N, dtype=torch.int32)}
    po, plse, pdq, pdk, pdv = _run(xp, N, True, scale, 0, True)
    assert torch.equal(po, pack(o))
    assert torch.equal(plse, lse.permute(1, 0, 2).reshape(Hq, B * N))
    assert torch.equal(pdq, pack(dq)) and torch.equal(pdk, pack(dk)) and torch.equal(pdv, pack(dv))


def test_bad_offsets_reported_not_faulted(cuda_lib):
    """Offsets that are not a non-decreasing prefix sum are caught on the
    device: the status word reports FA_ERR_INVALID_ARG and the bad sequence is
    skipped (no out-of-range access)."""
    x = make_varlen([100, 50, 80], 2, 2, 64, torch.bfloat16, seed=2)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    total = q.shape[0]
    cu = torch.tensor([0, 100, 60, total], dtype=torch.int32, device="cuda")  # second length negative
    o = torch.zeros_like(q)
    lse = torch.empty((2, total), dtype=torch.float32, device="cuda")
    _lib.fa_fwd_varlen(q, k, v, o, lse, cu, 200, True, 0.125)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_ERR_INVALID_ARG
    assert _lib.fa_get_device_status() == _lib.FA_OK  # reading clears it


@pytest.mark.parametrize("lengths,Hq,Hkv,d,causal,window", [
    ([0, 1, 127, 128, 129, 255, 256, 257, 1000, 0, 2048], 4, 2, 128, True, 0),
    ([5, 300, 1, 2049], 2, 2, 64, False, 0),
    ([700, 0, 3000, 64], 4, 1, 128, True, 200),
])
def test_varlen_persistent_and_plain_kernels_agree(cuda_lib, lengths, Hq, Hkv, d, causal, window):
    """fa_fwd_varlen runs the persistent forward when no row sees more than
    2048 keys (max_seqlen or the window) and O is 32-byte aligned, else one
    CTA per block: for the same batch both give the same bits (empty
    sequences and blocks past a sequence's end included), and the oracle's
    values within tolerance."""
    x = make_varlen(lengths, Hq, Hkv, d, torch.bfloat16, seed=len(lengths) + d, with_grad=False)
    q, k, v = (x[n].cuda().contiguous() for n in ("q", "k", "v"))
    cu = x["cu_seqlens"].cuda()
    total = q.shape[0]
    scale = d ** -0.5
    outs = []
    for align16 in (False, True):
        if align16:
            buf = torch.empty(q.numel() + 8, dtype=q.dtype, device="cuda")
            o = buf[8:].view(q.shape)
            assert o.data_ptr() % 32 == 16
        else:
            o = torch.empty_like(q)
        lse = torch.empty((Hq, total), dtype=torch.float32, device="cuda")
        _lib.fa_fwd_varlen(q, k, v, o, lse, cu, max(lengths), causal, scale, window)
        torch.cuda.synchronize()
        assert _lib.fa_get_device_status() == _lib.FA_OK
        outs.append((o, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    ro, rl = oracle.attention_fwd_varlen(x["q"], x["k"], x["v"], x["cu_seqlens"], causal, scale, window)
    check_o(outs[0][0], ro)
    check_lse(outs[0][1], rl)
