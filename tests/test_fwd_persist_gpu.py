"""Persistent forward (fa_fwd_persistent): blocks handed out dynamically by
cluster launch control, with loads, first MMAs and epilogues overlapping
across blocks.  Checked against the fp64 oracle (O element-wise within 4e-3
plus half an ulp of the output type, LSE max-abs 1e-3), and bit for bit
against the plain forward's fp32 output rounded to the 16-bit type (the two
kernels do the same arithmetic per block; only the schedule differs)."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_85_gb300 import _lib
from exact_attention_85_gb300.inputs import HEADLINE, WORKLOADS, make_custom, make_inputs

from _tol import check_lse, check_o

pytestmark = pytest.mark.gpu


def _run(x, causal, scale, fn=_lib.fa_fwd_persistent):
    q, k, v = (x[n].cuda().contiguous() for n in ("q", "k", "v"))
    B, Hq, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    fn(q, k, v, o, lse, causal, scale)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    return o, lse


def _plain_rounded(x, causal, scale):
    """The plain (one CTA per block) kernel's fp32 output, rounded."""
    q, k, v = (x[n].cuda().contiguous() for n in ("q", "k", "v"))
    B, Hq, N, d = q.shape
    o32 = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    _lib.fa_fwd_f32_out(q, k, v, o32, lse, causal, scale)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    return o32.to(q.dtype), lse


SHAPES = [
    # B, Hq, Hkv, N, d, dtype, causal
    (1, 1, 1, 1, 128, torch.bfloat16, True),
    (1, 2, 2, 127, 128, torch.bfloat16, True),
    (1, 2, 1, 129, 128, torch.bfloat16, False),
    (2, 4, 2, 300, 128, torch.bfloat16, True),
    (2, 4, 4, 300, 64, torch.float16, False),
    (1, 3, 1, 1000, 128, torch.bfloat16, True),
    (1, 4, 1, 1000, 64, torch.bfloat16, True),
    (3, 2, 2, 640, 128, torch.float16, True),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,dtype,causal", SHAPES)
def test_persistent_small_vs_oracle_and_plain(cuda_lib, B, Hq, Hkv, N, d, dtype, causal):
    x = make_custom(B, Hq, Hkv, N, d, dtype, seed=N * 5 + d + B, with_grad=False)
    scale = d ** -0.5
    o, lse = _run(x, causal, scale)
    o_ref, lse_ref = oracle.attention_fwd(x["q"], x["k"], x["v"], causal, scale)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
    o_plain, lse_plain = _plain_rounded(x, causal, scale)
    assert torch.equal(o, o_plain)
    assert torch.equal(lse, lse_plain)


@pytest.mark.parametrize("B,Hq,N,causal", [(64, 16, 256, True), (48, 8, 384, False), (16, 16, 1280, True)])
def test_persistent_many_short_blocks(cuda_lib, B, Hq, N, causal):
    """Far more blocks than SMs, each only a few K/V tiles long: most CTAs
    take many blocks in turn (ragged tails included at N = 384, 1280)."""
    d = 128
    x = make_custom(B, Hq, Hq, N, d, torch.bfloat16, seed=B + N, with_grad=False)
    scale = d ** -0.5
    o, lse = _run(x, causal, scale)
    o_ref, lse_ref = oracle.attention_fwd(x["q"], x["k"], x["v"], causal, scale)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
    o2, lse2 = _run(x, causal, scale)  # the schedule may differ; the results may not
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_persistent_training_shape_whole_tensor(cuda_lib):
    """B8 H16 N2048 d128 causal, the short-sequence shape the persistent
    kernel is for: whole O and LSE against the oracle, and bit-identical to
    the plain kernel."""
    w = WORKLOADS["train_bf16_b8_h16_n2k_causal"]
    x = make_inputs(w, with_grad=False)
    o, lse = _run(x, w.causal, w.scale)
    o_ref, lse_ref = oracle.attention_fwd(x["q"], x["k"], x["v"], w.causal, w.scale)
    check_o(o, o_ref, "persistent O")
    check_lse(lse, lse_ref, "persistent LSE")
    o_plain, lse_plain = _plain_rounded(x, w.causal, w.scale)
    assert torch.equal(o, o_plain) and torch.equal(lse, lse_plain)


@pytest.mark.parametrize("name", ["gqa_bf16_b4_hq32_hkv8_n4k_causal", HEADLINE])
def test_persistent_full_size_bit_identical_to_plain(cuda_lib, name):
    w = WORKLOADS[name]
    x = make_inputs(w, with_grad=False)
    o, lse = _run(x, w.causal, w.scale)
    o_plain, lse_plain = _plain_rounded(x, w.causal, w.scale)
    assert torch.equal(o, o_plain) and torch.equal(lse, lse_plain)
    # and a sample of rows against the oracle (first and last Q tile of the
    # first and last plane)
    rows = [(b, h, r) for b, h in ((0, 0), (w.B - 1, w.Hq - 1))
            for r in list(range(128)) + list(range(w.N - 128, w.N))]
    o_ref, lse_ref = oracle.attention_fwd_rows(x["q"], x["k"], x["v"], rows, w.causal, w.scale)
    idx = tuple(np.array(rows).T)
    check_o(o[idx], o_ref, f"{name} O")
    check_lse(lse[idx], lse_ref, f"{name} LSE")


def test_fwd_with_16_byte_aligned_output_falls_back(cuda_lib):
    """fa_fwd at a short sequence length with O only 16-byte aligned: the
    persistent kernel (32-byte row stores) is skipped for the one-CTA-per-block
    kernel, and the result still matches the oracle."""
    B, Hq, N, d = 2, 4, 700, 128
    x = make_custom(B, Hq, Hq, N, d, torch.bfloat16, seed=29, with_grad=False)
    q, k, v = (x[n].cuda().contiguous() for n in ("q", "k", "v"))
    buf = torch.empty(B * Hq * N * d + 8, dtype=torch.bfloat16, device="cuda")
    o = buf[8:].view(B, Hq, N, d)  # 16 bytes past a 32-byte boundary
    assert o.data_ptr() % 32 == 16
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    _lib.fa_fwd(q, k, v, o, lse, True, d ** -0.5)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    o_ref, lse_ref = oracle.attention_fwd(x["q"], x["k"], x["v"], True, d ** -0.5)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)
    with pytest.raises(_lib.FAError):
        _lib.fa_fwd_persistent(q, k, v, o, lse, True, d ** -0.5)


def test_persistent_concurrent_streams(cuda_lib):
    """Two persistent forwards with different inputs running at the same time
    on two streams: each grid takes only its own not-yet-launched CTAs' blocks
    (a cancelled CTA belongs to the grid that cancelled it), so both results
    match their oracle and their one-stream runs bit for bit."""
    d = 128
    xs = [make_custom(16, 8, 8, 1024, d, torch.bfloat16, seed=s, with_grad=False) for s in (41, 42)]
    dev = [{n: x[n].cuda().contiguous() for n in ("q", "k", "v")} for x in xs]
    outs = [(torch.empty_like(t["q"]), torch.empty((16, 8, 1024), dtype=torch.float32, device="cuda")) for t in dev]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for rep in range(3):
        for t, (o, lse), st in zip(dev, outs, streams):
            _lib.fa_fwd_persistent(t["q"], t["k"], t["v"], o, lse, True, d ** -0.5, st)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    for x, t, (o, lse) in zip(xs, dev, outs):
        alone_o, alone_lse = _run(x, True, d ** -0.5)
        assert torch.equal(o, alone_o) and torch.equal(lse, alone_lse)
    o_ref, lse_ref = oracle.attention_fwd(xs[1]["q"], xs[1]["k"], xs[1]["v"], True, d ** -0.5)
    check_o(outs[1][0], o_ref)
    check_lse(outs[1][1], lse_ref)
