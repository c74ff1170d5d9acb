"""fa_bwd_noalloc: the backward for callers that cannot allocate device
memory (for example a plugin that is handed only tensor pointers by its host
framework, or a process whose memory pool is fixed up front).  It uses a
scratch buffer built into the library instead of a caller workspace, so these
tests check that its results match fa_bwd's (same tolerance as the other
backward tests: relative Frobenius error <= 1e-2 per tensor) on two calls in
a row -- the second call must not see anything left in the shared buffer by
the first -- and that too-large problems are refused up front.

This file is named so that pytest collects it last."""
import pytest
import torch

from exact_attention_85_gb300 import _lib
from exact_attention_85_gb300.inputs import make_custom

from _tol import check_grad

FAKE = 1 << 20  # aligned non-null value; never dereferenced (refused first)


def test_noalloc_refuses_problems_larger_than_its_buffer():
    from exact_attention_85_gb300 import build
    build.build()
    lib = _lib.load()
    B, Hq, N, d = 4, 16, 8192, 128
    assert lib.fa_bwd_workspace_bytes(B, Hq, N, d) > (64 << 20)
    args = [FAKE] * 9 + [B, Hq, Hq, N, d, 1, 0.1, _lib.FA_BF16, None]
    assert lib.fa_bwd_noalloc(*args) == _lib.FA_ERR_WORKSPACE
    bad = [None] + [FAKE] * 8 + [1, 2, 1, 16, 128, 0, 0.1, _lib.FA_BF16, None]
    assert lib.fa_bwd_noalloc(*bad) == _lib.FA_ERR_INVALID_ARG


@pytest.mark.gpu
@pytest.mark.parametrize("B,Hq,Hkv,N,d,dtype,causal", [
    (2, 4, 2, 700, 128, torch.bfloat16, True),
    (1, 2, 2, 300, 64, torch.float16, False),
])
def test_noalloc_matches_fa_bwd_on_two_calls(cuda_lib, B, Hq, Hkv, N, d, dtype, causal):
    x = make_custom(B, Hq, Hkv, N, d, dtype, seed=17 + N)
    q, k, v, dO = (x[n].cuda().contiguous() for n in ("q", "k", "v", "dO"))
    scale = d ** -0.5
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    _lib.fa_fwd(q, k, v, o, lse, causal, scale)
    ws = torch.empty(_lib.fa_bwd_workspace_bytes(B, Hq, N, d), dtype=torch.uint8, device="cuda")
    ref = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    _lib.fa_bwd(q, k, v, o, lse, dO, *ref, causal, scale, ws)
    torch.cuda.synchronize()
    ref_np = [t.double().cpu().numpy() for t in ref]
    for call in range(2):
        got = [torch.full_like(q, float("nan")), torch.full_like(k, float("nan")), torch.full_like(v, float("nan"))]
        _lib.fa_bwd_noalloc(q, k, v, o, lse, dO, *got, causal, scale)
        torch.cuda.synchronize()
        assert _lib.fa_get_device_status() == _lib.FA_OK
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref_np):
            check_grad(g, r, f"call {call + 1} {name}")
