"""fa_bwd_noalloc: the backward for callers that cannot allocate device
memory (for example a plugin that is handed only tensor pointers by its host
framework, or a process whose memory pool is fixed up front).  It uses a
scratch buffer built into the library instead of a caller workspace.

These tests check, on two calls in a row (the second must not see anything
the first left in the shared buffer):
  * its gradients against the fp64 oracle (relative Frobenius error <= 1e-2
    per tensor, the tolerance of every backward test) and against fa_bwd's;
  * that a call allocates nothing: torch's allocated bytes and the device's
    free bytes (cudaMemGetInfo) are the same before and after the second
    call (the first call may commit the built-in buffer when the library
    part that holds it is loaded, so it is not measured);
  * that too-large problems are refused up front, and invalid arguments get
    fa_bwd's status codes.

This file is named so that pytest collects it last."""
import gc

import pytest
import torch

import oracle
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


@pytest.mark.parametrize("B,Hq,Hkv,N,d,scale,dtype,want", [
    (4, 16, 16, 8192, 256, 0.1, 1, "FA_ERR_UNSUPPORTED"),  # unsupported d, and too large for the buffer
    (4, 16, 5, 8192, 128, 0.1, 1, "FA_ERR_INVALID_ARG"),   # Hq % Hkv != 0, too large
    (4, 16, 16, 8192, 128, -1.0, 1, "FA_ERR_INVALID_ARG"),  # bad scale, too large
    (4, 16, 16, 8192, 128, 0.1, 7, "FA_ERR_INVALID_ARG"),   # bad element type, too large
])
def test_noalloc_classifies_invalid_arguments_like_fa_bwd(B, Hq, Hkv, N, d, scale, dtype, want):
    """The size of the built-in buffer is checked only once every other
    argument is valid, so a call gets the code fa_bwd would give."""
    lib = _lib.load()
    args = [FAKE] * 9 + [B, Hq, Hkv, N, d, 1, scale, dtype]
    assert lib.fa_bwd_noalloc(*args, None) == getattr(_lib, want)
    assert lib.fa_bwd(*args, FAKE, 1 << 40, None) == getattr(_lib, want)


@pytest.mark.gpu
@pytest.mark.parametrize("B,Hq,Hkv,N,d,dtype,causal", [
    (2, 4, 2, 700, 128, torch.bfloat16, True),
    (1, 2, 2, 300, 64, torch.float16, False),
])
def test_noalloc_matches_oracle_and_fa_bwd_on_two_calls(cuda_lib, B, Hq, Hkv, N, d, dtype, causal):
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
    exact = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dO"], causal, scale)
    for call in range(2):
        got = [torch.full_like(q, float("nan")), torch.full_like(k, float("nan")), torch.full_like(v, float("nan"))]
        torch.cuda.synchronize()
        # the collector is paused so that no unrelated tensor is freed
        # between the two readings
        gc.collect()
        gc.disable()
        try:
            alloc0 = torch.cuda.memory_allocated()
            free0, _ = torch.cuda.mem_get_info()
            _lib.fa_bwd_noalloc(q, k, v, o, lse, dO, *got, causal, scale)
            torch.cuda.synchronize()
            free1, _ = torch.cuda.mem_get_info()
            alloc1 = torch.cuda.memory_allocated()
        finally:
            gc.enable()
        assert alloc1 == alloc0
        if call == 1:
            assert free1 == free0, f"device free bytes changed across the call: {free0} -> {free1}"
        assert _lib.fa_get_device_status() == _lib.FA_OK
        for name, g, r, e in zip(("dQ", "dK", "dV"), got, ref_np, exact):
            check_grad(g, e, f"call {call + 1} {name} vs oracle")
            # the same kernels as fa_bwd: equal up to the order of the dQ atomics
            check_grad(g, r, f"call {call + 1} {name} vs fa_bwd")
