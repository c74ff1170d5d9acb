"""Tensors of more than 2^31 elements.

B33 H64 N8192 d128 holds 2.2e9 elements per tensor (4.4 GB in bf16), and
(batch, head) plane 2048 starts exactly at element 2^31.  Four planes on both
sides of that boundary hold seeded N(0, 1) values, every other plane zeros:
the inputs stay cheap to make, and an offset that wrapped at 32 bits would
land in a zero plane.  Checked against the fp64 oracle:

  * the forward (one CTA per block) on rows of the four planes, and the
    persistent forward bit for bit against it;
  * the atomic and the deterministic backward on whole planes (Hq = Hkv, so a
    plane is a whole (batch, kv-head) group), dK and dV of the two
    bit-identical;
  * a packed batch of the same rows (33 sequences of 8192) bit for bit
    against the dense forward;
  * the FP8 path (Hadamard quantisation of 2.2e9 values, FP8 forward) against
    the oracle's model of that pipeline.

Zero planes have a closed form: O = 0, L = ln(r + 1) for causal row r (every
visible score is 0), and zero gradients.  Tolerances as everywhere: O within
4e-3 plus half an output ulp, LSE max-abs 1e-3, gradients relative Frobenius
<= 1e-2, FP8 O relative RMS <= 0.03 against the pipeline model.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_85_gb300 import _lib, hadamard_quant_fp8

from _tol import FP8_REL_RMS, check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu

B, H, N, D = 33, 64, 8192, 128
PLANES = (0, 2047, 2048, 2111)  # plane p is (b, h) = divmod(p, H)
ZERO_PLANES = (1000, 2100)
SCALE = D ** -0.5
NAMES = ("q", "k", "v", "dO")


def _rows():
    g = np.random.default_rng(31)
    mid = sorted(int(r) for r in g.choice(np.arange(128, N - 128), 64, replace=False))
    return list(range(128)) + mid + list(range(N - 128, N))


@pytest.fixture(scope="module")
def big():
    assert B * H * N * D > 2 ** 31 and 2048 * N * D == 2 ** 31
    host = {}
    dev = {n: torch.zeros((B, H, N, D), dtype=torch.bfloat16, device="cuda") for n in NAMES}
    for p in PLANES:
        g = torch.Generator().manual_seed(7000 + p)
        b, h = divmod(p, H)
        for n in NAMES:
            t = torch.randn(N, D, generator=g).to(torch.bfloat16)
            host[(n, p)] = t.reshape(1, 1, N, D)
            dev[n][b, h].copy_(t)
    yield dev, host
    dev.clear()
    torch.cuda.empty_cache()


def _forward(dev, persistent=False):
    q, k, v = dev["q"], dev["k"], dev["v"]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    (_lib.fa_fwd_persistent if persistent else _lib.fa_fwd)(q, k, v, o, lse, True, SCALE)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    return o, lse


def _zero_plane_checks(o, lse, what):
    ln = np.log(np.arange(1, N + 1, dtype=np.float64))  # causal row r sees r + 1 zero scores
    for p in ZERO_PLANES:
        b, h = divmod(p, H)
        assert int(torch.count_nonzero(o[b, h])) == 0, f"{what}: plane {p} O not zero"
        check_lse(lse[b, h], ln, f"{what}: plane {p} LSE")


def test_forward_beyond_2g_elements(cuda_lib, big):
    dev, host = big
    o, lse = _forward(dev)
    rows = _rows()
    for p in PLANES:
        b, h = divmod(p, H)
        ro, rl = oracle.attention_fwd_rows(host[("q", p)], host[("k", p)], host[("v", p)],
                                           [(0, 0, r) for r in rows], True, SCALE)
        check_o(o[b, h, rows], ro, f"plane {p} O")
        check_lse(lse[b, h, rows], rl, f"plane {p} LSE")
    _zero_plane_checks(o, lse, "fa_fwd")
    o2, lse2 = _forward(dev, persistent=True)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_backward_beyond_2g_elements(cuda_lib, big):
    dev, host = big
    o, lse = _forward(dev)
    q, k, v, dO = (dev[n] for n in NAMES)
    grads = {}
    for two_pass in (False, True):
        size = (_lib.fa_bwd_two_pass_workspace_bytes if two_pass else _lib.fa_bwd_workspace_bytes)(B, H, N, D)
        ws = torch.empty(size, dtype=torch.uint8, device="cuda")
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        (_lib.fa_bwd_two_pass if two_pass else _lib.fa_bwd)(q, k, v, o, lse, dO, dq, dk, dv, True, SCALE, ws)
        torch.cuda.synchronize()
        assert _lib.fa_get_device_status() == _lib.FA_OK
        del ws
        grads[two_pass] = (dq, dk, dv)
    # the two backward variants sum dK and dV in the same order
    assert torch.equal(grads[False][1], grads[True][1]) and torch.equal(grads[False][2], grads[True][2])
    for p in (0, 2048, 2111):
        b, h = divmod(p, H)
        rq, rk, rv = oracle.attention_bwd(host[("q", p)], host[("k", p)], host[("v", p)], host[("dO", p)], True,
                                          SCALE)
        for two_pass, (dq, dk, dv) in grads.items():
            tag = f"plane {p} {'two-pass' if two_pass else 'atomic'}"
            check_grad(dq[b, h], rq[0, 0], f"{tag} dQ")
            check_grad(dk[b, h], rk[0, 0], f"{tag} dK")
            check_grad(dv[b, h], rv[0, 0], f"{tag} dV")
    for p in ZERO_PLANES:
        b, h = divmod(p, H)
        for dq, dk, dv in grads.values():
            assert all(int(torch.count_nonzero(t[b, h])) == 0 for t in (dq, dk, dv)), f"plane {p} gradients"


def test_packed_batch_beyond_2g_elements(cuda_lib, big):
    """The same rows as 33 packed sequences of 8192 (token-major, 2.2e9
    elements per tensor): the packed forward equals the dense one bit for
    bit (same kernels, same tiles)."""
    dev, _ = big
    o, lse = _forward(dev)
    pack = lambda t: t.transpose(1, 2).reshape(B * N, H, D).contiguous()  # noqa: E731
    qp, kp, vp = pack(dev["q"]), pack(dev["k"]), pack(dev["v"])
    cu = torch.arange(0, (B + 1) * N, N, dtype=torch.int32, device="cuda")
    op = torch.empty_like(qp)
    lsep = torch.empty((H, B * N), dtype=torch.float32, device="cuda")
    _lib.fa_fwd_varlen(qp, kp, vp, op, lsep, cu, N, True, SCALE)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    del qp, kp, vp
    assert torch.equal(op, pack(o))
    assert torch.equal(lsep, lse.permute(1, 0, 2).reshape(H, B * N))


def test_fp8_beyond_2g_elements(cuda_lib, big):
    """Hadamard quantisation of 2.2e9-element tensors and the FP8 forward
    (non-causal), rows of the planes past element 2^31 against the oracle's
    pipeline model.  The per-tensor scale comes from the amax of the whole
    tensor, i.e. of its non-zero planes, so the model quantises those planes
    alone."""
    dev, host = big
    g = torch.Generator().manual_seed(77)
    signs = (torch.randint(0, 2, (D,), generator=g) * 2 - 1).float()
    q8, qs = hadamard_quant_fp8(dev["q"], signs.cuda())
    k8, ks = hadamard_quant_fp8(dev["k"], signs.cuda())
    v8, vs = hadamard_quant_fp8(dev["v"], None)
    o = torch.empty((B, H, N, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    _lib.fa_fwd_fp8(q8, k8, v8, qs, ks, vs, o, lse, False, SCALE)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    del q8, k8, v8
    stack = {n: torch.cat([host[(n, p)] for p in PLANES], dim=1) for n in ("q", "k", "v")}  # [1, 4, N, D]
    qm, km, vm = oracle.fp8_dequantized(stack["q"], stack["k"], stack["v"], signs)
    rows = _rows()
    for i, p in enumerate(PLANES):
        if p < 2048:
            continue
        b, h = divmod(p, H)
        ro, _ = oracle.attention_fwd_rows(qm, km, vm, [(0, i, r) for r in rows], False, SCALE)
        got = o[b, h, rows].float().cpu().numpy().astype(np.float64)
        err = float(np.linalg.norm(got - ro) / np.linalg.norm(ro))
        assert err <= FP8_REL_RMS, f"plane {p}: FP8 O relative RMS {err:.4f} against the pipeline model"
    ln_n = np.full(N, np.log(N))  # non-causal: every row sees N zero scores
    for p in ZERO_PLANES:
        b, h = divmod(p, H)
        assert int(torch.count_nonzero(o[b, h])) == 0, f"plane {p} FP8 O not zero"
        check_lse(lse[b, h], ln_n, f"plane {p} FP8 LSE")
