"""FP8 path parity: the random-sign Hadamard + e4m3 quantisation against the
oracle's dense Hadamard and e4m3 grid, and the FP8 forward against the fp64
oracle.

Tolerances: the quantised codes must be a correct rounding of the exact
rotated value (within half an e4m3 ulp, plus fp32 noise); without the
rotation they must equal the oracle's codes exactly (both sides decide them
in fp32, exact ties included).  The forward is
gated on its relative RMS error ||O - O_model||_F / ||O_model||_F <= 0.03,
where O_model is the exact fp64 attention of the inputs as the FP8 path holds
them (the oracle's rotation and per-tensor e4m3 quantise-dequantise of Q, K
and V): what remains is the kernel's own rounding (P in e4m3, fp32
accumulation).  Against the exact attention of the unquantised bf16 inputs
the same measure is printed, and the rotated path must be no worse than the
same kernel without the rotation (the FlashAttention-3 summary's FP8 and
incoherent processing section reports the rotation lowering the error).
0.03 against exact attention is not met on the outlier workload by any
kernel that consumes per-tensor e4m3 inputs: the oracle's input model alone
is 0.096 from it (Q or K quantised alone already 0.07)."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_85_gb300 import _lib, attention_fwd_fp8, hadamard_quant_fp8
from exact_attention_85_gb300.inputs import WORKLOADS, make_custom, make_inputs, random_signs

from _tol import FP8_REL_RMS

pytestmark = pytest.mark.gpu


def _e4m3_half_ulp(y):
    y = np.abs(y)
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    return 0.5 * np.exp2(e - 3)


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("rotate", [True, False])
def test_hadamard_quant_matches_oracle(cuda_lib, d, rotate):
    g = torch.Generator().manual_seed(d + rotate)
    rows = 3001
    x = torch.randn(rows, d, generator=g)
    x[torch.randperm(rows * d, generator=g)[:50] // d, 3] *= 50.0
    x = x.to(torch.bfloat16)
    signs = random_signs(d, g) if rotate else None
    x8, descale = hadamard_quant_fp8(x.cuda(), None if signs is None else signs.cuda())
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    xr = oracle.hadamard(x, signs) if rotate else x.double().numpy()
    sigma = np.abs(xr).max() / 448.0
    ds = float(descale.item())
    assert abs(ds - sigma) <= 1e-5 * sigma
    deq = x8.float().cpu().numpy().astype(np.float64) * ds
    tol = _e4m3_half_ulp(xr / sigma) * sigma * 1.001 + 1e-6 * sigma
    err = np.abs(deq - xr)
    assert (err <= tol).all(), f"{int((err > tol).sum())} codes off the nearest e4m3 value"
    if not rotate:
        # without the rotation every input is exact in fp32 and both sides
        # decide the code in fp32 the same way: the codes (exact ties
        # included) and the scale are identical
        xm, _, _ = oracle.fp8_dequantized(x[None, None], x[None, None], x[None, None], None)
        assert ds == float(np.float32(np.abs(x.double().numpy()).max()) / np.float32(448.0))
        np.testing.assert_array_equal(deq, xm[0, 0])


def _fp8_forward(x, signs, causal, scale):
    q8, qs = hadamard_quant_fp8(x["q"].cuda(), None if signs is None else signs.cuda())
    k8, ks = hadamard_quant_fp8(x["k"].cuda(), None if signs is None else signs.cuda())
    v8, vs = hadamard_quant_fp8(x["v"].cuda(), None)
    o, lse = attention_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert _lib.fa_get_device_status() == _lib.FA_OK
    return o, lse


def _rel_rms(got, ref):
    """RMS error relative to the RMS of the reference output."""
    g = got.float().cpu().numpy().astype(np.float64) if hasattr(got, "cpu") else got
    return float(np.linalg.norm(g - ref) / np.linalg.norm(ref))


def _rms_vs_v(got, ref, v):
    """RMS error of O relative to the RMS of the values V."""
    g = got.float().cpu().numpy().astype(np.float64) if hasattr(got, "cpu") else got
    v_rms = float(v.float().pow(2).mean().sqrt()) if hasattr(v, "float") else float(np.sqrt(np.mean(v ** 2)))
    return float(np.sqrt(np.mean((g - ref) ** 2)) / v_rms)


@pytest.mark.parametrize("B,Hq,Hkv,N,causal", [(1, 2, 2, 300, False), (2, 4, 2, 513, True), (1, 1, 1, 128, False)])
def test_fp8_forward_small(cuda_lib, B, Hq, Hkv, N, causal):
    d = 128
    x = make_custom(B, Hq, Hkv, N, d, torch.bfloat16, seed=N + 7, with_grad=False)
    signs = random_signs(d, torch.Generator().manual_seed(N))
    scale = d ** -0.5
    o, lse = _fp8_forward(x, signs, causal, scale)
    o_ref, lse_ref = oracle.attention_fwd(x["q"], x["k"], x["v"], causal, scale)
    # kernel parity: against the exact attention of the quantised inputs
    o_model, lse_model = oracle.fp8_reference(x["q"], x["k"], x["v"], signs, causal, scale)
    kernel = _rel_rms(o, o_model)
    print(f"fp8 small: kernel vs model {kernel:.4f}; vs exact {_rel_rms(o, o_ref):.4f} "
          f"(input model vs exact {_rel_rms(o_model, o_ref):.4f}; RMS error / RMS(V) {_rms_vs_v(o, o_ref, x['v']):.4f})")
    assert kernel <= FP8_REL_RMS
    assert float(np.abs(lse.cpu().numpy() - lse_model).max()) < 0.1
    assert torch.isfinite(o).all()


def _plane_rows(B, Hq, N, full_planes):
    """Every row of the listed (b, h) planes plus the first and last 128 rows
    of every plane: all CTAs of three planes and the first and last Q-tile
    CTAs of the others (catches CTA-order and plane-index mistakes)."""
    rows = set()
    for b, h in full_planes:
        rows.update((b, h, r) for r in range(N))
    edge = list(range(min(128, N))) + list(range(max(0, N - 128), N))
    for b in range(B):
        for h in range(Hq):
            rows.update((b, h, r) for r in edge)
    return sorted(rows)


def test_fp8_outlier_workload_full_size(cuda_lib):
    """B4 H16 N8192 d128 with 0.1% of Q/K entries scaled by 50, non-causal:
    the rotated and the plain FP8 forward within 0.03 relative RMS of the
    oracle's model of their own pipeline, on every row of the first, a middle
    and the last (batch, head) plane and the first and last 128 rows of every
    plane; the rotated path no worse than plain FP8 against exact attention."""
    w = WORKLOADS["fp8_b4_h16_n8k_outliers"]
    x = make_inputs(w, with_grad=False)
    rows = _plane_rows(w.B, w.Hq, w.N, [(0, 0), (w.B // 2, w.Hq // 2), (w.B - 1, w.Hq - 1)])
    o_ref, _ = oracle.attention_fwd_rows(x["q"], x["k"], x["v"], rows, w.causal, w.scale)
    idx = tuple(np.array(rows).T)
    # keep only the checked rows of each GPU output (host memory is bounded)
    got = {}
    for signs, tag in ((x["signs"], "hadamard"), (None, "plain")):
        o, _ = _fp8_forward(x, signs, w.causal, w.scale)
        assert torch.isfinite(o).all()
        got[tag] = o[idx].float().cpu().numpy().astype(np.float64)
        del o
    for signs, tag in ((x["signs"], "hadamard"), (None, "plain")):
        qm, km, vm = oracle.fp8_dequantized(x["q"], x["k"], x["v"], signs)
        o_model, _ = oracle.attention_fwd_rows(qm, km, vm, rows, w.causal, w.scale)
        del qm, km, vm
        dev = _rel_rms(got[tag], o_model)
        print(f"fp8 outliers {tag}: kernel vs pipeline model {dev:.4f}; model vs exact {_rel_rms(o_model, o_ref):.4f}")
        assert dev <= FP8_REL_RMS
    e_had = _rel_rms(got["hadamard"], o_ref)
    e_plain = _rel_rms(got["plain"], o_ref)
    # printed only: the error relative to the RMS of all of V (every head of
    # V is drawn from the same distribution)
    print(f"fp8 outliers vs exact attention (relative RMS, bound 0.03 not met by e4m3 inputs): "
          f"hadamard {e_had:.4f}, plain {e_plain:.4f}, ratio {e_plain / e_had:.2f}; RMS error / RMS(V): "
          f"hadamard {_rms_vs_v(got['hadamard'], o_ref, x['v']):.4f}, "
          f"plain {_rms_vs_v(got['plain'], o_ref, x['v']):.4f}")
    assert e_had <= e_plain
