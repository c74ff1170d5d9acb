"""How close can any FP8 forward come to exact attention on the outlier
workload?  CPU only: the oracle's model of the FP8 inputs (rotation, e4m3
quantise-dequantise) fed to the exact fp64 attention.

The FlashAttention-3 summary page (FP8 and incoherent processing) runs FP8
attention on N(0,1) inputs with 0.1% large entries and reports the random
orthogonal (Hadamard) rotation lowering the error.  The stated bound for this
workload is a relative RMS error of O <= 0.03 against exact attention.  These
tests pin the reading that the bound is out of reach for e4m3 inputs, whatever
the kernel does: the inputs alone, before any kernel arithmetic, put O about
0.1 away from exact attention, and a per-row scale for Q and K (the next
scaling scheme one would try) does not lower that floor on the rotated path.
"""
import numpy as np
import pytest

import oracle
from exact_attention_85_gb300.inputs import WORKLOADS, make_inputs

FP8_REL_RMS = 0.03


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _qdq(t, sigma):
    return oracle.e4m3_round(t / sigma) * sigma


def _sigma(t):
    return np.abs(t).max() / 448.0


def _qdq_rows(t):
    s = np.abs(t).max(axis=-1, keepdims=True) / 448.0
    s[s == 0] = 1.0
    return oracle.e4m3_round(t / s) * s


@pytest.fixture(scope="module")
def c5():
    """Four (batch, head) planes of the outlier workload, 16 sampled query
    rows each, with the per-tensor scales of the whole tensors."""
    w = WORKLOADS["fp8_b4_h16_n8k_outliers"]
    x = make_inputs(w, with_grad=False)
    q, k, v = (x[n].double().numpy() for n in ("q", "k", "v"))
    s = x["signs"].double().numpy()
    qh, kh = oracle.hadamard(q, s), oracle.hadamard(k, s)
    sig = {"q": _sigma(q), "k": _sigma(k), "v": _sigma(v), "qh": _sigma(qh), "kh": _sigma(kh)}
    planes = [(0, 0), (1, 7), (2, 11), (3, 15)]
    sub = lambda t: np.ascontiguousarray(np.stack([t[b, h] for b, h in planes])[None])
    t = {"q": sub(q), "k": sub(k), "v": sub(v), "qh": sub(qh), "kh": sub(kh)}
    g = np.random.default_rng(5)
    rows = [(0, p, int(g.integers(w.N))) for p in range(len(planes)) for _ in range(16)]
    o_ref, _ = oracle.attention_fwd_rows(t["q"], t["k"], t["v"], rows, w.causal, w.scale)
    return w, t, sig, rows, o_ref


def _err(c5, qq, kk, vv):
    w, _, _, rows, o_ref = c5
    o, _ = oracle.attention_fwd_rows(qq, kk, vv, rows, w.causal, w.scale)
    return _rel(o, o_ref)


def test_input_quantisation_alone_exceeds_the_bound(c5):
    _, t, sig, _, _ = c5
    vq = _qdq(t["v"], sig["v"])
    rot = _err(c5, _qdq(t["qh"], sig["qh"]), _qdq(t["kh"], sig["kh"]), vq)
    plain = _err(c5, _qdq(t["q"], sig["q"]), _qdq(t["k"], sig["k"]), vq)
    q_only = _err(c5, _qdq(t["qh"], sig["qh"]), t["kh"], t["v"])
    v_only = _err(c5, t["q"], t["k"], vq)
    print(f"input model vs exact: rotated {rot:.4f}, plain {plain:.4f}, rotated Q only {q_only:.4f}, V only {v_only:.4f}")
    # the rotation lowers the error, as the page reports ...
    assert rot < plain / 1.5
    # ... but quantising Q alone already exceeds the bound, and V alone does not
    assert q_only > 2 * FP8_REL_RMS
    assert v_only < FP8_REL_RMS
    assert rot > 3 * FP8_REL_RMS


def test_per_row_scales_do_not_lower_the_rotated_floor(c5):
    _, t, sig, _, _ = c5
    vq = _qdq(t["v"], sig["v"])
    per_tensor = _err(c5, _qdq(t["qh"], sig["qh"]), _qdq(t["kh"], sig["kh"]), vq)
    per_row = _err(c5, _qdq_rows(t["qh"]), _qdq_rows(t["kh"]), vq)
    print(f"rotated: per-tensor scales {per_tensor:.4f}, per-row Q/K scales {per_row:.4f}")
    # e4m3 keeps a 3-bit mantissa at every scale: moving the scale per row
    # changes which grid points the values land on, not how fine the grid is
    assert per_row > 0.9 * per_tensor
    assert per_row > 3 * FP8_REL_RMS
