"""CPU pins of the fp64 oracle.

Each test ties the oracle to something other than itself: the page's worked
two-block example (hand-derived golden values), closed forms, invariants,
central finite differences, and library routines (torch's fp64 CPU attention
with autograd, scipy's logsumexp and Hadamard matrix, torch's e4m3 cast).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ev(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}},
                      {"ln2": math.log(2.0), "ln3": math.log(3.0), "ln6": math.log(6.0)}))


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _torch_ref(q, k, v, causal, scale):
    """torch fp64 CPU attention with autograd (library cross-check)."""
    G = q.shape[1] // k.shape[1]
    qt = torch.tensor(q, requires_grad=True)
    kt = torch.tensor(k, requires_grad=True)
    vt = torch.tensor(v, requires_grad=True)
    ke = kt.repeat_interleave(G, dim=1)
    ve = vt.repeat_interleave(G, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, ke, ve, is_causal=causal, scale=scale)
    return o, qt, kt, vt


# ------------------------------------------------------------------ golden


def test_golden_two_block_forward_and_causal():
    g = json.load(open(os.path.join(GOLDEN, "two_block_worked_example.json")))
    inp = g["inputs"]
    q = np.array([_ev(x) for x in inp["q"]]).reshape(1, 1, 3, 1)
    k = np.array([_ev(x) for x in inp["k"]]).reshape(1, 1, 3, 1)
    v = np.array([_ev(x) for x in inp["v"]]).reshape(1, 1, 3, 1)
    scale = _ev(inp["scale"])
    for mode, causal in (("noncausal", False), ("causal", True)):
        o, lse = oracle.attention_fwd(q, k, v, causal, scale)
        np.testing.assert_allclose(o.ravel(), [_ev(x) for x in g[mode]["O"]], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse.ravel(), [_ev(x) for x in g[mode]["L"]], rtol=0, atol=1e-12)


def test_golden_two_block_recurrence_matches_page_values():
    """The page's two-block recurrence, run on the worked example, gives the
    stored intermediates, and its final O, L equal the oracle's."""
    g = json.load(open(os.path.join(GOLDEN, "two_block_worked_example.json")))
    inp, tb = g["inputs"], g["two_block"]
    kk = [_ev(x) for x in inp["k"]]
    vv = [_ev(x) for x in inp["v"]]
    s = [1.0 * x for x in kk]  # q = 1, scale = 1
    sp = tb["split"]
    m1 = max(s[:sp])
    l1 = sum(math.exp(x - m1) for x in s[:sp])
    o1 = sum(math.exp(x - m1) * vv[c] for c, x in enumerate(s[:sp]))
    m2 = max(m1, max(s[sp:]))
    l2 = math.exp(m1 - m2) * l1 + sum(math.exp(x - m2) for x in s[sp:])
    o2 = math.exp(m1 - m2) * o1 + sum(math.exp(x - m2) * vv[sp + c] for c, x in enumerate(s[sp:]))
    for name, val in (("m1", m1), ("l1", l1), ("Otilde1", o1), ("m2", m2), ("l2", l2), ("Otilde2", o2)):
        assert abs(val - _ev(tb[name])) < 1e-12, name
    q = np.ones((1, 1, 3, 1))
    o, lse = oracle.attention_fwd(q, np.array(kk).reshape(1, 1, 3, 1), np.array(vv).reshape(1, 1, 3, 1), False, 1.0)
    assert abs(o[0, 0, 2, 0] - o2 / l2) < 1e-12
    assert abs(lse[0, 0, 2] - (m2 + math.log(l2))) < 1e-12
    assert abs(o2 / l2 - _ev(tb["O"])) < 1e-12


def test_golden_backward():
    g = json.load(open(os.path.join(GOLDEN, "two_block_worked_example.json")))
    inp, bw = g["inputs"], g["backward_noncausal"]
    sh = (1, 1, 3, 1)
    q, k, v, dO = (np.array([_ev(x) for x in inp[n]]).reshape(sh) for n in ("q", "k", "v", "dO"))
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, False, 1.0)
    np.testing.assert_allclose(dq.ravel(), [_ev(x) for x in bw["dQ"]], atol=1e-12)
    np.testing.assert_allclose(dk.ravel(), [_ev(x) for x in bw["dK"]], atol=1e-12)
    np.testing.assert_allclose(dv.ravel(), [_ev(x) for x in bw["dV"]], atol=1e-12)


# --------------------------------------------------------- library checks


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,N,d", [(1, 1, 1, 1, 4), (2, 2, 2, 17, 8), (1, 4, 2, 33, 16), (2, 3, 1, 9, 5)])
def test_forward_matches_torch_fp64(B, Hq, Hkv, N, d, causal):
    q = _rand((B, Hq, N, d), 1)
    k = _rand((B, Hkv, N, d), 2)
    v = _rand((B, Hkv, N, d), 3)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attention_fwd(q, k, v, causal, scale)
    ot, *_ = _torch_ref(q, k, v, causal, scale)
    np.testing.assert_allclose(o, ot.detach().numpy(), rtol=0, atol=1e-12)
    # L against scipy's logsumexp of the explicitly formed masked scores
    from scipy.special import logsumexp
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            s = scale * q[b, h] @ k[b, h // G].T
            if causal:
                s = np.where(np.tril(np.ones((N, N), bool)), s, -np.inf)
            np.testing.assert_allclose(lse[b, h], logsumexp(s, axis=1), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,N,d", [(1, 1, 1, 5, 4), (2, 4, 2, 19, 8), (1, 3, 1, 12, 6)])
def test_backward_matches_torch_autograd(B, Hq, Hkv, N, d, causal):
    q = _rand((B, Hq, N, d), 4)
    k = _rand((B, Hkv, N, d), 5)
    v = _rand((B, Hkv, N, d), 6)
    dO = _rand((B, Hq, N, d), 7)
    scale = 0.7 / math.sqrt(d)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, causal, scale)
    ot, qt, kt, vt = _torch_ref(q, k, v, causal, scale)
    ot.backward(torch.tensor(dO))
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-11)


# ---------------------------------------------------- finite differences


@pytest.mark.parametrize("causal", [False, True])
def test_backward_central_finite_differences(causal):
    """Pins the backward to the forward without any library: loss = sum(dO o O)."""
    B, Hq, Hkv, N, d = 1, 2, 1, 7, 3
    q = _rand((B, Hq, N, d), 11)
    k = _rand((B, Hkv, N, d), 12)
    v = _rand((B, Hkv, N, d), 13)
    dO = _rand((B, Hq, N, d), 14)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, causal, scale)
    h = 1e-6

    def loss(q_, k_, v_):
        o, _ = oracle.attention_fwd(q_, k_, v_, causal, scale)
        return float((o * dO).sum())

    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}; args_p[name] = xp
            args_m = {"q": q, "k": k, "v": v}; args_m[name] = xm
            num[idx] = (loss(**{a + "_": b for a, b in args_p.items()})
                        - loss(**{a + "_": b for a, b in args_m.items()})) / (2 * h)
        np.testing.assert_allclose(grad, num, atol=2e-8, err_msg=name)


def test_lse_is_gradient_consistent():
    """dL_r/dq_r = scale * sum_c P_rc k_c (softmax-weighted key mean), checked
    by finite differences on L: pins the L output's units (natural log)."""
    N, d = 6, 4
    q = _rand((1, 1, N, d), 21)
    k = _rand((1, 1, N, d), 22)
    v = _rand((1, 1, N, d), 23)
    scale = 0.5
    _, lse = oracle.attention_fwd(q, k, v, False, scale)
    o_k, _ = oracle.attention_fwd(q, k, k, False, scale)  # V = K gives sum_c P k_c
    h = 1e-6
    for r in range(N):
        for t in range(d):
            qp = q.copy(); qp[0, 0, r, t] += h
            qm = q.copy(); qm[0, 0, r, t] -= h
            num = (oracle.attention_fwd(qp, k, v, False, scale)[1][0, 0, r]
                   - oracle.attention_fwd(qm, k, v, False, scale)[1][0, 0, r]) / (2 * h)
            assert abs(num - scale * o_k[0, 0, r, t]) < 1e-8


# --------------------------------------------------------------- invariants


@pytest.mark.parametrize("causal", [False, True])
def test_rows_are_probabilities(causal):
    """With V = I (d = N) the output row is the probability row itself."""
    N = 13
    q = _rand((1, 1, N, N), 31)
    k = _rand((1, 1, N, N), 32)
    v = np.eye(N).reshape(1, 1, N, N)
    p, _ = oracle.attention_fwd(q, k, v, causal, 0.3)
    p = p[0, 0]
    assert np.all(p >= 0)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    if causal:
        assert np.all(p[np.triu_indices(N, 1)] == 0.0)


def test_shift_invariance_per_row():
    """Adding c_r to every score of row r leaves O unchanged and shifts L by c_r.
    Realised with one extra feature: q' = [q, c/scale], k' = [k, 1]."""
    B, H, N, d = 1, 2, 11, 5
    q = _rand((B, H, N, d), 41)
    k = _rand((B, H, N, d), 42)
    v = _rand((B, H, N, d), 43)
    c = 3.0 * _rand((B, H, N, 1), 44)
    scale = 0.4
    for causal in (False, True):
        o, lse = oracle.attention_fwd(q, k, v, causal, scale)
        q2 = np.concatenate([q, c / scale], axis=-1)
        k2 = np.concatenate([k, np.ones((B, H, N, 1))], axis=-1)
        v2 = np.concatenate([v, np.zeros((B, H, N, 1))], axis=-1)
        o2, lse2 = oracle.attention_fwd(q2, k2, v2, causal, scale)
        np.testing.assert_allclose(o2[..., :d], o, atol=1e-12)
        np.testing.assert_allclose(lse2, lse + c[..., 0], atol=1e-12)


def test_causal_row0_is_v0_exactly():
    B, Hq, Hkv, N, d = 2, 4, 2, 9, 8
    q = _rand((B, Hq, N, d), 51)
    k = _rand((B, Hkv, N, d), 52)
    v = _rand((B, Hkv, N, d), 53)
    o, lse = oracle.attention_fwd(q, k, v, True, 0.35)
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(o[b, h, 0], v[b, h // 2, 0])
            assert abs(lse[b, h, 0] - 0.35 * q[b, h, 0] @ k[b, h // 2, 0]) < 1e-13


def test_zero_query_closed_form():
    """Q = 0: uniform weights over visible keys, O = mean of visible V,
    L = ln(#visible)."""
    B, H, N, d = 1, 1, 10, 3
    q = np.zeros((B, H, N, d))
    k = _rand((B, H, N, d), 61)
    v = _rand((B, H, N, d), 62)
    o, lse = oracle.attention_fwd(q, k, v, True, 1.0)
    for r in range(N):
        np.testing.assert_allclose(o[0, 0, r], v[0, 0, : r + 1].mean(axis=0), atol=1e-13)
        assert abs(lse[0, 0, r] - math.log(r + 1)) < 1e-13
    o, lse = oracle.attention_fwd(q, k, v, False, 1.0)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0].mean(axis=0), (N, d)), atol=1e-13)
    np.testing.assert_allclose(lse, math.log(N), atol=1e-13)


def test_two_block_identity_random():
    """Splitting the keys in two and merging (m, l, O~) by the page's
    recurrence reproduces the full-row O and L (non-causal)."""
    N, d, split = 40, 6, 17
    q = _rand((1, 1, N, d), 71)
    k = _rand((1, 1, N, d), 72)
    v = _rand((1, 1, N, d), 73)
    scale = 0.8
    o, lse = oracle.attention_fwd(q, k, v, False, scale)
    # attention of every query against each key block alone (keys are a
    # separate problem with fewer rows: use the rows oracle on a padded copy)
    def block(lo, hi):
        n = hi - lo
        kb, vb = k[:, :, lo:hi], v[:, :, lo:hi]
        ob = np.zeros((N, d)); lb = np.zeros(N)
        for r in range(N):
            qq = np.repeat(q[:, :, r:r + 1], n, axis=2)
            orow, lrow = oracle.attention_fwd(qq, kb, vb, False, scale)
            ob[r], lb[r] = orow[0, 0, 0], lrow[0, 0, 0]
        return ob, lb
    o1, L1 = block(0, split)
    o2, L2 = block(split, N)
    # block results carry O = O~/l and L = m + ln l; recombine with the
    # running max of the recurrence
    m = np.maximum(L1, L2)
    l = np.exp(L1 - m) + np.exp(L2 - m)
    o_merged = (np.exp(L1 - m)[:, None] * o1 + np.exp(L2 - m)[:, None] * o2) / l[:, None]
    np.testing.assert_allclose(o_merged, o[0, 0], atol=1e-13)
    np.testing.assert_allclose(m + np.log(l), lse[0, 0], atol=1e-13)


def test_gqa_head_mapping_equals_expanded_mha():
    B, Hq, Hkv, N, d = 1, 6, 2, 8, 4
    q = _rand((B, Hq, N, d), 81)
    k = _rand((B, Hkv, N, d), 82)
    v = _rand((B, Hkv, N, d), 83)
    dO = _rand((B, Hq, N, d), 84)
    o, lse = oracle.attention_fwd(q, k, v, True, 0.5)
    ke, ve = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    o2, lse2 = oracle.attention_fwd(q, ke, ve, True, 0.5)
    np.testing.assert_array_equal(o, o2)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, True, 0.5)
    dq2, dk2, dv2 = oracle.attention_bwd(q, ke, ve, dO, True, 0.5)
    np.testing.assert_allclose(dq, dq2, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(B, Hkv, 3, N, d).sum(axis=2), atol=1e-12)
    np.testing.assert_allclose(dv, dv2.reshape(B, Hkv, 3, N, d).sum(axis=2), atol=1e-12)


def test_rows_and_group_entry_points_agree_with_full():
    B, Hq, Hkv, N, d = 2, 4, 2, 21, 8
    q = _rand((B, Hq, N, d), 91)
    k = _rand((B, Hkv, N, d), 92)
    v = _rand((B, Hkv, N, d), 93)
    dO = _rand((B, Hq, N, d), 94)
    o, lse = oracle.attention_fwd(q, k, v, True, 0.3)
    rows = [(1, 3, 20), (0, 0, 0), (1, 2, 7)]
    orow, lrow = oracle.attention_fwd_rows(q, k, v, rows, True, 0.3)
    for i, (b, h, r) in enumerate(rows):
        np.testing.assert_array_equal(orow[i], o[b, h, r])
        assert lrow[i] == lse[b, h, r]
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, True, 0.3)
    gq, gk, gv = oracle.attention_bwd_group(q, k, v, dO, 1, 1, True, 0.3)
    np.testing.assert_array_equal(gq, dq[1, 2:4])
    np.testing.assert_array_equal(gk, dk[1, 1])
    np.testing.assert_array_equal(gv, dv[1, 1])


def test_invalid_arguments_rejected():
    q = np.zeros((1, 3, 4, 2))
    k = np.zeros((1, 2, 4, 2))
    with pytest.raises(ValueError):
        oracle.attention_fwd(q, k, k, False, 1.0)


# -------------------------------------------------------------- FP8 model


@pytest.mark.parametrize("d", [2, 8, 64, 128])
def test_hadamard_is_scipy_sylvester_with_signs(d):
    from scipy.linalg import hadamard as sp_hadamard
    rng = np.random.default_rng(d)
    s = rng.choice([-1.0, 1.0], size=d)
    M = oracle.hadamard(np.eye(d), s)  # row i = s_i H[i, :] / sqrt(d)
    np.testing.assert_allclose(M, np.diag(s) @ sp_hadamard(d) / math.sqrt(d), atol=1e-15)
    np.testing.assert_allclose(M @ M.T, np.eye(d), atol=1e-13)


def test_hadamard_preserves_scores():
    d = 128
    rng = np.random.default_rng(5)
    s = rng.choice([-1.0, 1.0], size=d)
    q = rng.standard_normal((20, d))
    k = rng.standard_normal((30, d))
    np.testing.assert_allclose(oracle.hadamard(q, s) @ oracle.hadamard(k, s).T, q @ k.T, atol=1e-11)


def test_e4m3_matches_torch_cast_in_range():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000) * 30.0,
        rng.standard_normal(5000) * 1e-2,                 # subnormal range
        np.array([0.0, -0.0, 448.0, -448.0, 2 ** -9, 2 ** -10, 3 * 2 ** -11]),
    ])
    x = np.clip(x, -448.0, 448.0)
    # compare on values exactly representable in fp32 (torch casts from fp32)
    x32 = x.astype(np.float32).astype(np.float64)
    ref = torch.tensor(x32, dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.e4m3_round(x32), ref)


def test_e4m3_saturates_and_ties_to_even():
    vals = oracle.e4m3_round(np.array([1000.0, -1e6, 464.0, 1.0625, 1.1875, 2 ** -10, 3 * 2 ** -10]))
    # 464 is halfway between 448 and 480: ties to even mantissa -> 448; 1.0625 halfway 1 and 1.125 -> 1;
    # 1.1875 halfway 1.125 and 1.25 -> 1.25; 2^-10 halfway 0 and 2^-9 -> 0; 3*2^-10 halfway 2^-9, 2^-8 -> 2^-8
    np.testing.assert_array_equal(vals, [448.0, -448.0, 448.0, 1.0, 1.25, 0.0, 2 ** -8])


def test_fp8_reference_without_quantisation_error_is_exact():
    """On inputs already on the e4m3 grid with amax 448 and no rotation, the
    FP8 model returns the exact attention."""
    rng = np.random.default_rng(9)
    N, d = 16, 8
    def on_grid(shape):
        x = oracle.e4m3_round(rng.standard_normal(shape) * 20)
        x.flat[0] = 448.0
        return x
    q, k, v = on_grid((1, 1, N, d)), on_grid((1, 1, N, d)), on_grid((1, 1, N, d))
    o, lse = oracle.attention_fwd(q, k, v, False, 0.01)
    o8, lse8 = oracle.fp8_reference(q, k, v, None, False, 0.01)
    np.testing.assert_allclose(o8, o, atol=1e-12)


# ------------------------------------------------------- sliding window


def _window_mask(N, window):
    r = np.arange(N)[:, None]
    c = np.arange(N)[None, :]
    return (c <= r) & (r - c < window)


@pytest.mark.parametrize("window", [1, 2, 5, 16, 40])
def test_window_matches_torch_masked_sdpa(window):
    """Sliding window = causal mask plus r - c < W; torch's SDPA with that
    boolean mask (fp64, autograd) is the independent reference."""
    B, Hq, Hkv, N, d = 2, 4, 2, 23, 8
    q, k, v, dO = (_rand((B, h, N, d), s) for h, s in ((Hq, 11), (Hkv, 12), (Hkv, 13), (Hq, 14)))
    scale = 0.9 / math.sqrt(d)
    o, lse = oracle.attention_fwd(q, k, v, True, scale, window=window)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, True, scale, window=window)
    G = Hq // Hkv
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    mask = torch.tensor(_window_mask(N, window))
    ot = torch.nn.functional.scaled_dot_product_attention(
        qt, kt.repeat_interleave(G, 1), vt.repeat_interleave(G, 1), attn_mask=mask, scale=scale)
    ot.backward(torch.tensor(dO))
    np.testing.assert_allclose(o, ot.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-11)
    from scipy.special import logsumexp
    for b in range(B):
        for h in range(Hq):
            s = np.where(_window_mask(N, window), scale * q[b, h] @ k[b, h // G].T, -np.inf)
            np.testing.assert_allclose(lse[b, h], logsumexp(s, axis=1), atol=1e-12)


def test_window_one_closed_form():
    """A window of one key: every query sees only itself, so O = V row for
    row, L = its own score, dQ = dK = 0 and dV = dO (summed over a group)."""
    B, Hq, Hkv, N, d = 1, 2, 1, 9, 4
    q, k, v, dO = (_rand((B, h, N, d), s) for h, s in ((Hq, 21), (Hkv, 22), (Hkv, 23), (Hq, 24)))
    o, lse = oracle.attention_fwd(q, k, v, True, 0.5, window=1)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, True, 0.5, window=1)
    assert np.array_equal(o, np.repeat(v, 2, axis=1))
    np.testing.assert_allclose(lse, 0.5 * np.einsum("bhnd,bnd->bhn", q, k[:, 0]), atol=1e-14)
    assert np.abs(dq).max() == 0 and np.abs(dk).max() == 0
    np.testing.assert_allclose(dv[:, 0], dO.sum(axis=1), atol=1e-14)


def test_window_at_least_n_is_plain_causal():
    B, Hq, Hkv, N, d = 1, 2, 2, 12, 4
    q, k, v = (_rand((B, h, N, d), s) for h, s in ((Hq, 31), (Hkv, 32), (Hkv, 33)))
    for w in (N, N + 7):
        a = oracle.attention_fwd(q, k, v, True, 0.3, window=w)
        b = oracle.attention_fwd(q, k, v, True, 0.3)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ------------------------------------------------- packed variable lengths


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 3)])
def test_varlen_matches_block_diagonal_sdpa(causal, window):
    """Packed sequences attend only within themselves: torch SDPA on the
    whole packed batch with a block-diagonal (and causal / window) mask is the
    independent reference, forward and backward.  Includes an empty sequence
    and one of a single row."""
    lengths = [5, 0, 1, 9, 4]
    Hq, Hkv, d = 4, 2, 8
    total = sum(lengths)
    q, k, v, dO = (_rand((total, h, d), s) for h, s in ((Hq, 41), (Hkv, 42), (Hkv, 43), (Hq, 44)))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    scale = 0.5
    o, lse = oracle.attention_fwd_varlen(q, k, v, cu, causal, scale, window)
    dq, dk, dv = oracle.attention_bwd_varlen(q, k, v, dO, cu, causal, scale, window)
    seq = np.repeat(np.arange(len(lengths)), lengths)
    pos = np.concatenate([np.arange(n) for n in lengths])
    mask = seq[:, None] == seq[None, :]
    if causal:
        mask &= pos[None, :] <= pos[:, None]
    if window:
        mask &= pos[:, None] - pos[None, :] < window
    G = Hq // Hkv
    qt, kt, vt = (torch.tensor(x.transpose(1, 0, 2)[None].copy(), requires_grad=True) for x in (q, k, v))
    ot = torch.nn.functional.scaled_dot_product_attention(
        qt, kt.repeat_interleave(G, 1), vt.repeat_interleave(G, 1), attn_mask=torch.tensor(mask), scale=scale)
    ot.backward(torch.tensor(dO.transpose(1, 0, 2)[None].copy()))
    np.testing.assert_allclose(o, ot.detach().numpy()[0].transpose(1, 0, 2), atol=1e-12)
    np.testing.assert_allclose(dq, qt.grad.numpy()[0].transpose(1, 0, 2), atol=1e-11)
    np.testing.assert_allclose(dk, kt.grad.numpy()[0].transpose(1, 0, 2), atol=1e-11)
    np.testing.assert_allclose(dv, vt.grad.numpy()[0].transpose(1, 0, 2), atol=1e-11)
    from scipy.special import logsumexp
    for h in range(Hq):
        s = np.where(mask, scale * q[:, h] @ k[:, h // G].T, -np.inf)
        np.testing.assert_allclose(lse[h], logsumexp(s, axis=1), atol=1e-12)


def test_thread_count_does_not_change_results():
    """The OpenMP thread count (set for the single-thread timing baseline)
    leaves every result bit-identical: each output element is computed by
    one thread in a fixed order."""
    g = torch.Generator().manual_seed(3)
    q, k, v, dO = (torch.randn(1, 4, 97, 64, generator=g, dtype=torch.float64) for _ in range(4))
    k, v = k[:, :2], v[:, :2]
    try:
        oracle.set_threads(1)
        o1, l1 = oracle.attention_fwd(q, k, v, True, 0.125)
        g1 = oracle.attention_bwd(q, k, v, dO, True, 0.125)
        assert oracle.set_threads(3) == 3
        o3, l3 = oracle.attention_fwd(q, k, v, True, 0.125)
        g3 = oracle.attention_bwd(q, k, v, dO, True, 0.125)
    finally:
        oracle.set_threads(0)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)
    for a, b in zip(g1, g3):
        assert np.array_equal(a, b)
