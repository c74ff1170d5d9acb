"""Plants plausible mistakes in a copy of the oracle's C source and checks
that the pins catch each one.

Every mutant is compiled from a modified copy of ``oracle/fa_oracle.c`` into
a temporary directory (the committed oracle is never touched) and swapped in
for the duration of one battery of pin checks.  A mutant that passes every
check would mean the pins leave that part of the oracle unconstrained.
"""
import ctypes
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "fa_oracle.c")

MUTANTS = {
    "dq_drops_scale": ("dqr[t] += scale * ds * kc[t];", "dqr[t] += ds * kc[t];"),
    "causal_off_by_one": ("causal ? (r + 1 < N ? r + 1 : N) : N", "causal ? (r + 2 < N ? r + 2 : N) : N"),
    "ds_wrong_sign": ("double ds = p * (dp - Dg[idx]);", "double ds = p * (dp + Dg[idx]);"),
    "gqa_wrong_head": ("long G = Hq / Hkv, hk = hq / G;", "long G = Hq / Hkv, hk = hq % Hkv;"),
    "lse_drops_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "dk_wrong_operand": ("dkc[t] += scale * ds * qr[t];", "dkc[t] += scale * ds * dor[t];"),
    "dv_wrong_operand": ("dvc[t] += p * dor[t];", "dvc[t] += p * qr[t];"),
    "o_not_normalised": ("double p = s[c] / l;", "double p = s[c];"),
    "hadamard_ignores_signs": ("(signs ? signs[i] : 1.0)", "1.0"),
    "hadamard_transposed_index": ("sylvester(i, j)", "sylvester(i, (j + 1) % d)"),
    "e4m3_ties_away": ("nearbyint(a / quantum)", "floor(a / quantum + 0.5)"),
    "e4m3_no_saturation": ("if (r > 448.0) r = 448.0;", ""),
    "window_keys_off_by_one": ("r - window + 1 > 0) ? r - window + 1 : 0", "r - window > 0) ? r - window : 0"),
    "window_rows_off_by_one": ("c + window < N) ? c + window : N", "c + window + 1 < N) ? c + window + 1 : N"),
    "window_ignored_by_dk_dv": ("*r1 = (window > 0 && c + window < N) ? c + window : N;", "*r1 = N;"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor missing for {name}"
    mutated = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                    "-o", str(so), str(c), "-lm"], check=True)
    return str(so)


def _battery():
    """Returns the list of failed check names (empty: all pins hold)."""
    failed = []
    rng = np.random.default_rng(123)

    def torch_ref(q, k, v, causal, scale, dO):
        G = q.shape[1] // k.shape[1]
        qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        o = torch.nn.functional.scaled_dot_product_attention(
            qt, kt.repeat_interleave(G, 1), vt.repeat_interleave(G, 1),
            is_causal=causal, scale=scale)
        o.backward(torch.tensor(dO))
        return o.detach().numpy(), qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()

    for causal in (False, True):
        B, Hq, Hkv, N, d = 1, 4, 2, 9, 4
        q, k, v, dO = (rng.standard_normal(s) for s in
                       ((B, Hq, N, d), (B, Hkv, N, d), (B, Hkv, N, d), (B, Hq, N, d)))
        scale = 0.6
        o_ref, dq_ref, dk_ref, dv_ref = torch_ref(q, k, v, causal, scale, dO)
        o, lse = oracle.attention_fwd(q, k, v, causal, scale)
        if not np.allclose(o, o_ref, atol=1e-10):
            failed.append(f"fwd_O_causal{causal}")
        s = scale * np.einsum("bhnd,bhmd->bhnm", q, np.repeat(k, 2, axis=1))
        if causal:
            s = np.where(np.tril(np.ones((N, N), bool)), s, -np.inf)
        from scipy.special import logsumexp
        if not np.allclose(lse, logsumexp(s, axis=-1), atol=1e-10):
            failed.append(f"fwd_L_causal{causal}")
        dq, dk, dv = oracle.attention_bwd(q, k, v, dO, causal, scale)
        for nm, a, b in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
            if not np.allclose(a, b, atol=1e-10):
                failed.append(f"bwd_{nm}_causal{causal}")

    # sliding window: closed forms for windows of one and two keys
    B, Hq, Hkv, N, d = 1, 4, 2, 7, 4
    q, k, v, dO = (rng.standard_normal(sh) for sh in
                   ((B, Hq, N, d), (B, Hkv, N, d), (B, Hkv, N, d), (B, Hq, N, d)))
    scale = 0.7
    kx, vx = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    o1, l1 = oracle.attention_fwd(q, k, v, True, scale, window=1)
    if not (np.allclose(o1, vx, atol=1e-14) and
            np.allclose(l1, scale * np.einsum("bhnd,bhnd->bhn", q, kx), atol=1e-12)):
        failed.append("window1_fwd")
    dq1, dk1, dv1 = oracle.attention_bwd(q, k, v, dO, True, scale, window=1)
    if not (np.allclose(dq1, 0, atol=1e-14) and np.allclose(dk1, 0, atol=1e-14) and
            np.allclose(dv1, dO.reshape(B, Hkv, 2, N, d).sum(2), atol=1e-12)):
        failed.append("window1_bwd")
    o2, _ = oracle.attention_fwd(q, k, v, True, scale, window=2)
    s_prev = scale * np.einsum("bhnd,bhnd->bhn", q[:, :, 1:], kx[:, :, :-1])
    s_self = scale * np.einsum("bhnd,bhnd->bhn", q[:, :, 1:], kx[:, :, 1:])
    w_prev = (1.0 / (1.0 + np.exp(s_self - s_prev)))[..., None]
    o2_ref = np.concatenate([vx[:, :, :1], w_prev * vx[:, :, :-1] + (1 - w_prev) * vx[:, :, 1:]], axis=2)
    if not np.allclose(o2, o2_ref, atol=1e-12):
        failed.append("window2_fwd")
    if not np.array_equal(oracle.attention_fwd(q, k, v, True, scale, window=N)[0],
                          oracle.attention_fwd(q, k, v, True, scale)[0]):
        failed.append("window_N_is_causal")

    from scipy.linalg import hadamard as sp_h
    for d in (8, 128):
        sg = rng.choice([-1.0, 1.0], size=d)
        if not np.allclose(oracle.hadamard(np.eye(d), sg), np.diag(sg) @ sp_h(d) / math.sqrt(d), atol=1e-14):
            failed.append(f"hadamard_{d}")

    x = np.clip(rng.standard_normal(4000) * 40, -448, 448).astype(np.float32).astype(np.float64)
    ref = torch.tensor(x, dtype=torch.float32).to(torch.float8_e4m3fn).double().numpy()
    if not np.array_equal(oracle.e4m3_round(x), ref):
        failed.append("e4m3_vs_torch")
    if not np.array_equal(oracle.e4m3_round(np.array([1000.0, 1.0625, 2 ** -10])), [448.0, 1.0, 0.0]):
        failed.append("e4m3_edges")
    return failed


def test_battery_passes_on_committed_oracle():
    assert _battery() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name, monkeypatch):
    old, new = MUTANTS[name]
    so = _build_mutant(tmp_path, name, old, new)
    real = oracle._load()
    lib = ctypes.CDLL(so)
    for fn in ("oracle_fwd", "oracle_fwd_rows", "oracle_bwd_group", "oracle_bwd",
               "oracle_hadamard", "oracle_e4m3_round"):
        getattr(lib, fn).argtypes = getattr(real, fn).argtypes
        getattr(lib, fn).restype = ctypes.c_int
    monkeypatch.setattr(oracle, "_lib", lib)
    failed = _battery()
    assert failed, f"planted mistake {name} passed every pin"
