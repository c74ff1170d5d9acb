"""CPU pins of the oracle's block-scaled e4m3 quantiser and of its model of an
FP8 backward (all five products of the backward step list on quantised
operands).

The e4m3 grid is enumerated here from its bit patterns (sign, 4 exponent
bits with bias 7, 3 mantissa bits; no infinities, 0x7F is NaN), independent
of the oracle's rounding routine, and the tiny-case pin recomputes the whole
model with plain per-row / per-column scales."""
import math

import numpy as np
import pytest

import oracle


def _grid():
    """All finite non-negative e4m3fn values by code (0 .. 0x7E)."""
    vals = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (8 + m) * 2.0 ** (e - 10))
    return np.array(vals)


GRID = _grid()


def _nearest(y):
    """Round |y| <= 448 to the nearest grid value, ties to the even code."""
    a = np.abs(y)
    hi = np.clip(np.searchsorted(GRID, a), 0, len(GRID) - 1)
    lo = np.clip(hi - 1, 0, len(GRID) - 1)
    dlo, dhi = a - GRID[lo], GRID[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    return np.sign(y) * GRID[pick]


def _pow2_scale(amax):
    """Smallest power of two 2^e with amax <= 448 * 2^e (1 for amax = 0)."""
    if amax == 0.0:
        return 1.0
    e = math.ceil(math.log2(amax / 448.0))
    while amax > 448.0 * 2.0 ** e:
        e += 1
    while amax <= 448.0 * 2.0 ** (e - 1):
        e -= 1
    return 2.0 ** e


def test_grid_enumeration():
    assert GRID[0] == 0.0 and GRID[1] == 2.0 ** -9 and GRID[8] == 2.0 ** -6 and GRID[-1] == 448.0
    assert np.all(np.diff(GRID) > 0) and len(GRID) == 127


@pytest.mark.parametrize("axis", [0, 1])
def test_mx_e4m3_matches_brute_force(axis):
    rng = np.random.default_rng(11)
    # 70 entries along the blocked axis (two full blocks and a ragged one of 6),
    # magnitudes spread over many binades, one all-zero block
    x = rng.standard_normal((70, 9)) * np.exp2(rng.integers(-30, 30, size=(70, 9)))
    x[32:64, 3] = 0.0
    # a block whose largest entry is exactly 448 * 2^-3: scale 2^-3, not 2^-2
    x[64:70, 7] = [-56.0, 55.0, 3.0, -1.0, 0.25, 40.0]
    if axis == 1:
        x = x.T.copy()
    deq, exps = oracle.mx_e4m3(x, axis)
    xm = np.moveaxis(x, axis, 0)
    dm = np.moveaxis(deq, axis, 0)
    em = np.moveaxis(exps, axis, 0)
    assert em.shape == (3, 9)
    for j, (a, b) in enumerate([(0, 32), (32, 64), (64, 70)]):
        for c in range(9):
            blk = xm[a:b, c]
            s = _pow2_scale(float(np.abs(blk).max()))
            assert 2.0 ** em[j, c] == s
            assert np.abs(blk / s).max() <= 448.0          # never saturates
            if blk.any():
                assert np.abs(blk / s).max() > 224.0       # and no smaller scale would do
            np.testing.assert_array_equal(dm[a:b, c], _nearest(blk / s) * s)


def test_mx_e4m3_axis_transpose_and_power_of_two_equivariance():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((40, 33)) * 3.0
    d0, e0 = oracle.mx_e4m3(x, 0)
    d1, e1 = oracle.mx_e4m3(x.T, 1)
    np.testing.assert_array_equal(d0, d1.T)
    np.testing.assert_array_equal(e0, e1.T)
    d5, e5 = oracle.mx_e4m3(x * 2.0 ** 5, 0)
    np.testing.assert_array_equal(d5, d0 * 2.0 ** 5)
    np.testing.assert_array_equal(e5, e0 + 5)
    # blocks are independent: changing one block leaves the others alone
    y = x.copy()
    y[0:32] *= 1e6
    dy, _ = oracle.mx_e4m3(y, 0)
    np.testing.assert_array_equal(dy[32:], d0[32:])


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_bwd_model_without_quantisation_is_exact(causal):
    """Mode None (and mode mx32 with no product quantised) is the exact
    backward, with the Hadamard rotation and its inverse and a GQA group."""
    rng = np.random.default_rng(13)
    B, Hq, Hkv, N, d = 1, 4, 2, 40, 16
    q, dO = rng.standard_normal((B, Hq, N, d)), rng.standard_normal((B, Hq, N, d))
    k, v = rng.standard_normal((B, Hkv, N, d)), rng.standard_normal((B, Hkv, N, d))
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    ref = oracle.attention_bwd(q, k, v, dO, causal, 0.3)
    for args in [(None, signs), (None, None), ("mx32", signs, ())]:
        got = oracle.fp8_bwd_model(q, k, v, dO, causal, 0.3, *args)
        for g, r in zip(got, ref):
            np.testing.assert_allclose(g, r, rtol=1e-11, atol=1e-12)


ALL = ("S", "dP", "dV", "dK", "dQ")


# The later products re-round what the earlier ones changed, so S and dP are
# also checked on their own.
@pytest.mark.parametrize("prods", [ALL, ("S",), ("dP",), ("dV", "dK", "dQ")])
def test_fp8_bwd_model_tiny_case_recomputed_by_hand(prods):
    """N = d = 32: one block along every axis, so the mx32 scales are plain
    per-row scales for the products that reduce over d (S, dP) and per-column
    scales for those that reduce over queries (dV, dK) or keys (dQ)."""
    rng = np.random.default_rng(14)
    N = d = 32

    def structured(s):
        # Scaling by a power of two moves no entry between grid points unless
        # it leaves e4m3's normal range, so per-row and per-column scales give
        # different values only for entries far (> 2^14) below their block's
        # largest: rows and columns span 2^20 here.
        a = rng.integers(-10, 1, size=(N, 1))
        c = rng.integers(-10, 1, size=(1, d))
        return rng.standard_normal((N, d)) * s * np.exp2(a + c)

    q, k, v, dO = (structured(s) for s in (2.0, 2.0, 1.0, 1.0))
    for x in (q, k, v, dO):
        assert not np.array_equal(oracle.mx_e4m3(x, 0)[0], oracle.mx_e4m3(x, 1)[0])
    scale = 0.2

    def rows(x, prod):  # one scale per row
        if prod not in prods:
            return x
        return np.stack([_nearest(r / _pow2_scale(np.abs(r).max())) * _pow2_scale(np.abs(r).max()) for r in x])

    def cols(x, prod):  # one scale per column
        return rows(x.T, prod).T

    S = scale * rows(q, "S") @ rows(k, "S").T
    S = np.where(np.tril(np.ones((N, N), dtype=bool)), S, -np.inf)
    P = np.exp(S - np.log(np.exp(S - S.max(1, keepdims=True)).sum(1, keepdims=True)) - S.max(1, keepdims=True))
    assert np.median(P.max(axis=1)) < 0.5
    D = (dO * (P @ v)).sum(1, keepdims=True)
    dS = P * (rows(dO, "dP") @ rows(v, "dP").T - D)
    dv = cols(P, "dV").T @ cols(dO, "dV")
    dk = scale * cols(dS, "dK").T @ cols(q, "dK")
    dq = scale * rows(dS, "dQ") @ cols(k, "dQ")
    got = oracle.fp8_bwd_model(q[None, None], k[None, None], v[None, None], dO[None, None], True, scale,
                               "mx32", None, prods)
    for g, r in zip(got, (dq, dk, dv)):
        # rounding order only: far below what any one product's quantisation moves
        assert np.abs(g[0, 0] - r).max() <= 1e-12 * np.abs(r).max()


def test_fp8_bwd_model_products_are_attributed():
    """Quantising one product changes only the gradients that depend on it."""
    rng = np.random.default_rng(15)
    q, k, v, dO = (rng.standard_normal((1, 1, 64, 32)) for _ in range(4))
    exact = oracle.fp8_bwd_model(q, k, v, dO, True, 0.2, None)
    depends = {"S": (1, 1, 1), "dP": (1, 1, 0), "dV": (0, 0, 1), "dK": (0, 1, 0), "dQ": (1, 0, 0)}
    for prod, dep in depends.items():
        got = oracle.fp8_bwd_model(q, k, v, dO, True, 0.2, "mx32", None, (prod,))
        for g, e, changed in zip(got, exact, dep):
            assert (not np.array_equal(g, e)) == bool(changed), prod


def test_fp8_bwd_error_floor_of_e4m3_products():
    """Each product on block-scaled e4m3 operands alone puts a 2-6 % relative
    error on the gradients it feeds (causal, N(0,1) inputs): e4m3's 3-bit
    mantissa, not the choice of scales, sets this floor, so no FP8 product
    of the backward meets a 1e-2 gradient bound."""
    rng = np.random.default_rng(16)
    q, k, v, dO = (rng.standard_normal((1, 2, 256, 64)) for _ in range(4))
    exact = oracle.attention_bwd(q, k, v, dO, True, 0.125)
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)  # noqa: E731
    for prod, idx in [("S", 0), ("dP", 0), ("dV", 2), ("dK", 1), ("dQ", 0)]:
        for mode in ("mx32", "tensor"):
            g = oracle.fp8_bwd_model(q, k, v, dO, True, 0.125, mode, None, (prod,))
            assert 0.02 < rel(g[idx], exact[idx]) < 0.06, (prod, mode)


# ----------------------------------------------------------- planted mistakes

MUTANTS = {
    "dv_blocks_along_keys": ('qz(P, 0, "dV").T @ qz(dOh, 0, "dV")', 'qz(P, 1, "dV").T @ qz(dOh, 1, "dV")'),
    "dq_k_blocks_along_d": ('qz(K, 0, "dQ")', 'qz(K, 1, "dQ")'),
    "dk_ds_blocks_along_keys": ('qz(dS, 0, "dK")', 'qz(dS, 1, "dK")'),
    "s_q_blocks_along_queries": ('qz(Q, 1, "S")', 'qz(Q, 0, "S")'),
    "dp_v_under_wrong_product": ('qz(V, 1, "dP")', 'qz(V, 1, "dV")'),
    "scale_one_too_large_at_powers_of_two":
        ("ev = np.where(amax[nz] <= np.ldexp(448.0, ev - 1), ev - 1, ev)", "pass"),
    "scale_always_one_too_large": ("e[nz] = np.clip(ev, -127, 127)", "e[nz] = np.clip(ev + 1, -127, 127)"),
    "rotation_not_undone": ("dq, dk = hadamard(dq) * s, hadamard(dk) * s", "dq, dk = hadamard(dq, s), hadamard(dk, s)"),
    "d_without_output": ("D = (dOh * (P @ V)).sum(axis=1, keepdims=True)", "D = (dOh * V).sum(axis=1, keepdims=True)"),
    "blocks_of_16": ("def mx_e4m3(x, axis: int, block: int = 32):", "def mx_e4m3(x, axis: int, block: int = 16):"),
}

_PINS = None


def _pins():
    global _PINS
    if _PINS is None:
        g = globals()
        _PINS = [
            lambda: g["test_mx_e4m3_matches_brute_force"](0),
            lambda: g["test_mx_e4m3_matches_brute_force"](1),
            g["test_mx_e4m3_axis_transpose_and_power_of_two_equivariance"],
            lambda: g["test_fp8_bwd_model_without_quantisation_is_exact"](True),
            *[(lambda p=p: g["test_fp8_bwd_model_tiny_case_recomputed_by_hand"](p))
              for p in (ALL, ("S",), ("dP",), ("dV", "dK", "dQ"))],
            g["test_fp8_bwd_model_products_are_attributed"],
        ]
    return _PINS


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    """Each mutant of the model's source, loaded as its own module and swapped
    in for the oracle's functions, fails at least one of the pins above."""
    import inspect
    import types

    old, new = MUTANTS[name]
    src = inspect.getsource(oracle)
    assert src.count(old) == 1, f"mutation anchor missing for {name}"
    mod = types.ModuleType(f"oracle_mutant_{name}")
    mod.__dict__["__file__"] = oracle.__file__
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    monkeypatch.setattr(oracle, "mx_e4m3", mod.mx_e4m3)
    monkeypatch.setattr(oracle, "fp8_bwd_model", mod.fp8_bwd_model)
    caught = 0
    for pin in _pins():
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin fails for {name}"


# ------------------------------------------- per-tensor model of the forward

def test_fp8_dequantized_matches_brute_force_per_tensor_scale():
    """The FP8 forward's input model: Q and K rotated (here by an explicit
    signed Sylvester matrix built in the test), then every tensor scaled by
    sigma = amax / 448, rounded to the nearest e4m3 value (brute force over the
    grid) and scaled back; V is not rotated.  The rounding decision is taken
    in fp32, as a product by the fp32 reciprocal 448 / amax after the 1/sqrt(d)
    factor (numpy float32 arithmetic here)."""
    f32 = np.float32
    rng = np.random.default_rng(17)
    d = 32  # 1/sqrt(d) = 2^-2.5 is not a power of two, like the kernels' 2^-3.5 at d = 128
    q, k, v = (rng.standard_normal((1, 2, 24, d)) * s for s in (3.0, 0.2, 50.0))
    # a power-of-two change of sigma moves only values in e4m3's subnormal
    # range (|x / sigma| < 2^-6), so V gets a few of those
    v[0, 0, 0, :4] = np.abs(v).max() * np.array([1e-5, 2.5e-5, -3e-6, 1.7e-5])
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    Hs = np.array([[(-1.0) ** bin(i & j).count("1") for j in range(d)] for i in range(d)])
    qm, km, vm = oracle.fp8_dequantized(q, k, v, signs)
    for got, xp, c in ((qm, (q * signs) @ Hs, f32(1.0 / np.sqrt(d))), (km, (k * signs) @ Hs, f32(1.0 / np.sqrt(d))),
                       (vm, v, f32(1.0))):
        x32 = xp.astype(f32)
        amax = f32(np.abs(x32).max() * c)
        t = (x32 * c) * (f32(448.0) / amax)
        assert np.abs(t).max() == pytest.approx(448.0, rel=1e-6)
        want = _nearest(t.astype(np.float64)) * float(amax / f32(448.0))
        np.testing.assert_array_equal(got, want)


def test_fp8_dequantized_splits_exact_ties_to_even():
    """16-bit values whose x * 448 / amax lies exactly on an e4m3 midpoint go
    to the even code.  With amax = 122 (so sigma = 122 / 448 is not exact in
    any binary format): 45.75 maps to exactly 168, halfway between 160 and
    176, and 22.875 to exactly 84, halfway between 80 and 88; both go down to
    the even codes 160 and 80.  47.6640625 maps to about 175.03 and goes to
    the nearest value, 176; 30.5 maps to 112, on the grid."""
    x = np.zeros((1, 1, 2, 8))
    x[0, 0, 0, :5] = [122.0, 45.75, -45.75, 30.5, 22.875]
    x[0, 0, 1, :2] = [47.6640625, 1.0]
    xm, _, _ = oracle.fp8_dequantized(x, x, x, None)
    sigma = float(np.float32(122.0) / np.float32(448.0))
    codes = np.round(xm / sigma, 6)
    np.testing.assert_array_equal(codes[0, 0, 0, :5], [448.0, 160.0, -160.0, 112.0, 80.0])
    assert codes[0, 0, 1, 0] == 176.0


# ------------------------------- planted mistakes in the forward's input model

DQ_MUTANTS = {
    "code_from_fp64_quotient": ("t = (part(i) * c) * inv  # two fp32 products",
                                "t = part(i).astype(np.float64) * float(c) / (float(amax) / 448.0)  # "),
    "value_without_inv_sqrt_d": ("t = (part(i) * c) * inv  # two fp32 products", "t = part(i) * inv  # "),
    "amax_without_inv_sqrt_d": ("amax = f32(max(f32(np.abs(part(i)).max()) for i in range(x.shape[0])) * c)",
                                "amax = f32(max(f32(np.abs(part(i)).max()) for i in range(x.shape[0])))"),
    "sigma_off_grid_maximum": ("sigma = float(amax / f32(448.0))", "sigma = float(amax / f32(480.0))"),
    "v_rotated": ("return qdq(q, rot), qdq(k, rot), qdq(v, False)", "return qdq(q, rot), qdq(k, rot), qdq(v, rot)"),
}


@pytest.mark.parametrize("name", sorted(DQ_MUTANTS))
def test_dequantized_pins_catch_planted_mistake(name, monkeypatch):
    """Each mutant of the FP8 forward's input model (the fp32 code decision,
    the 1/sqrt(d) factor, the scale, which tensors are rotated) fails the
    brute-force pin or the exact-tie pin."""
    import inspect
    import types

    old, new = DQ_MUTANTS[name]
    src = inspect.getsource(oracle)
    assert src.count(old) == 1, f"mutation anchor missing for {name}"
    mod = types.ModuleType(f"oracle_mutant_{name}")
    mod.__dict__["__file__"] = oracle.__file__
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    monkeypatch.setattr(oracle, "fp8_dequantized", mod.fp8_dequantized)
    caught = 0
    for pin in (test_fp8_dequantized_matches_brute_force_per_tensor_scale, test_fp8_dequantized_splits_exact_ties_to_even):
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin fails for {name}"
