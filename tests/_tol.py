"""Parity tolerances (the numbers are stated in the tests that use them).

Forward O: |O_gpu - O_ref| <= 4e-3 + half an ulp of the output element type
at |O_ref|, element-wise.  The 4e-3 bound is the stated O tolerance; the
half-ulp term is the rounding of the stored output itself, which alone can
exceed 4e-3 for bf16 values of magnitude >= 1 (ulp 2^-7 on [1, 2)).
LSE: max-abs <= 1e-3.  Gradients: relative Frobenius error <= 1e-2 per tensor.
FP8 O: RMS error relative to the RMS of V <= 0.03, and no worse than the
same kernel without the Hadamard rotation.
"""
import numpy as np
import torch

O_ABS = 4e-3
LSE_ABS = 1e-3
GRAD_REL = 1e-2
FP8_REL_RMS = 0.03

_MANT = {torch.bfloat16: 7, torch.float16: 10}


def half_ulp(ref: np.ndarray, dtype) -> np.ndarray:
    a = np.maximum(np.abs(ref), 2.0 ** -14)
    e = np.floor(np.log2(a))
    return 0.5 * np.exp2(e - _MANT[dtype])


def check_o(got: torch.Tensor, ref: np.ndarray, what: str = "O"):
    g = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    bound = O_ABS + half_ulp(ref, got.dtype)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements over tolerance; max err {err.max():.3e}, "
                           f"worst excess {(err - bound).max():.3e}")
    return float(err.max())


def check_lse(got: torch.Tensor, ref: np.ndarray, what: str = "LSE"):
    err = float(np.abs(got.float().cpu().numpy().astype(np.float64) - ref).max())
    assert err <= LSE_ABS, f"{what}: max-abs {err:.3e} > {LSE_ABS}"
    return err


def rel_fro(got, ref: np.ndarray) -> float:
    g = got.float().cpu().numpy().astype(np.float64) if hasattr(got, "cpu") else got
    return float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-300))


def check_grad(got, ref: np.ndarray, what: str):
    if np.linalg.norm(ref) == 0.0:
        # degenerate case (e.g. a single key: softmax is constant, dQ = dK = 0
        # exactly); a relative error is undefined, so bound the absolute value
        a = float(np.abs(got.float().cpu().numpy()).max())
        assert a <= 1e-3, f"{what}: exact gradient is zero but max |got| = {a:.3e}"
        return 0.0
    r = rel_fro(got, ref)
    assert r <= GRAD_REL, f"{what}: relative Frobenius error {r:.3e} > {GRAD_REL}"
    return r
