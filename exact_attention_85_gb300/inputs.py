"""Seeded synthetic inputs shared by the CUDA path, the oracle and the bench.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic, so both sides of a parity test can take their inputs
from here without sharing any of the method.

Recipe (the same for every workload): a CPU ``torch.Generator`` seeded with
``seed`` draws, in this order, fp32 N(0, 1) tensors for Q, K, V and dO, which
are then cast to the workload's element type.  The identical bits go to the
GPU and (widened to fp64) to the oracle.  For the FP8 workload the same
generator then draws the outlier positions of Q and of K (exactly
round(0.001 * numel) entries each, without replacement, multiplied by 50)
and a random sign vector s in {-1, +1}^d; this mirrors the synthetic outlier
experiment of the FlashAttention-3 summary page (FP8 and incoherent
processing section: N(0,1) inputs with 0.1% large-magnitude entries).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    dtype: str          # "fp16" | "bf16" | "e4m3"
    causal: bool
    backward: bool = True
    outliers: bool = False
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)

    @property
    def torch_dtype(self) -> torch.dtype:
        # the e4m3 workload is drawn in bf16 and quantised by the FP8 path
        return {"fp16": torch.float16, "bf16": torch.bfloat16,
                "e4m3": torch.bfloat16}[self.dtype]

    def fwd_flops(self) -> float:
        """4 B Hq N^2 d, halved when causal (two GEMMs; mask work not counted)."""
        f = 4.0 * self.B * self.Hq * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        """2.5x the forward count (five GEMMs against two)."""
        return 2.5 * self.fwd_flops()


# The five workloads of the method's evaluation plus the headline shape.
WORKLOADS = {
    "tiny_fp16_d64_n256": Workload("tiny_fp16_d64_n256", 1, 2, 2, 256, 64, "fp16", False, seed=1000),
    "train_bf16_b8_h16_n2k_causal": Workload("train_bf16_b8_h16_n2k_causal", 8, 16, 16, 2048, 128, "bf16", True, seed=1001),
    "long_bf16_b1_h16_n16k_causal": Workload("long_bf16_b1_h16_n16k_causal", 1, 16, 16, 16384, 128, "bf16", True, seed=1002),
    "gqa_bf16_b4_hq32_hkv8_n4k_causal": Workload("gqa_bf16_b4_hq32_hkv8_n4k_causal", 4, 32, 8, 4096, 128, "bf16", True, seed=1003),
    "fp8_b4_h16_n8k_outliers": Workload("fp8_b4_h16_n8k_outliers", 4, 16, 16, 8192, 128, "e4m3", False, backward=False, outliers=True, seed=1004),
    "bf16_b4_h16_n8k_d128_causal": Workload("bf16_b4_h16_n8k_d128_causal", 4, 16, 16, 8192, 128, "bf16", True, seed=1005),
}

HEADLINE = "bf16_b4_h16_n8k_d128_causal"


def make_inputs(w: Workload, seed: int | None = None, with_grad: bool = True):
    """Draw Q, K, V (and dO) on the CPU for workload ``w``.

    Returns a dict of CPU tensors: q [B,Hq,N,d], k/v [B,Hkv,N,d], dO like q,
    and for the outlier workload also ``signs`` (fp32, +-1, length d).
    """
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    dt = w.torch_dtype
    out = {}
    out["q"] = torch.randn(w.B, w.Hq, w.N, w.d, generator=g).to(dt)
    out["k"] = torch.randn(w.B, w.Hkv, w.N, w.d, generator=g).to(dt)
    out["v"] = torch.randn(w.B, w.Hkv, w.N, w.d, generator=g).to(dt)
    if with_grad:
        out["dO"] = torch.randn(w.B, w.Hq, w.N, w.d, generator=g).to(dt)
    if w.outliers:
        for name in ("q", "k"):
            t = out[name].float().reshape(-1)
            n_out = int(round(0.001 * t.numel()))
            idx = torch.randperm(t.numel(), generator=g)[:n_out]
            t[idx] *= 50.0
            out[name] = t.reshape(out[name].shape).to(dt)
        out["signs"] = random_signs(w.d, g)
    return out


def random_signs(d: int, g: torch.Generator) -> torch.Tensor:
    """A vector of d independent fair +-1 draws (fp32)."""
    bits = torch.randint(0, 2, (d,), generator=g)
    return (bits * 2 - 1).to(torch.float32)


def make_custom(B, Hq, Hkv, N, d, dtype=torch.bfloat16, seed=0, with_grad=True):
    """Same recipe for an arbitrary shape (edge-case tests)."""
    g = torch.Generator().manual_seed(seed)
    out = {
        "q": torch.randn(B, Hq, N, d, generator=g).to(dtype),
        "k": torch.randn(B, Hkv, N, d, generator=g).to(dtype),
        "v": torch.randn(B, Hkv, N, d, generator=g).to(dtype),
    }
    if with_grad:
        out["dO"] = torch.randn(B, Hq, N, d, generator=g).to(dtype)
    return out


def varlen_lengths(B: int, max_len: int, seed: int = 0) -> list[int]:
    """A seeded length mix for a packed batch: B lengths drawn uniformly
    from 1 .. max_len (the pages name variable-length batches but give no
    length distribution; tests add the edge lengths explicitly)."""
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(1, max_len + 1, (B,), generator=g)]


def make_varlen(lengths, Hq: int, Hkv: int, d: int, dtype=torch.bfloat16, seed: int = 0,
                with_grad: bool = True) -> dict:
    """Packed token-major tensors for sequences of the given lengths:
    q [total, Hq, d], k, v [total, Hkv, d], dO [total, Hq, d] drawn N(0, 1)
    in that order (then cast), and cu_seqlens int32 [B + 1] (prefix sums)."""
    g = torch.Generator().manual_seed(seed)
    total = int(sum(lengths))
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    out = {
        "q": torch.randn(total, Hq, d, generator=g).to(dtype),
        "k": torch.randn(total, Hkv, d, generator=g).to(dtype),
        "v": torch.randn(total, Hkv, d, generator=g).to(dtype),
        "cu_seqlens": torch.tensor(cu, dtype=torch.int32),
    }
    if with_grad:
        out["dO"] = torch.randn(total, Hq, d, generator=g).to(dtype)
    return out
