"""Seeded synthetic inputs shared by the tests, the bench and the CPU oracle.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic.  Both the CUDA path and the oracle consume the very same
buffers produced here, so a parity comparison never depends on two generators
agreeing.

Recipe (the pages print no workload of their own, so the shapes are the five
configurations this library is measured on):

* every tensor is drawn i.i.d. N(0, 1) in fp32 from ``torch.Generator`` with a
  fixed seed, multiplied by ``scale`` (0.5 for the long-sequence case), then
  rounded to the storage dtype with torch's round-to-nearest-even cast;
* tensors are drawn in a fixed order (Q, K, V, then the upstream gradient G);
* decode-step inputs are drawn per step from a generator seeded with
  ``step_seed(seed, step)`` so that any single step can be regenerated alone.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _DTYPES[name]


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: the op it feeds, its shape, dtype, scale and seed."""

    name: str
    op: str  # "causal_fwd", "noncausal_fwd", "causal_fwd_bwd", "decode"
    B: int
    H: int
    N: int
    D: int
    M: int
    dtype: str
    scale: float
    seed: int
    prefill: int = 0  # decode only: tokens of causal prefill
    steps: int = 0  # decode only: number of decode steps

    def describe(self) -> str:
        if self.op == "decode":
            return (f"{self.name}: recurrent decode, {self.B} sequences x H{self.H}, "
                    f"D=M={self.D}, prefill {self.prefill} + {self.steps} steps, "
                    f"{self.dtype} q/k/v, fp32 S/Z")
        return (f"{self.name}: {self.op} B{self.B} H{self.H} N{self.N} D{self.D} M{self.M} "
                f"{self.dtype}, N(0,1)*{self.scale:g}")


# The five workloads: a tiny fp32 causal case, a non-causal fp32 case, the
# bf16 causal training case, a long bf16 causal case and autoregressive decode.
WORKLOADS = {
    "causal_tiny_f32": Workload("causal_tiny_f32", "causal_fwd", 1, 1, 256, 32, 32, "f32", 1.0, 1001),
    "noncausal_f32": Workload("noncausal_f32", "noncausal_fwd", 8, 8, 4096, 64, 64, "f32", 1.0, 1002),
    "causal_train_bf16": Workload("causal_train_bf16", "causal_fwd_bwd", 4, 16, 8192, 64, 64, "bf16", 1.0, 1003),
    "causal_long_bf16": Workload("causal_long_bf16", "causal_fwd", 1, 16, 65536, 128, 128, "bf16", 0.5, 1004),
    "decode_bf16": Workload("decode_bf16", "decode", 256, 16, 1, 64, 64, "bf16", 1.0, 1005,
                            prefill=2048, steps=2048),
}


def _gen(seed: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn(shape, dtype: str, seed: int, scale: float = 1.0, device: str = "cpu") -> torch.Tensor:
    """One N(0,1)*scale tensor drawn in fp32 and rounded to ``dtype``."""
    g = _gen(seed, device)
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch_dtype(dtype))


def qkv(B: int, H: int, N: int, D: int, M: int, dtype: str, seed: int, scale: float = 1.0,
        with_grad: bool = False, device: str = "cpu", qk_mean: float = 0.0) -> dict:
    """Q, K [B,H,N,D], V [B,H,N,M] and optionally G [B,H,N,M], drawn in that order.

    Every tensor is N(0,1)*scale; Q and K are then moved by qk_mean (e.g. -4
    puts nearly every entry of Q and K below zero)."""
    g = _gen(seed, device)
    out = {}
    shapes = [("Q", (B, H, N, D)), ("K", (B, H, N, D)), ("V", (B, H, N, M))]
    if with_grad:
        shapes.append(("G", (B, H, N, M)))
    for name, shp in shapes:
        x = torch.randn(shp, generator=g, dtype=torch.float32, device=device)
        if scale != 1.0:
            x.mul_(scale)
        if qk_mean != 0.0 and name in ("Q", "K"):
            x.add_(qk_mean)
        out[name] = x.to(torch_dtype(dtype))
    return out


def step_seed(seed: int, step: int) -> int:
    """Seed of decode step ``step`` (0-based) of a run seeded with ``seed``."""
    return int(seed) * 1_000_003 + 7919 * (int(step) + 1)


def decode_step_qkv(B: int, H: int, D: int, M: int, dtype: str, seed: int, step: int,
                    device: str = "cpu", scale: float = 1.0, qk_mean: float = 0.0) -> dict:
    """q, k [B,H,D] and v [B,H,M] of one decode step (N(0,1)*scale, q and k moved by qk_mean)."""
    g = _gen(step_seed(seed, step), device)
    out = {}
    for name, shp in (("q", (B, H, D)), ("k", (B, H, D)), ("v", (B, H, M))):
        x = torch.randn(shp, generator=g, dtype=torch.float32, device=device)
        if scale != 1.0:
            x.mul_(scale)
        if qk_mean != 0.0 and name in ("q", "k"):
            x.add_(qk_mean)
        out[name] = x.to(torch_dtype(dtype))
    return out


def decays(shape, seed: int, lo: float = 0.85, hi: float = 1.0, device: str = "cpu") -> torch.Tensor:
    """fp32 decays drawn uniformly in [lo, hi): one per head (RetNet's gamma) or
    one per token (gated retention's gamma_t)."""
    g = _gen(seed, device)
    return torch.rand(tuple(shape), generator=g, dtype=torch.float32, device=device).mul_(hi - lo).add_(lo)
