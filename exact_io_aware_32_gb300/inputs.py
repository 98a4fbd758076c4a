"""Seeded synthetic inputs for the attention workloads.

This module holds no attention arithmetic: it only draws random tensors. Both
the CUDA path's tests and the CPU oracle consume what it produces.

Every workload draws q, k, v and dO, in that order, as float32 i.i.d. N(0, 1)
from a CPU ``torch.Generator`` seeded with the workload's seed, then rounds them
to bf16 (round to nearest even). The long-sequence workload multiplies q and k
by 2.0 before rounding (exact: a power of two), which sharpens the softmax.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: tuple
    seed: int
    qk_mult: float = 1.0
    note: str = ""
    scale: float = field(default=0.0)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale else 1.0 / math.sqrt(self.d)

    @property
    def BH(self) -> int:
        return self.B * self.H


# The five workload shapes. Seeds: the first workload states seed 0; the
# others take their position in this list.
WORKLOADS = {
    "single_head_n256_d64": Workload("single_head_n256_d64", 1, 1, 256, 64, (False, True), 0,
                                     note="float32 N(0,1) inputs rounded to bf16"),
    "gpt2_small_n1024_d64": Workload("gpt2_small_n1024_d64", 8, 12, 1024, 64, (True,), 1, scale=0.125),
    "gpt2_medium_n1024_d64": Workload("gpt2_medium_n1024_d64", 64, 16, 1024, 64, (True,), 2, scale=0.125),
    "d128_n4096": Workload("d128_n4096", 4, 32, 4096, 128, (True, False), 3),
    "long_n16384_d128": Workload("long_n16384_d128", 1, 16, 16384, 128, (True,), 4, qk_mult=2.0),
}


def make_inputs(B: int, H: int, N: int, d: int, seed: int, qk_mult: float = 1.0, device: str = "cpu"):
    """Return dict(q, k, v, dO) of bf16 tensors [B, H, N, d], drawn on the CPU."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    dO = torch.randn(shape, generator=g, dtype=torch.float32)
    if qk_mult != 1.0:
        q.mul_(qk_mult)
        k.mul_(qk_mult)
    out = {}
    for name, t in (("q", q), ("k", k), ("v", v), ("dO", dO)):
        out[name] = t.to(torch.bfloat16).to(device)
    return out


def make_fp8_inputs(B: int, H: int, N: int, d: int, seed: int, qk_mult: float = 1.0, device: str = "cpu"):
    """E4M3 versions of q, k, v for the 8-bit forward: the same float32 draws as
    make_inputs, each tensor divided by its own factor amax / 448 (so that its
    largest magnitude lands on the largest E4M3 value) and rounded to E4M3 by
    torch's float8_e4m3fn conversion. Returns dict(q, k, v) of uint8 code
    tensors [B, H, N, d] and dict(q, k, v) of the dequantisation factors."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (B, H, N, d)
    x = {name: torch.randn(shape, generator=g, dtype=torch.float32) for name in ("q", "k", "v")}
    if qk_mult != 1.0:
        x["q"].mul_(qk_mult)
        x["k"].mul_(qk_mult)
    codes, desc = {}, {}
    for name, t in x.items():
        desc[name] = float(t.abs().max()) / 448.0
        codes[name] = (t / desc[name]).to(torch.float8_e4m3fn).view(torch.uint8).to(device)
    return codes, desc


def workload_inputs(w: Workload, device: str = "cpu"):
    return make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult, device=device)
