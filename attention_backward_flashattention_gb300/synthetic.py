"""Seeded synthetic inputs for attention forward/backward.

This module only draws random tensors and sequence lengths; it holds none of
the attention arithmetic.  The CUDA-path tests, the oracle tests and the
benchmark all take their inputs from here, so both sides of every parity check
see the same bits.

Recipe (fixed; every test and benchmark line uses it):
  * values are drawn in fp32 from ``torch.Generator`` (CPU) seeded with
    ``seed`` (default 0), in the order Q, K, V, dO -- or, for the packed
    layout, one (B, T, 3, H, d) QKV tensor and then dO;
  * dO is multiplied by ``do_scale`` (0.1 for the GPT-2-shaped layer);
  * every tensor is rounded to bf16 (round to nearest even).
Variable-length batches draw lengths log-uniformly in [lo, hi] with
``numpy.random.default_rng(seed)``: L = floor(exp(U(ln lo, ln hi))), drawn
while the running total is below ``total``; the last length is cut so the
lengths sum to ``total`` exactly.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

LAYOUT_BTHD = 0     # (B, T, H, d) per tensor
LAYOUT_PACKED = 1   # (B, T, 3, H, d) for Q, K, V together


@dataclass(frozen=True)
class Workload:
    """One attention problem shape (sizes only, no data)."""
    name: str
    B: int
    H: int
    T: int
    dqk: int
    dv: int
    causal: bool
    layout: int = LAYOUT_BTHD
    do_scale: float = 1.0
    varlen: tuple = field(default=())   # sequence lengths; empty = fixed T
    deterministic: bool = False

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dqk)

    @property
    def total_tokens(self) -> int:
        return sum(self.varlen) if self.varlen else self.B * self.T

    def bwd_flops(self) -> float:
        """2*B*H*Tq*Tk*(3*dqk+2*dv), halved for causal (per sequence for varlen)."""
        per = 2.0 * self.H * (3 * self.dqk + 2 * self.dv)
        lens = self.varlen if self.varlen else (self.T,) * self.B
        tot = sum(per * L * L for L in lens)
        return tot / 2 if self.causal else tot

    def fwd_flops(self) -> float:
        """2*B*H*Tq*Tk*(dqk+dv), halved for causal."""
        per = 2.0 * self.H * (self.dqk + self.dv)
        lens = self.varlen if self.varlen else (self.T,) * self.B
        tot = sum(per * L * L for L in lens)
        return tot / 2 if self.causal else tot


def varlen_lengths(total: int = 32768, lo: int = 512, hi: int = 16384,
                   seed: int = 0) -> tuple:
    """Log-uniform lengths in [lo, hi], cut so that they sum to ``total``."""
    rng = np.random.default_rng(seed)
    out, s = [], 0
    while s < total:
        L = int(math.floor(math.exp(rng.uniform(math.log(lo), math.log(hi)))))
        L = max(1, min(L, total - s))
        out.append(L)
        s += L
    return tuple(out)


def _sweep(causal):
    return [Workload(f"d128_T{T // 1024}K_{'causal' if causal else 'noncausal'}",
                     B=32768 // T, H=16, T=T, dqk=128, dv=128, causal=causal)
            for T in (1024, 2048, 4096, 8192, 16384, 32768)]


# The five workload families (sizes only).
TINY = [Workload("tiny_noncausal", 1, 2, 128, 64, 64, False),
        Workload("tiny_causal", 1, 2, 128, 64, 64, True)]
GPT2 = Workload("gpt2_small_packed", 8, 12, 1024, 64, 64, True,
                layout=LAYOUT_PACKED, do_scale=0.1)
SWEEP_D128 = _sweep(True) + _sweep(False)
D192 = [Workload(f"d192_128_T{T // 1024}K_causal", 32768 // T, 16, T, 192, 128, True)
        for T in (2048, 8192, 32768)]
VARLEN = Workload("varlen_det", B=len(varlen_lengths()), H=16, T=max(varlen_lengths()),
                  dqk=128, dv=128, causal=True, varlen=varlen_lengths(),
                  deterministic=True)
HEADLINE = [w for w in SWEEP_D128 if w.T == 32768 and w.causal][0]

ALL = {w.name: w for w in TINY + [GPT2] + SWEEP_D128 + D192 + [VARLEN]}


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """bf16 CPU tensors for workload ``w``.

    Returns a dict with q, k, v, dO (views into qkv for the packed layout),
    plus 'qkv' for packed and 'cu_seqlens' (int32, CPU) for varlen.
    Shapes: fixed-length (B,T,H,d); packed qkv (B,T,3,H,d); varlen (sum T,H,d).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = {}
    if w.varlen:
        lead = (w.total_tokens,)
        cu = np.concatenate([[0], np.cumsum(w.varlen)]).astype(np.int32)
        out["cu_seqlens"] = torch.from_numpy(cu)
    else:
        lead = (w.B, w.T)
    if w.layout == LAYOUT_PACKED:
        if w.dqk != w.dv:
            raise ValueError("packed layout needs dqk == dv")
        qkv = torch.randn(*lead, 3, w.H, w.dqk, generator=g, dtype=torch.float32)
        qkv = qkv.to(torch.bfloat16)
        out["qkv"] = qkv
        out["q"], out["k"], out["v"] = qkv.select(-3, 0), qkv.select(-3, 1), qkv.select(-3, 2)
    else:
        out["q"] = torch.randn(*lead, w.H, w.dqk, generator=g).to(torch.bfloat16)
        out["k"] = torch.randn(*lead, w.H, w.dqk, generator=g).to(torch.bfloat16)
        out["v"] = torch.randn(*lead, w.H, w.dv, generator=g).to(torch.bfloat16)
    dO = torch.randn(*lead, w.H, w.dv, generator=g, dtype=torch.float32)
    if w.do_scale != 1.0:
        dO = dO * w.do_scale
    out["dO"] = dO.to(torch.bfloat16)
    return out


def small_random(B, H, T, dqk, dv, seed=0, Tk=None):
    """Small fp32/bf16 inputs for unit checks: dict of bf16 (B,T,H,d) tensors."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    Tk = T if Tk is None else Tk
    q = torch.randn(B, T, H, dqk, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Tk, H, dqk, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Tk, H, dv, generator=g).to(torch.bfloat16)
    dO = torch.randn(B, T, H, dv, generator=g).to(torch.bfloat16)
    return {"q": q, "k": k, "v": v, "dO": dO}
