"""Seeded synthetic workloads for the attention backward pass.

This module only draws random numbers and builds shapes: it holds none of the
method's arithmetic, so both the CUDA path's tests and the CPU oracle can take
their inputs from it.

The five workloads follow the configurations the attention-backward pages are
measured on (shapes, dtypes, masks and value distributions); every tensor is
drawn from ``torch.Generator`` with a fixed seed, in the order Q, K, V, dO
(varlen lengths first).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int                      # batch (number of sequences when varlen)
    Sq: int                     # query length (max length when varlen)
    Sk: int
    Hq: int
    Hkv: int
    D: int
    dtype: str                  # "bf16" | "fp16"
    causal: bool
    deterministic: bool = False
    scale: Optional[float] = None      # None -> 1/sqrt(D)
    qk_dist: tuple = ("normal", 1.0)   # ("normal", std) | ("uniform", half_width)
    vdo_dist: tuple = ("normal", 1.0)
    varlen: Optional[tuple] = None     # (nseq, lo, hi): lengths uniform in [lo, hi]
    seed: int = 0
    Dv: Optional[int] = None           # value head dim (v, o, dout, dv); None -> D

    @property
    def value_dim(self) -> int:
        return self.D if self.Dv is None else self.Dv

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # 1x1x128x128x64, bf16, non-causal
    "b1_h1_s128_d64": Workload("b1_h1_s128_d64", 1, 128, 128, 1, 1, 64, "bf16", False),
    # 4x16x2048x2048x128, bf16, causal
    "b4_h16_s2048_d128_causal": Workload("b4_h16_s2048_d128_causal", 4, 2048, 2048, 16, 16, 128,
                                         "bf16", True),
    # 2x(32 q heads / 8 kv heads)x8192x8192x128, bf16, causal GQA
    "b2_hq32_hkv8_s8192_d128_causal_gqa": Workload("b2_hq32_hkv8_s8192_d128_causal_gqa", 2, 8192,
                                                   8192, 32, 8, 128, "bf16", True),
    # varlen: 16 sequences, lengths uniform in [256, 2048], H=16, D=64, fp16, causal
    "varlen16_h16_d64_fp16_causal": Workload("varlen16_h16_d64_fp16_causal", 16, 2048, 2048, 16,
                                             16, 64, "fp16", True, qk_dist=("normal", 0.5),
                                             vdo_dist=("normal", 0.5), varlen=(16, 256, 2048)),
    # 1x16x32768x32768x128, bf16, non-causal, deterministic dQ accumulation
    "b1_h16_s32768_d128_deterministic": Workload("b1_h16_s32768_d128_deterministic", 1, 32768,
                                                 32768, 16, 16, 128, "bf16", False,
                                                 deterministic=True, qk_dist=("normal", 1.0),
                                                 vdo_dist=("uniform", 1.0)),
}
WORKLOAD_ORDER = list(WORKLOADS)
BENCH_WORKLOAD = "b2_hq32_hkv8_s8192_d128_causal_gqa"


def _draw(shape, dist, gen, device):
    kind, p = dist
    if kind == "normal":
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * p
    if kind == "uniform":
        return (torch.rand(shape, generator=gen, device=device, dtype=torch.float32) * 2 - 1) * p
    raise ValueError(kind)


def varlen_lengths(w: Workload, gen: torch.Generator) -> list:
    nseq, lo, hi = w.varlen
    return torch.randint(lo, hi + 1, (nseq,), generator=gen).tolist()


def generate(w: Workload, device="cpu", seed: Optional[int] = None) -> dict:
    """Draws Q, K, V, dO (and varlen lengths) for workload ``w``.

    Returns a dict with q, k, v, dout (in ``w.dtype``), and for varlen
    ``cu_q`` / ``cu_k`` (int32 prefix sums, on ``device``), ``lengths`` and
    ``max_len``.  Dense tensors are [B, S, H, D]; varlen tensors are packed
    [total, H, D].
    """
    s = w.seed if seed is None else seed
    gen = torch.Generator(device=device)
    gen.manual_seed(s)
    out = {}
    if w.varlen is not None:
        cpu_gen = torch.Generator()
        cpu_gen.manual_seed(s)
        lengths = varlen_lengths(w, cpu_gen)
        cu = [0]
        for L in lengths:
            cu.append(cu[-1] + L)
        total = cu[-1]
        qshape, kshape = (total, w.Hq, w.D), (total, w.Hkv, w.D)
        oshape, vshape = (total, w.Hq, w.value_dim), (total, w.Hkv, w.value_dim)
        out["lengths"] = lengths
        out["max_len"] = max(lengths)
        out["cu_q"] = torch.tensor(cu, dtype=torch.int32, device=device)
        out["cu_k"] = out["cu_q"].clone()
    else:
        qshape, kshape = (w.B, w.Sq, w.Hq, w.D), (w.B, w.Sk, w.Hkv, w.D)
        oshape, vshape = (w.B, w.Sq, w.Hq, w.value_dim), (w.B, w.Sk, w.Hkv, w.value_dim)
    dt = w.torch_dtype
    out["q"] = _draw(qshape, w.qk_dist, gen, device).to(dt)
    out["k"] = _draw(kshape, w.qk_dist, gen, device).to(dt)
    out["v"] = _draw(vshape, w.vdo_dist, gen, device).to(dt)
    out["dout"] = _draw(oshape, w.vdo_dist, gen, device).to(dt)
    return out


def attention_pairs(w: Workload, lengths=None) -> float:
    """Number of (query, key) pairs the FLOP count is taken over: B*Hq*Sq*Sk,
    halved when causal (varlen: Hq * sum L_q*L_k, halved when causal)."""
    if w.varlen is not None:
        if lengths is None:
            raise ValueError("varlen needs lengths")
        pairs = float(sum(L * L for L in lengths)) * w.Hq
    else:
        pairs = float(w.B) * w.Hq * w.Sq * w.Sk
    return pairs / 2 if w.causal else pairs


def bwd_flops(w: Workload, lengths=None) -> float:
    """Algorithmic FLOPs of one backward pass: five GEMMs of 2 FLOPs per pair
    and head-dim column each -- S and dQ, dK over D, dP and dV over Dv:
    (6 D + 4 Dv) per pair, 10 D per pair when Dv = D."""
    return attention_pairs(w, lengths) * (6.0 * w.D + 4.0 * w.value_dim)
