"""Seeded synthetic inputs for MoE token dispatch / combine.

This module only *generates inputs*: router output (``topk_idx``, ``topk_w``),
token activations ``x`` and expert outputs ``y``.  It holds none of the
arithmetic of dispatch or combine, so both the CPU oracle's tests and the CUDA
path's tests and benchmark draw their inputs from here.

The routing recipes follow the MoE shapes the pages' serving runs use
(Qwen3-30B-A3B and DeepSeek-V3, SGLang PR "Add DeepEPv2 (ElasticBuffer) MoE A2A
backend", section "Supported scope"); the models themselves, their weights and
their datasets are not available, so seeded synthetic routing stands in for them:

* ``softmax``: logits ~ N(0,1) fp32, p = softmax(logits), top-K by p (ties to the
  lower expert id), weights = p_sel / sum(p_sel).
* ``grouped_sigmoid`` (DeepSeek-V3 style): s = sigmoid(logits), a fixed bias
  b ~ N(0, 0.1) per expert, c = s + b; experts split into ``n_group`` groups,
  group score = sum of the two largest c in the group, the ``topk_group`` best
  groups are kept, top-K of c among them, weights = s_sel / sum(s_sel).
* ``zipf``: expert popularity p_e ~ (e+1)^-s, K distinct experts per token drawn
  without replacement (Gumbel-top-K on log p, kept in sampled order),
  weights ~ Dirichlet(1).

All draws come from ``numpy.random.default_rng(seed)``; bf16 tensors are fp32
draws rounded to nearest-even by torch's CPU cast.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = [
    "Workload",
    "CONFIGS",
    "route",
    "make_x",
    "make_expert_outputs",
    "make_inputs",
    "bf16_bits_from_f32",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic MoE dispatch/combine problem."""

    name: str
    T: int  # tokens
    H: int  # hidden size
    E: int  # experts
    K: int  # top-k
    routing: str  # "softmax" | "grouped_sigmoid" | "zipf"
    layout: str  # "contig" | "masked"
    quant: str  # "none" | "fp8_f32" | "fp8_ue8m0"
    align: int = 128  # row alignment of expert segments (contiguous layout)
    cap: int = 0  # masked slab capacity per expert
    R: int = 1  # logical expert-parallel ranks (partitions of the expert set)
    n_group: int = 8
    topk_group: int = 4
    bias_std: float = 0.1
    zipf_s: float = 1.2
    identity_experts: bool = False  # combine input y = the dispatched rows
    seed: int = 0

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads, by what they are.
CONFIGS = {
    "tiny": Workload("tiny", T=64, H=256, E=8, K=2, routing="softmax",
                     layout="contig", quant="none", align=128,
                     identity_experts=True),
    "qwen3_30b_a3b_decode": Workload(
        "qwen3_30b_a3b_decode", T=256, H=2048, E=128, K=8, routing="softmax",
        layout="masked", quant="fp8_f32", cap=256),
    "dsv3_decode": Workload(
        "dsv3_decode", T=1024, H=7168, E=256, K=8, routing="grouped_sigmoid",
        layout="masked", quant="fp8_ue8m0", cap=1024),
    "dsv3_prefill": Workload(
        "dsv3_prefill", T=16384, H=7168, E=256, K=8, routing="grouped_sigmoid",
        layout="contig", quant="fp8_f32", align=128),
    "skewed_zipf": Workload(
        "skewed_zipf", T=8192, H=4096, E=128, K=8, routing="zipf",
        layout="contig", quant="none", align=128, R=8),
}


def _topk_desc(score: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries per row, descending; ties -> lower index."""
    order = np.argsort(-score, axis=1, kind="stable")
    return order[:, :k]


def route(w: Workload, rng: Optional[np.random.Generator] = None):
    """Router output for workload ``w``: (topk_idx int32 [T,K], topk_w fp32 [T,K])."""
    rng = rng if rng is not None else np.random.default_rng(w.seed)
    T, E, K = w.T, w.E, w.K
    if w.routing == "softmax":
        logits = rng.standard_normal((T, E), dtype=np.float32)
        z = logits - logits.max(axis=1, keepdims=True)
        p = np.exp(z)
        p /= p.sum(axis=1, keepdims=True)
        idx = _topk_desc(p, K)
        sel = np.take_along_axis(p, idx, axis=1)
        wts = sel / sel.sum(axis=1, keepdims=True)
    elif w.routing == "grouped_sigmoid":
        logits = rng.standard_normal((T, E), dtype=np.float32)
        bias = rng.normal(0.0, w.bias_std, size=E).astype(np.float32)
        s = 1.0 / (1.0 + np.exp(-logits))
        c = s + bias[None, :]
        G = w.n_group
        assert E % G == 0
        cg = c.reshape(T, G, E // G)
        top2 = -np.sort(-cg, axis=2)[:, :, :2].sum(axis=2)  # [T, G]
        keep = _topk_desc(top2, w.topk_group)  # [T, topk_group]
        mask = np.zeros((T, G), dtype=bool)
        np.put_along_axis(mask, keep, True, axis=1)
        cm = np.where(np.repeat(mask, E // G, axis=1), c, -np.inf)
        idx = _topk_desc(cm, K)
        sel = np.take_along_axis(s, idx, axis=1)
        wts = sel / sel.sum(axis=1, keepdims=True)
    elif w.routing == "zipf":
        pe = (np.arange(E, dtype=np.float64) + 1.0) ** (-w.zipf_s)
        pe /= pe.sum()
        keys = np.log(pe)[None, :] + rng.gumbel(size=(T, E))
        idx = _topk_desc(keys, K)  # sampled order = descending perturbed key
        wts = rng.dirichlet(np.ones(K), size=T)
    else:
        raise ValueError(f"unknown routing {w.routing!r}")
    return (np.ascontiguousarray(idx, dtype=np.int32),
            np.ascontiguousarray(wts, dtype=np.float32))


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), rounded to nearest-even by torch."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def make_x(w: Workload, rng: Optional[np.random.Generator] = None) -> np.ndarray:
    """Token activations x: bf16 bits [T, H], N(0,1) draws."""
    rng = rng if rng is not None else np.random.default_rng(w.seed + 1000)
    return bf16_bits_from_f32(rng.standard_normal((w.T, w.H), dtype=np.float32))


def make_expert_outputs(rows: int, H: int, seed: int, device="cpu", chunk_rows: int = 8192):
    """Synthetic expert outputs y: a torch bf16 tensor [rows, H] of N(0,1) draws.

    Generated with a seeded torch generator on ``device`` (large slabs are made on
    the GPU directly).  The values depend on the device's generator; whatever is
    generated is what both sides of a comparison are given.
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty((rows, H), dtype=torch.bfloat16, device=device)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = torch.randn((r1 - r0, H), generator=g, device=device,
                                 dtype=torch.float32).to(torch.bfloat16)
    return out


def make_inputs(w: Workload):
    """(topk_idx, topk_w, x_bits) for workload ``w`` (numpy, host)."""
    rng = np.random.default_rng(w.seed)
    idx, wts = route(w, rng)
    x = make_x(w, np.random.default_rng(w.seed + 1000))
    return idx, wts, x
