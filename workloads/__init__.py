"""Seeded synthetic inputs shaped like the MoE workloads the pages describe.

This module holds input generation only: router logits, top-k selection and
router probabilities (all upstream of the dispatch -> expert -> combine path),
token activations and expert weights.  It contains none of the path's own
arithmetic, so both the CUDA library's tests and the CPU oracle may consume
what it produces.

Workloads (all synthetic; no dataset is involved):

* ``tiny``    512 tokens, hidden 1024, 16 experts, top-4, intermediate 256, pad 32,
  no capacity limit.  x ~ N(0,1); logits ~ N(0,1) -> softmax over all 16 experts
  -> the top-4 values (not renormalised).  Weights ~ N(0, 0.02).  Shape basis:
  DeepEP PR #716 "perf: reuse HybridEP routing allgather buffer", Testing
  (512 tokens/rank, hidden 1024, padding multiple 32).
* ``mid``     4096 tokens, hidden 2048, 64 experts, top-8, intermediate 1024, pad 32,
  sparse Boolean routing map from logits ~ N(0,1); probs = softmax over the 8
  chosen logits; x and weights ~ N(0, 0.02); capacity factor 1.5 (4-aligned).
  Shape basis: Megatron-LM PR #4632 "moe: add DeepEP V2 ElasticBuffer support",
  Evidence (Qwen3-30B-A3B-style hidden 2048, ffn 1024, top-8).
* ``permute`` 8192 tokens, hidden 7168, 32 experts, top-8, pad 32, dense int16
  ids from uniform logits; probs = softmax over the chosen logits; identity
  experts.  NeMo Automodel PR #3931 "perf(moe): sync-free HybridEP dispatch",
  Validation (32 experts top-8, 8192 rows x 7168, capacity 1x/1.5x/2x, 1/2x).
* ``dsv3``    8192 tokens, hidden 7168, 256 experts, top-8, intermediate 2048, pad 32,
  Zipf(1.2)-skewed expert popularity (Gumbel top-8 sampling without
  replacement, probability proportional to rank^-1.2 over a seeded permutation
  of the experts); probs = softmax over the chosen N(0,1) logits; x ~ N(0,1);
  weights ~ N(0, 0.02); FP8.
* ``stress``  65536 tokens, hidden 1024, 256 experts, top-36, pad 32, N(0,1) logits.
  DeepEP PR #716, Memory impact and the standalone allgather stress test.
* ``decode64`` / ``decode256``  64 / 256 tokens, hidden 7168, 256 experts, top-8,
  intermediate 2048, N(0,1) logits, NVFP4 weights and activations.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    K: int
    I: int = 0           # 0: identity experts (no MLP)
    m: int = 32          # per-expert padding multiple
    routing: str = "dense"      # "dense" int16 ids or "sparse" Boolean map
    logits: str = "normal"      # "normal" N(0,1), "uniform" U(0,1), "zipf"
    probs: str = "renorm"       # "renorm": softmax over chosen; "softmax_all": softmax over E, top-k values
    x_std: float = 1.0
    w_std: float = 0.02
    dtype: str = "bf16"         # "bf16", "fp8", "nvfp4"
    cap_factor: float = 0.0     # 0: no capacity limit


WORKLOADS = {
    "tiny": Workload("tiny", T=512, H=1024, E=16, K=4, I=256, probs="softmax_all"),
    "mid": Workload("mid", T=4096, H=2048, E=64, K=8, I=1024, routing="sparse", x_std=0.02, cap_factor=1.5),
    "permute": Workload("permute", T=8192, H=7168, E=32, K=8, I=0, logits="uniform"),
    "dsv3": Workload("dsv3", T=8192, H=7168, E=256, K=8, I=2048, logits="zipf", dtype="fp8"),
    "stress": Workload("stress", T=65536, H=1024, E=256, K=36, I=0),
    "decode64": Workload("decode64", T=64, H=7168, E=256, K=8, I=2048, dtype="nvfp4"),
    "decode256": Workload("decode256", T=256, H=7168, E=256, K=8, I=2048, dtype="nvfp4"),
}


def unbounded_capacity(T: int, K: int, E: int, m: int) -> int:
    """A capacity no routing can exceed: every route kept plus the worst-case padding."""
    return T * K + E * (m - 1)


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (smaller parity cases)."""
    return dataclasses.replace(w, **changes)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream]))


def router(w: Workload, seed: int):
    """Top-k routing for every token.

    Returns (topk_idx int16 [T, K] with each row's ids in ascending order,
    probs float32 [T, K] aligned with topk_idx).
    """
    g = _rng(seed, 1)
    T, E, K = w.T, w.E, w.K
    if w.logits == "zipf":
        ranks = g.permutation(E) + 1
        logw = -1.2 * np.log(ranks.astype(np.float64))
        gumbel = -np.log(-np.log(g.uniform(np.finfo(np.float64).tiny, 1.0, size=(T, E))))
        chosen = np.argsort(-(logw[None, :] + gumbel), axis=1, kind="stable")[:, :K]
        logits = g.standard_normal((T, E))
    else:
        logits = g.uniform(0.0, 1.0, (T, E)) if w.logits == "uniform" else g.standard_normal((T, E))
        chosen = np.argsort(-logits, axis=1, kind="stable")[:, :K]
    chosen = np.sort(chosen, axis=1)
    sel = np.take_along_axis(logits, chosen, axis=1)
    if w.probs == "softmax_all":
        z = np.exp(logits - logits.max(axis=1, keepdims=True))
        p = np.take_along_axis(z / z.sum(axis=1, keepdims=True), chosen, axis=1)
    else:
        z = np.exp(sel - sel.max(axis=1, keepdims=True))
        p = z / z.sum(axis=1, keepdims=True)
    return chosen.astype(np.int16), p.astype(np.float32)


def to_sparse(topk_idx: np.ndarray, probs: np.ndarray, E: int):
    """The same routing as a Boolean tokens x experts map with probs [T, E] (0 off the map)."""
    T, K = topk_idx.shape
    m = np.zeros((T, E), np.uint8)
    p = np.zeros((T, E), np.float32)
    rows = np.repeat(np.arange(T), K)
    m[rows, topk_idx.reshape(-1).astype(np.int64)] = 1
    p[rows, topk_idx.reshape(-1).astype(np.int64)] = probs.reshape(-1)
    return m, p


def routing_inputs(w: Workload, seed: int, routing: str | None = None):
    """(routing_fmt, map, probs) in the workload's (or the given) routing format."""
    idx, p = router(w, seed)
    fmt = routing or w.routing
    if fmt == "sparse":
        m, ps = to_sparse(idx, p, w.E)
        return 1, m, ps
    return 0, idx, p


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """A bf16 tensor's raw bit patterns as uint16."""
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def activations(w: Workload, seed: int, device: str = "cpu") -> torch.Tensor:
    """x ~ N(0, x_std) rounded to bf16, [T, H]."""
    g = torch.Generator(device=device).manual_seed(seed * 1000 + 2)
    x = torch.randn(w.T, w.H, generator=g, device=device, dtype=torch.float32)
    return (x * w.x_std).to(torch.bfloat16)


def grad_outputs(w: Workload, seed: int, device: str = "cpu") -> torch.Tensor:
    """Gradient of the layer output, dL/dy ~ N(0, 1) rounded to bf16, [T, H]."""
    g = torch.Generator(device=device).manual_seed(seed * 1000 + 4)
    return torch.randn(w.T, w.H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def expert_weights(w: Workload, seed: int, device: str = "cpu", experts=None):
    """bf16 (w13 [E, 2I, H], w2 [E, H, I]) ~ N(0, w_std), generated expert by expert.

    ``experts`` restricts generation to a list of experts (the rest are not
    produced; the returned tensors then hold only those experts, in order).
    Expert e's values do not depend on which other experts are generated.
    """
    ids = range(w.E) if experts is None else list(experts)
    w13 = torch.empty(len(ids), 2 * w.I, w.H, dtype=torch.bfloat16, device=device)
    w2 = torch.empty(len(ids), w.H, w.I, dtype=torch.bfloat16, device=device)
    for j, e in enumerate(ids):
        g = torch.Generator(device=device).manual_seed(seed * 1000003 + 7919 * (e + 1))
        w13[j] = (torch.randn(2 * w.I, w.H, generator=g, device=device) * w.w_std).to(torch.bfloat16)
        w2[j] = (torch.randn(w.H, w.I, generator=g, device=device) * w.w_std).to(torch.bfloat16)
    return w13, w2
