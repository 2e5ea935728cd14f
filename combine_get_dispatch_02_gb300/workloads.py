"""Seeded synthetic workloads for MoE dispatch / combine.

This module only draws inputs: token activations, routing (top-k expert ids
and their weights) and stand-in expert outputs for the combine.  It contains
none of the dispatch / combine arithmetic, so both the CUDA path's tests and
the CPU oracle's tests take their inputs from here.

All draws use numpy's PCG64 with fixed seeds, so the same workload is produced
on every machine.  BF16 tensors are returned as ``uint16`` bit patterns (the
bf16 cast is torch's CPU cast).

Workloads (hidden 7168 / top-8 / 128 tokens per rank is the DeepSeek-V3/R1
low-latency setting of "如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南",
section 核心优势; group-limited gating is the routing the DeepTech
announcement of DeepEP (010bt.com) says the normal kernels are aligned with):

* ``tiny``   R=4 x 32 tokens, H=1024, E=32, top-4, BF16 dispatch, padded.
* ``ll``     R=32 x 128 tokens, H=7168, x ~ N(0,1) times a per-token
             log-uniform[1e-2, 1e2] scale, E=256, top-8, FP8 dispatch, padded
             per-expert buffers of 32*128 rows.
* ``normal`` R=8 x 4096 tokens, H=7168, E=256 in 8 groups of 32; top-4 groups
             by group max of the softmax score, then top-8 experts inside them;
             packed (prefix-sum) layout; BF16 and FP8 dispatch.
* ``skew``   R=16 x 512 tokens, H=4096, E=64, top-6 drawn without replacement
             with popularity (pi(e)+1)^-1.2 for a seeded permutation pi.
* sweep points: ``sweep_points()``.
"""
from __future__ import annotations

import dataclasses
import itertools

import numpy as np
import torch

PADDED = "padded"
PACKED = "packed"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_ranks: int            # R virtual EP ranks
    tokens_per_rank: int      # T tokens on each rank
    max_tokens_per_rank: int  # T_max = num_max_dispatch_tokens_per_rank
    hidden: int               # H
    num_experts: int          # E (E % R == 0; expert e lives on rank e // (E // R))
    topk: int                 # K
    layout: str               # PADDED or PACKED
    use_fp8: bool             # FP8 (e4m3, per-128 scales) or BF16 dispatch
    routing: str              # "uniform", "group", "zipf"
    x_scale: str              # "unit" or "loguniform"
    seed: int

    @property
    def num_tokens(self) -> int:
        return self.num_ranks * self.tokens_per_rank

    @property
    def num_entries(self) -> int:
        return self.num_tokens * self.topk

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


TINY = Workload("tiny", 4, 32, 32, 1024, 32, 4, PADDED, False, "uniform", "unit", 1001)
LL = Workload("ll", 32, 128, 128, 7168, 256, 8, PADDED, True, "uniform", "loguniform", 1002)
NORMAL = Workload("normal", 8, 4096, 4096, 7168, 256, 8, PACKED, False, "group", "unit", 1003)
SKEW = Workload("skew", 16, 512, 512, 4096, 64, 6, PADDED, True, "zipf", "unit", 1004)

WORKLOADS = {w.name: w for w in (TINY, LL, NORMAL, SKEW)}

# Groups for group-limited gating in the ``normal`` workload.
NORMAL_GROUPS = 8
NORMAL_TOPK_GROUPS = 4
ZIPF_S = 1.2


def sweep_points(padded_budget_bytes: int = 48 << 30):
    """The sweep grid: T x R x H x E x K x {BF16, FP8}.  Padded layout when
    E*R*T*H*2 bytes fit the budget, else packed."""
    pts = []
    for T, R, H, E, K, fp8 in itertools.product(
            (1, 8, 32, 128, 512, 2048, 8192), (8, 32), (2048, 4096, 7168),
            (64, 256), (2, 6, 8), (False, True)):
        lay = PADDED if E * R * T * H * 2 <= padded_budget_bytes else PACKED
        name = f"sweep_T{T}_R{R}_H{H}_E{E}_K{K}_{'fp8' if fp8 else 'bf16'}"
        seed = 5000 + len(pts)
        pts.append(Workload(name, R, T, T, H, E, K, lay, fp8, "uniform", "unit", seed))
    return pts


# ---------------------------------------------------------------- helpers

def _bf16_bits(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _softmax(z: np.ndarray) -> np.ndarray:
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def _topk_desc(v: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries per row, largest first, ties to the
    lower index (stable sort of -v)."""
    return np.argsort(-v, axis=-1, kind="stable")[..., :k]


def _route(w: Workload, rng: np.random.Generator):
    N, E, K = w.num_tokens, w.num_experts, w.topk
    if w.routing == "uniform":
        logits = rng.standard_normal((N, E), dtype=np.float32)
        idx = _topk_desc(logits, K)
        chosen = np.take_along_axis(logits, idx, axis=1)
        weights = _softmax(chosen.astype(np.float64))
    elif w.routing == "group":
        G, TG = NORMAL_GROUPS, NORMAL_TOPK_GROUPS
        logits = rng.standard_normal((N, E), dtype=np.float32)
        score = _softmax(logits.astype(np.float64))
        gmax = score.reshape(N, G, E // G).max(axis=2)
        keep = _topk_desc(gmax, TG)
        mask = np.zeros((N, G), bool)
        np.put_along_axis(mask, keep, True, axis=1)
        masked = np.where(np.repeat(mask, E // G, axis=1), score, -np.inf)
        idx = _topk_desc(masked, K)
        chosen = np.take_along_axis(score, idx, axis=1)
        weights = chosen / chosen.sum(axis=1, keepdims=True)
    elif w.routing == "zipf":
        perm = rng.permutation(E)
        pop = (perm + 1.0) ** (-ZIPF_S)
        pop /= pop.sum()
        # sampling K without replacement with probability proportional to pop
        # is the top-K of log(pop) + Gumbel noise
        gumbel = rng.gumbel(size=(N, E))
        idx = _topk_desc(np.log(pop)[None, :] + gumbel, K)
        logits = rng.standard_normal((N, E), dtype=np.float32)
        chosen = np.take_along_axis(logits, idx, axis=1)
        weights = _softmax(chosen.astype(np.float64))
    else:
        raise ValueError(w.routing)
    return idx.astype(np.int64), weights.astype(np.float32)


def generate(w: Workload, with_x: bool = True) -> dict:
    """x_bits uint16 [R, T, H] (unless with_x is False); topk_idx int64
    [R, T, K]; topk_weights float32 [R, T, K].  The routing is drawn before
    x, so it does not depend on with_x."""
    rng = np.random.default_rng(w.seed)
    R, T, H, K = w.num_ranks, w.tokens_per_rank, w.hidden, w.topk
    idx, weights = _route(w, rng)
    if not with_x:
        return dict(topk_idx=idx.reshape(R, T, K), topk_weights=weights.reshape(R, T, K))
    x = rng.standard_normal((R * T, H), dtype=np.float32)
    if w.x_scale == "loguniform":
        s = 10.0 ** rng.uniform(-2.0, 2.0, size=(R * T, 1))
        x = (x * s.astype(np.float32)).astype(np.float32)
    return dict(x_bits=_bf16_bits(x).reshape(R, T, H),
                topk_idx=idx.reshape(R, T, K),
                topk_weights=weights.reshape(R, T, K))


def expert_outputs(w: Workload, tokens=None) -> np.ndarray:
    """Stand-in expert outputs for the combine: bf16 bits [len(tokens), K, H]
    ~ N(0,1), row (g, k) being what expert topk_idx[g, k] returns for token g.
    Each token has its own seeded stream, so any subset can be drawn."""
    tokens = np.arange(w.num_tokens) if tokens is None else np.asarray(tokens)
    out = np.empty((len(tokens), w.topk, w.hidden), np.uint16)
    for i, g in enumerate(tokens):
        rng = np.random.default_rng([w.seed, 2, int(g)])
        out[i] = _bf16_bits(rng.standard_normal((w.topk, w.hidden), dtype=np.float32))
    return out


def inject_masks(topk_idx: np.ndarray, frac: float, seed: int) -> np.ndarray:
    """Copy of topk_idx with a seeded fraction of entries set to -1 ("no expert")."""
    rng = np.random.default_rng(seed)
    out = topk_idx.copy()
    out[rng.random(out.shape) < frac] = -1
    return out
