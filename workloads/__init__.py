"""Seeded synthetic inputs for speculative-sampling verification.

This module is shared by the tests, the benchmark and the smoke check: it
feeds the same bytes to the CUDA path and to the oracle.  It holds none of the
verification arithmetic (no softmax, no acceptance test, no inverse CDF).  The
draft tokens are drawn with the Gumbel-max trick (argmax of z/T plus Gumbel
noise), which samples from softmax(z/T) without computing it; the uniforms
come from Philox4x32-10 (see ``philox.py``).

The five workloads follow the rollout-shaped batches used for measurement:
vocabulary sizes of Qwen-class (151936) and Llama-3-class (128256) models,
draft lengths k=3 (the best setting reported in "Accelerating RL Post-Training
Rollouts via System-Integrated Speculative Decoding", §4 main findings) and
k=7 (the long draft that page reports as too costly), ragged per-sequence
draft lengths with 0 meaning speculation is off ("EfficientRollout:
System-Aware Self-Speculative Decoding for RL Rollouts", abstract: SD toggle
policy), and GRPO groups whose samples share a prompt ("ReSpec: Towards
Optimizing Speculative Decoding in Reinforcement Learning Systems",
background).  None of the pages' datasets is used; these synthetic logits
stand in for them.

Tensor layout (all row-major, contiguous):
  target    [B, k+1, V]  float32 or bfloat16; rows i > k_b are padding
  draft     [B, k,   V]  same dtype; rows i >= k_b are padding
  tokens    [B, k]       int32; entries i >= k_b are -1
  draft_len [B]          int32 in [0, k]
  uniforms  [B, k+1]     float32 in [0, 1); columns 0..k-1 are the accept
                         tests, column k is the sampling uniform
Padding rows are filled with NaN so that any read of them is visible.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

from .philox import philox_uniforms, philox4x32_10  # noqa: F401

__all__ = [
    "Workload", "WORKLOADS", "get_workload", "make_inputs", "make_tables",
    "philox_uniforms", "philox4x32_10", "gumbel_argmax_tokens", "algorithmic_bytes",
    "TreeWorkload", "TREE_WORKLOADS", "get_tree_workload", "tree_parents", "tree_algorithmic_bytes",
    "make_tree_inputs",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    k: int
    V: int
    dtype: str             # "f32" or "bf16"
    T: float
    kind: str              # generator recipe, see make_inputs
    draft_sigma: float
    ragged: bool = False
    group: int = 1         # GRPO group size (rows of a group share a base)
    seed: int = 0

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elt(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def describe(self) -> str:
        kk = f"k_b~U{{0..{self.k}}}" if self.ragged else f"k={self.k}"
        return f"{self.name}: B={self.B} {kk} V={self.V} {self.dtype} T={self.T}"


WORKLOADS = {
    # tiny: N(0, 2^2) target, draft = target + N(0, 0.5^2), fp32
    "tiny": Workload("tiny", 4, 3, 1024, "f32", 1.0, "normal", 0.5, seed=1),
    # Qwen vocabulary, N(0, 3^2) + 20 peaked ids per row, draft noise 1.0
    "qwen_b32": Workload("qwen_b32", 32, 3, 151936, "bf16", 1.0, "peaked", 1.0, seed=2),
    # ragged draft lengths k_b in {0,1,2,3}, Llama-3 vocabulary
    "ragged": Workload("ragged", 256, 3, 128256, "bf16", 1.0, "peaked", 0.7, ragged=True, seed=3),
    # the same shape with every k_b = 3
    "ragged_dense": Workload("ragged_dense", 256, 3, 128256, "bf16", 1.0, "peaked", 0.7, seed=3),
    # long stale draft, heavy-tailed logits, T = 0.6
    "long_draft": Workload("long_draft", 512, 7, 151936, "bf16", 0.6, "student_t", 1.5, seed=4),
    # GRPO groups of 8 sharing a base, near-full acceptance self-drafter
    "grpo": Workload("grpo", 1024, 3, 151936, "bf16", 1.0, "grpo", 0.1, group=8, seed=5),
}


def get_workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return dataclasses.replace(w, **overrides) if overrides else w


def algorithmic_bytes(draft_len: np.ndarray, k: int, V: int, elt: int) -> int:
    """Bytes the verification must move once: every needed logit row read
    once (target rows 0..k_b, draft rows 0..k_b-1), the small inputs
    (tokens, lengths, uniforms) and the outputs (tokens [B,k+1], lengths)."""
    kb = np.asarray(draft_len, dtype=np.int64)
    B = kb.shape[0]
    rows = int(np.sum(2 * kb + 1))
    small = B * k * 4 + B * 4 + B * (k + 1) * 4
    outs = B * (k + 1) * 4 + B * 4
    return rows * V * elt + small + outs


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _peaked_rows(n, V, g, device, sigma=3.0, peaks=20, boost=8.0, chunk=256):
    out = torch.empty(n, V, dtype=torch.float32, device=device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        r = torch.randn(e - s, V, generator=g, device=device) * sigma
        keys = torch.rand(e - s, V, generator=g, device=device)
        ids = keys.topk(peaks, dim=1).indices
        r.scatter_add_(1, ids, torch.full_like(ids, boost, dtype=torch.float32))
        out[s:e] = r
    return out


def _student_t_rows(n, V, g, device, dof=3, scale=2.5, chunk=256):
    out = torch.empty(n, V, dtype=torch.float32, device=device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        z = torch.randn(e - s, V, generator=g, device=device)
        chi = torch.zeros_like(z)
        for _ in range(dof):
            chi += torch.randn(e - s, V, generator=g, device=device) ** 2
        out[s:e] = scale * z / torch.sqrt(chi / dof)
    return out


def gumbel_argmax_tokens(logits: torch.Tensor, T: float, g, chunk=256) -> torch.Tensor:
    """One draw per row from softmax(logits/T) by the Gumbel-max trick
    (argmax of logits/T + Gumbel noise).  T == 0 gives the row argmax.
    logits: [n, V] (any float dtype).  Returns int32 [n]."""
    n, V = logits.shape
    out = torch.empty(n, dtype=torch.int32, device=logits.device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        z = logits[s:e].float()
        if T > 0:
            u = torch.rand(e - s, V, generator=g, device=logits.device).clamp_(min=1e-30)
            z = z / T - torch.log(-torch.log(u))
        out[s:e] = torch.argmax(z, dim=1).to(torch.int32)
    return out


def make_inputs(w: Workload, device="cpu", seed=None, B=None, uniform_seed=0):
    """Generate the inputs of workload ``w`` on ``device``.

    ``B`` overrides the batch size (for bounded samples); ``seed`` overrides
    the workload's logit seed.  Uniforms always come from Philox with key
    ``uniform_seed`` (0 by default), counter = b*(k+1) + j.
    Returns a dict of tensors on ``device`` plus ``meta``.
    """
    B = w.B if B is None else B
    k, V = w.k, w.V
    g = _gen(device, w.seed if seed is None else seed)
    rows_t = B * (k + 1)

    if w.kind == "normal":
        zt = torch.randn(rows_t, V, generator=g, device=device) * 2.0
    elif w.kind == "peaked":
        zt = _peaked_rows(rows_t, V, g, device)
    elif w.kind == "student_t":
        zt = _student_t_rows(rows_t, V, g, device)
    elif w.kind == "grpo":
        groups = math.ceil(B / w.group)
        base = _peaked_rows(groups * (k + 1), V, g, device).view(groups, k + 1, V)
        zt = torch.empty(B, k + 1, V, dtype=torch.float32, device=device)
        for b in range(0, B, 64):
            e = min(B, b + 64)
            gi = torch.arange(b, e, device=device) // w.group
            zt[b:e] = base[gi] + 0.2 * torch.randn(e - b, k + 1, V, generator=g, device=device)
        zt = zt.view(rows_t, V)
        del base
    else:
        raise ValueError(w.kind)

    target = zt.to(w.torch_dtype).view(B, k + 1, V)
    del zt
    draft = torch.empty(B, k, V, dtype=w.torch_dtype, device=device)
    for b in range(0, B, 64):
        e = min(B, b + 64)
        noise = torch.randn(e - b, k, V, generator=g, device=device) * w.draft_sigma
        draft[b:e] = (target[b:e, :k].float() + noise).to(w.torch_dtype)

    if w.ragged:
        draft_len = torch.randint(0, k + 1, (B,), generator=g, device=device, dtype=torch.int64).to(torch.int32)
    else:
        draft_len = torch.full((B,), k, dtype=torch.int32, device=device)

    tokens = gumbel_argmax_tokens(draft.view(B * k, V), w.T, g).view(B, k)
    pos = torch.arange(k, device=device).view(1, k)
    tokens = torch.where(pos < draft_len.view(B, 1).long(), tokens, torch.full_like(tokens, -1))

    # NaN-poison the padding rows: they must never be read.
    kb = draft_len.long().view(B, 1)
    pad_t = torch.arange(k + 1, device=device).view(1, k + 1) > kb
    pad_d = torch.arange(k, device=device).view(1, k) >= kb
    target[pad_t] = float("nan")
    draft[pad_d] = float("nan")

    u = philox_uniforms(B * (k + 1), seed=uniform_seed).reshape(B, k + 1)
    uniforms = torch.from_numpy(u).to(device)
    return {
        "target": target.contiguous(), "draft": draft.contiguous(),
        "tokens": tokens.contiguous(), "draft_len": draft_len.contiguous(),
        "uniforms": uniforms.contiguous(), "T": w.T,
        "meta": {"workload": w, "B": B, "k": k, "V": V},
    }


def make_tables(rng: np.random.Generator, V: int, depth: int, scale: float = 1.5):
    """Prefix-conditioned logit tables for exhaustive enumeration tests:
    a dict mapping every token prefix of length < depth to a float64 row."""
    tab = {(): rng.normal(0.0, scale, V)}
    frontier = [()]
    for _ in range(depth - 1):
        nxt = []
        for pre in frontier:
            for v in range(V):
                p = pre + (v,)
                tab[p] = rng.normal(0.0, scale, V)
                nxt.append(p)
        frontier = nxt
    return tab


# --- draft trees ----------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class TreeWorkload:
    """A batch of draft trees.  ``branching`` gives the children of every
    node per level (a full tree in breadth-first order: node 0 is the root,
    parents precede children); ``ragged`` keeps a random prefix of 1..M nodes
    per sequence (a prefix of a breadth-first order is itself a tree)."""
    name: str
    B: int
    branching: tuple
    V: int
    dtype: str
    T: float
    kind: str
    draft_sigma: float
    ragged: bool = False
    seed: int = 0

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elt(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def M(self) -> int:
        return len(tree_parents(self.branching))

    def describe(self) -> str:
        shape = "x".join(str(t) for t in self.branching)
        nodes = f"1..{self.M} nodes" if self.ragged else f"{self.M} nodes"
        return f"{self.name}: B={self.B} branching {shape} ({nodes}) V={self.V} {self.dtype} T={self.T}"


TREE_WORKLOADS = {
    # ReSpec-style configuration: branching 2 over 3 levels (15 nodes), Qwen
    # vocabulary, the same logit recipe as qwen_b32
    "tree": TreeWorkload("tree", 64, (2, 2, 2), 151936, "bf16", 1.0, "peaked", 1.0, seed=6),
    # wider first level, ragged node counts, Llama-3 vocabulary
    "tree_wide": TreeWorkload("tree_wide", 128, (4, 2), 128256, "bf16", 1.0, "peaked", 0.7, ragged=True, seed=7),
}


def get_tree_workload(name: str, **overrides) -> TreeWorkload:
    w = TREE_WORKLOADS[name]
    return dataclasses.replace(w, **overrides) if overrides else w


def tree_parents(branching) -> list:
    """Parents of a full tree with ``branching[l]`` children per node of
    level l, in breadth-first order (parents[0] = -1)."""
    parents, level = [-1], [0]
    for t in branching:
        nxt = []
        for p in level:
            for _ in range(t):
                parents.append(p)
                nxt.append(len(parents) - 1)
        level = nxt
    return parents


def tree_algorithmic_bytes(visited_t: int, visited_d: int, B: int, M: int, V: int, elt: int) -> int:
    """Bytes a tree verification must move once: the target rows of the
    visited nodes and the draft rows of the visited nodes with children, the
    small inputs (parents, tokens, n_nodes, uniforms) and the outputs."""
    small = B * M * 4 * 3 + B * 4
    outs = B * M * 4 * 2 + B * 4 * 2
    return (visited_t + visited_d) * V * elt + small + outs


def make_tree_inputs(w: TreeWorkload, device="cpu", seed=None, B=None, uniform_seed=0):
    """Inputs of tree workload ``w``: target, draft [B, M, V], parents,
    tokens [B, M] int32, n_nodes [B] int32, uniforms [B, M] float32
    (Philox, counter b*M + j; column 0 samples).  Each child's token is a
    draw from softmax(z^d/T) of its parent's draft row (T = 1 for greedy
    workloads).  Draft rows of nodes without children and every row past a
    sequence's last node are NaN: they must never be read."""
    B = w.B if B is None else B
    V = w.V
    par = tree_parents(w.branching)
    M = len(par)
    g = _gen(device, w.seed if seed is None else seed)
    rows = B * M
    if w.kind == "peaked":
        zt = _peaked_rows(rows, V, g, device)
    elif w.kind == "normal":
        zt = torch.randn(rows, V, generator=g, device=device) * 2.0
    else:
        raise ValueError(w.kind)
    target = zt.to(w.torch_dtype).view(B, M, V)
    del zt
    draft = torch.empty(B, M, V, dtype=w.torch_dtype, device=device)
    for b in range(0, B, 32):
        e = min(B, b + 32)
        noise = torch.randn(e - b, M, V, generator=g, device=device) * w.draft_sigma
        draft[b:e] = (target[b:e].float() + noise).to(w.torch_dtype)
    if w.ragged:
        n_nodes = torch.randint(1, M + 1, (B,), generator=g, device=device, dtype=torch.int64).to(torch.int32)
    else:
        n_nodes = torch.full((B,), M, dtype=torch.int32, device=device)
    parents = torch.tensor(par, dtype=torch.int32, device=device).view(1, M).repeat(B, 1)
    # child j's token: one draw from its parent's draft distribution
    pidx = torch.tensor([max(p, 0) for p in par], dtype=torch.long, device=device)
    tokens = torch.zeros(B, M, dtype=torch.int32, device=device)
    for b in range(0, B, 32):
        e = min(B, b + 32)
        src = draft[b:e, pidx].reshape((e - b) * M, V)
        tokens[b:e] = gumbel_argmax_tokens(src, w.T if w.T > 0 else 1.0, g).view(e - b, M)
    tokens[:, 0] = 0
    # poison what must not be read
    node = torch.arange(M, device=device).view(1, M)
    has_kids = torch.zeros(M, dtype=torch.bool, device=device)
    for j in range(1, M):
        has_kids[par[j]] = True
    beyond = node >= n_nodes.view(B, 1).long()
    kid_in = torch.zeros(B, M, dtype=torch.bool, device=device)
    for j in range(1, M):
        kid_in[:, par[j]] |= j < n_nodes.long()
    target[beyond] = float("nan")
    draft[beyond | ~kid_in] = float("nan")
    u = philox_uniforms(B * M, seed=uniform_seed).reshape(B, M)
    return {
        "target": target.contiguous(), "draft": draft.contiguous(), "parents": parents.contiguous(),
        "tokens": tokens.contiguous(), "n_nodes": n_nodes.contiguous(),
        "uniforms": torch.from_numpy(u).to(device).contiguous(), "T": w.T,
        "meta": {"workload": w, "B": B, "M": M, "V": V},
    }
