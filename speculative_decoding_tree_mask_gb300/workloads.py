"""Seeded synthetic verify workloads (draft trees, logits, draft rows, uniforms).

This module only draws inputs; it computes no step of verification. The test suite feeds the
same tensors to the CUDA path and to the oracle.

The shapes follow the workloads of EmbodiInfer PR #11 "perf(activevln): grammar-trie
speculation and lossless throughput" (commit 4b728e2: a grammar trie of N most likely nodes
verified in one forward over a Qwen2-VL-class ~152k vocabulary, N=32 at B=4) and of its decode
benchmarks (B=4/8, trees of 15-31 nodes); no dataset, policy or grammar is available, so:

* tries are grown breadth-first (parent[i] < i) with a per-node branching count drawn
  uniformly from 1..max_branch, up to a depth limit;
* child tokens are distinct among siblings, drawn as Zipf(1.1) ranks mapped through a
  per-node random affine bijection of the vocabulary (a stand-in for "top-ranked tokens of a
  seeded prior");
* logits are N(0, sigma) (bf16 or fp32), plus a boost on one "grammar" token per node, which
  is the node's first child's token with probability 0.7 and a uniform token otherwise;
* uniforms are fp32 in [0, 1), shape [B, N+1].
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    N: int
    V: int
    dtype: str            # "bf16" | "f32"
    sigma: float
    mode: str             # "greedy" | "sample" | "dense"
    temperature: float = 0.0
    boost: float = 0.0
    p_boost_child: float = 0.7
    max_depth: int = 8
    max_branch: int = 4
    chain: bool = False
    p_argmax_draft: float = 0.0   # tiny chain: draft = row argmax with this probability
    draft_noise: float = 0.0      # dense chain: draft logits = target + N(0, draft_noise)
    seed: int = 0

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    @property
    def draft_nodes(self) -> int:
        return self.B * (self.N - 1)

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_chain": Workload("tiny_chain", B=2, N=5, V=1000, dtype="f32", sigma=2.0,
                           mode="greedy", chain=True, p_argmax_draft=0.7, seed=1001),
    "greedy_trie": Workload("greedy_trie", B=4, N=32, V=151936, dtype="bf16", sigma=3.0,
                            mode="greedy", boost=8.0, max_depth=8, max_branch=4, seed=1002),
    "sampling_trie": Workload("sampling_trie", B=8, N=32, V=151936, dtype="bf16", sigma=3.0,
                              mode="sample", temperature=0.7, boost=8.0, max_depth=8,
                              max_branch=4, seed=1003),
    "dense_chain": Workload("dense_chain", B=64, N=6, V=128256, dtype="bf16", sigma=2.0,
                            mode="dense", temperature=1.0, chain=True, draft_noise=0.5,
                            seed=1004),
    "large_tree": Workload("large_tree", B=256, N=64, V=152064, dtype="bf16", sigma=3.0,
                           mode="sample", temperature=1.0, boost=8.0, max_depth=10,
                           max_branch=6, seed=1005),
}


# ---- trees -------------------------------------------------------------------------------

def random_trie(rng: np.random.Generator, N: int, max_depth: int, max_branch: int) -> np.ndarray:
    """Breadth-first trie of exactly N nodes (parent[0] = -1, parent[i] < i)."""
    if N == 1:
        return np.array([-1], np.int32)
    parent = [-1]
    depth = [0]
    frontier = [0]
    while len(parent) < N:
        if not frontier:
            # depth limit exhausted the frontier: widen the shallowest nodes again
            frontier = [i for i in range(len(parent)) if depth[i] < max_depth]
            if not frontier:
                raise ValueError("N does not fit under max_depth")
        nxt = []
        for node in frontier:
            if depth[node] >= max_depth:
                continue
            k = int(rng.integers(1, max_branch + 1))
            for _ in range(k):
                if len(parent) == N:
                    break
                parent.append(node)
                depth.append(depth[node] + 1)
                nxt.append(len(parent) - 1)
        frontier = nxt
    return np.array(parent, np.int32)


def chain(N: int) -> np.ndarray:
    return np.arange(-1, N - 1, dtype=np.int32)


def _affine_perm(rng: np.random.Generator, V: int):
    if V == 1:
        return lambda rank: 0
    while True:
        a = int(rng.integers(1, V))
        if math.gcd(a, V) == 1:
            break
    c = int(rng.integers(0, V))
    return lambda rank: (a * rank + c) % V


def child_tokens(rng: np.random.Generator, parent: np.ndarray, V: int) -> np.ndarray:
    """Sibling tokens drawn as Zipf(1.1) ranks through a per-node bijection, distinct among
    siblings while the vocabulary allows (a node with more children than V tokens repeats
    tokens). The root's token is a placeholder (0)."""
    N = len(parent)
    tok = np.zeros(N, np.int32)
    for node in range(N):
        kids = [c for c in range(node + 1, N) if parent[c] == node]
        if not kids:
            continue
        perm = _affine_perm(rng, V)
        used = set()
        for c in kids:
            if len(used) >= V:
                t = int(rng.integers(0, V))
            else:
                for _ in range(64):
                    rank = int(rng.zipf(1.1)) - 1
                    if rank < V and perm(rank) not in used:
                        break
                else:   # rare: fall back to the lowest unused rank
                    rank = next(r for r in range(V) if perm(r) not in used)
                t = perm(rank)
                used.add(t)
            tok[c] = t
    return tok


def make_trees(w: Workload, seed: int | None = None):
    """parent, draft_token int32 [B, N] (numpy)."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    parents, toks = [], []
    for _ in range(w.B):
        par = chain(w.N) if w.chain else random_trie(rng, w.N, w.max_depth, w.max_branch)
        parents.append(par)
        toks.append(child_tokens(rng, par, w.V))
    return np.stack(parents), np.stack(toks)


# ---- logits, drafts, uniforms ----------------------------------------------------------------

def make_logits(w: Workload, parent: np.ndarray, tok: np.ndarray, device="cpu",
                seed: int | None = None, rows_per_chunk: int = 512) -> torch.Tensor:
    """logits [B, N, V] in the workload dtype: N(0, sigma) plus the per-node boost."""
    seed = w.seed if seed is None else seed
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty((w.B, w.N, w.V), dtype=w.torch_dtype, device=device)
    flat = out.view(w.B * w.N, w.V)
    for r0 in range(0, w.B * w.N, rows_per_chunk):
        r1 = min(w.B * w.N, r0 + rows_per_chunk)
        x = torch.randn((r1 - r0, w.V), generator=g, device=device, dtype=torch.float32)
        flat[r0:r1] = (x * w.sigma).to(w.torch_dtype)
    if w.boost:
        rng = np.random.default_rng(seed + 7)
        rows, cols = [], []
        for b in range(w.B):
            for i in range(w.N):
                kids = [c for c in range(i + 1, w.N) if parent[b, c] == i]
                if kids and rng.random() < w.p_boost_child:
                    gtok = int(tok[b, kids[0]])
                else:
                    gtok = int(rng.integers(0, w.V))
                rows.append(b * w.N + i)
                cols.append(gtok)
        ri = torch.tensor(rows, device=device)
        ci = torch.tensor(cols, device=device)
        vals = flat[ri, ci].float() + w.boost
        flat[ri, ci] = vals.to(w.torch_dtype)
    return out


def plant_argmax_drafts(w: Workload, logits: torch.Tensor, tok: np.ndarray,
                        seed: int | None = None) -> np.ndarray:
    """Tiny-chain recipe: draft token i+1 is row i's argmax with probability p_argmax_draft,
    else uniform. Returns a new token array."""
    rng = np.random.default_rng((w.seed if seed is None else seed) + 11)
    tok = tok.copy()
    am = logits.float().argmax(dim=-1).cpu().numpy()
    for b in range(w.B):
        for i in range(1, w.N):
            if rng.random() < w.p_argmax_draft:
                tok[b, i] = am[b, i - 1]
            else:
                tok[b, i] = int(rng.integers(0, w.V))
    return tok


def make_dense_draft(w: Workload, logits: torch.Tensor, seed: int | None = None):
    """Dense-chain recipe: draft logits = target + N(0, draft_noise) in the workload dtype,
    and draft token i+1 sampled from softmax(draft row i / T). Returns (draft, tok)."""
    seed = (w.seed if seed is None else seed) + 13
    dev = logits.device
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    draft = torch.empty_like(logits)
    for b in range(w.B):
        noise = torch.randn(logits[b].shape, generator=g, device=dev, dtype=torch.float32)
        draft[b] = (logits[b].float() + w.draft_noise * noise).to(logits.dtype)
    probs = torch.softmax(draft[:, :-1].float() / w.temperature, dim=-1)
    picks = torch.multinomial(probs.reshape(-1, w.V), 1, generator=g).reshape(w.B, w.N - 1)
    tok = np.zeros((w.B, w.N), np.int32)
    tok[:, 1:] = picks.cpu().numpy()
    return draft, tok


def make_uniforms(w: Workload, device="cpu", seed: int | None = None) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed((w.seed if seed is None else seed) + 17)
    return torch.rand((w.B, w.N + 1), generator=g, device=device, dtype=torch.float32)


def make(w: Workload, device="cpu", seed: int | None = None) -> dict:
    """All inputs of one verify step. Tensors on ``device``; trees also as numpy."""
    parent, tok = make_trees(w, seed)
    out = {}
    if w.mode == "dense":
        logits = make_logits(w, parent, tok, device, seed)
        draft, tok = make_dense_draft(w, logits, seed)
        out["draft"] = draft
    else:
        logits = make_logits(w, parent, tok, device, seed)
        if w.p_argmax_draft:
            tok = plant_argmax_drafts(w, logits, tok, seed)
    out.update(
        logits=logits,
        parent_np=parent,
        tok_np=tok,
        parent=torch.from_numpy(parent).to(device),
        draft_token=torch.from_numpy(tok).to(device),
        uniforms=make_uniforms(w, device, seed),
    )
    return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host view of a bf16 tensor as uint16 bit patterns (the oracle's bf16 input form)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host_logits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.detach().contiguous().cpu().numpy().astype(np.float32, copy=False)
