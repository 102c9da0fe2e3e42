"""Exact output distributions of tree verification on tiny vocabularies (pure Python, float64).

TEST INFRASTRUCTURE: part of the oracle, used only by the test suite. Shares no code with the
CUDA path.

Losslessness is the claim of EmbodiInfer PR #11 "perf(activevln): grammar-trie speculation and
lossless throughput", commit 4b728e2: greedy keeps the argmax path and sampling uses standard
rejection sampling against the draft, so the output distribution is unchanged. This module
states that claim as arithmetic that can be checked:

* ``SyntheticLM`` is a table of logits for every prefix (any path of the tree has a row), so a
  tree's logits rows and the target's autoregressive distribution come from one object.
* ``verify_point_dist`` / ``verify_dense_dist`` integrate the verify procedure over its
  uniforms analytically: each accept test ``u < x`` with ``u ~ U[0, 1)`` succeeds with
  probability ``min(1, max(x, 0))`` and the bonus draw picks ``v`` with probability
  ``r(v) / sum r``.
* ``target_stopped_dist`` samples the target autoregressively and stops at the first token
  that leaves the tree (the token is emitted); ``extend`` continues any emitted prefix with
  target samples up to a fixed length and ``target_joint`` is the target's joint law.

Losslessness means ``verify_*_dist`` (mixed over the draft's own sampling for dense drafts),
extended to a fixed length, equals ``target_joint``; for point-mass tries also the stopped law.
"""
from __future__ import annotations

import itertools
import math
from collections import defaultdict

import numpy as np


def softmax(z, T: float) -> list[float]:
    """softmax(z / T) in float64: exp((z - m)/T) / sum exp((z_w - m)/T), m = max z."""
    m = max(z)
    e = [math.exp((float(x) - m) / T) if x != -math.inf else 0.0 for x in z]
    s = sum(e)
    return [x / s for x in e]


class SyntheticLM:
    """Deterministic logits for every prefix: float32 values ~ N(0, scale), seeded by the
    prefix, with an optional set of (prefix, token, value) overrides."""

    def __init__(self, V: int, seed: int, scale: float = 1.5):
        self.V, self.seed, self.scale = V, seed, scale
        self.overrides: dict[tuple, dict[int, float]] = {}
        self._cache: dict[tuple, np.ndarray] = {}

    def logits(self, prefix: tuple) -> np.ndarray:
        prefix = tuple(int(t) for t in prefix)
        if prefix not in self._cache:
            key = [self.seed, len(prefix)] + [t + 1 for t in prefix]
            rng = np.random.default_rng(key)
            z = (rng.standard_normal(self.V) * self.scale).astype(np.float32)
            for t, val in self.overrides.get(prefix, {}).items():
                z[t] = np.float32(val)
            self._cache[prefix] = z
        return self._cache[prefix]

    def probs(self, prefix: tuple, T: float) -> list[float]:
        return softmax([float(x) for x in self.logits(prefix)], T)


def children(parent, node: int) -> list[int]:
    return [c for c in range(node + 1, len(parent)) if parent[c] == node]


def prefixes(tokens, parent) -> list[tuple]:
    """Prefix (tokens after the root) of every node of a topologically ordered tree."""
    out = [()]
    for i in range(1, len(parent)):
        out.append(out[parent[i]] + (int(tokens[i]),))
    return out


def tree_rows(model: SyntheticLM, tokens, parent) -> np.ndarray:
    """Logits rows [N, V] float32: row i is the model's logits after node i's prefix."""
    return np.stack([model.logits(p) for p in prefixes(tokens, parent)])


def verify_point_dist(model, tokens, parent, T: float) -> dict:
    """Exact law of the emitted sequence (accepted tokens then bonus) for point-mass drafts."""
    pre = prefixes(tokens, parent)

    def at(node):
        p = model.probs(pre[node], T)
        out = defaultdict(float)
        reach, R = 1.0, set()
        for c in children(parent, node):
            t = int(tokens[c])
            if t in R:
                rhat = 0.0
            else:
                S = sum(p[v] for v in range(model.V) if v not in R)
                rhat = p[t] / S
            if rhat > 0:
                for seq, pr in at(c).items():
                    out[(t,) + seq] += reach * min(1.0, rhat) * pr
            reach *= 1.0 - min(1.0, rhat)
            R.add(t)
        r = [0.0 if v in R else p[v] for v in range(model.V)]
        Sr = sum(r)
        for v in range(model.V):
            if r[v] > 0:
                out[(v,)] += reach * r[v] / Sr
        return out

    return dict(at(0))


def verify_dense_dist(model, draft_model, tokens, parent, T: float) -> dict:
    """Exact law of the emitted sequence for one fixed draft tree with dense draft rows
    q_i = draft_model.probs(prefix(i)). Residuals follow max(r - q, 0) / Z per rejection."""
    pre = prefixes(tokens, parent)

    def at(node):
        p = model.probs(pre[node], T)
        r = list(p)
        out = defaultdict(float)
        kids = children(parent, node)
        reach = 1.0
        if kids:
            q = draft_model.probs(pre[node], T)
            for c in kids:
                x = int(tokens[c])
                if q[x] > 0:
                    acc = min(1.0, r[x] / q[x])
                else:
                    acc = 1.0 if r[x] > 0 else 0.0
                if acc > 0:
                    for seq, pr in at(c).items():
                        out[(x,) + seq] += reach * acc * pr
                reach *= 1.0 - acc
                d = [max(r[v] - q[v], 0.0) for v in range(model.V)]
                Z = sum(d)
                if Z > 0:
                    r = [x_ / Z for x_ in d]
        Sr = sum(r)
        for v in range(model.V):
            if r[v] > 0:
                out[(v,)] += reach * r[v] / Sr
        return out

    return dict(at(0))


def dense_chain_mixture(model, draft_model, k: int, T: float) -> dict:
    """Emitted-sequence law for a chain of k drafts sampled from the draft model itself
    (x_{i+1} ~ q(. | x_1..x_i)), mixed over all V^k draft chains."""
    parent = [-1] + list(range(k))
    out = defaultdict(float)
    for xs in itertools.product(range(model.V), repeat=k):
        w, pre = 1.0, ()
        for x in xs:
            w *= draft_model.probs(pre, T)[x]
            pre = pre + (x,)
        if w == 0:
            continue
        for seq, pr in verify_dense_dist(model, draft_model, (0,) + xs, parent, T).items():
            out[seq] += w * pr
    return dict(out)


def dense_tree_mixture(model, draft_model, parent, T: float) -> dict:
    """Emitted-sequence law for a tree shape whose children are drawn i.i.d. (with
    replacement) from their parent's draft row, mixed over all token assignments."""
    N = len(parent)
    out = defaultdict(float)
    for xs in itertools.product(range(model.V), repeat=N - 1):
        tokens = (0,) + xs
        pre = prefixes(tokens, parent)
        w = 1.0
        for i in range(1, N):
            w *= draft_model.probs(pre[parent[i]], T)[tokens[i]]
            if w == 0:
                break
        if w == 0:
            continue
        for seq, pr in verify_dense_dist(model, draft_model, tokens, parent, T).items():
            out[seq] += w * pr
    return dict(out)


def target_stopped_dist(model, tokens, parent, T: float) -> dict:
    """Target autoregressive sampling from the root, following the tree while the sampled
    token equals a child's token (the first such child) and stopping after the first token
    that leaves the tree."""
    pre = prefixes(tokens, parent)

    def at(node):
        p = model.probs(pre[node], T)
        out = defaultdict(float)
        kids = children(parent, node)
        for v in range(model.V):
            if p[v] == 0:
                continue
            nxt = next((c for c in kids if int(tokens[c]) == v), None)
            if nxt is None:
                out[(v,)] += p[v]
            else:
                for seq, pr in at(nxt).items():
                    out[(v,) + seq] += p[v] * pr
        return out

    return dict(at(0))


def extend(dist: dict, model, T: float, length: int) -> dict:
    """Continue every emitted prefix with target samples up to ``length`` tokens."""
    out = defaultdict(float)

    def grow(seq, pr):
        if len(seq) >= length:
            out[seq[:length]] += pr
            return
        p = model.probs(seq, T)
        for v in range(model.V):
            if p[v] > 0:
                grow(seq + (v,), pr * p[v])

    for seq, pr in dist.items():
        grow(tuple(seq), pr)
    return dict(out)


def target_joint(model, T: float, length: int) -> dict:
    return extend({(): 1.0}, model, T, length)


def max_abs_diff(a: dict, b: dict) -> float:
    keys = set(a) | set(b)
    return max((abs(a.get(k, 0.0) - b.get(k, 0.0)) for k in keys), default=0.0)
