"""Oracle of the node budget and of the adaptive budget controller (plain Python).

TEST INFRASTRUCTURE: used by the test suite only; shares no code with the CUDA path.

IluvatarLabs/vllm PR #3 ("SCV vectorized masking"), adaptive mode: the number of speculative
tokens verified per step is adjusted from the recent acceptance ratios so as to hold a target
ratio. The page gives no formula. The reading written out here:

* Node budget. Draft nodes are numbered in topological order (parent[i] < i), so the first n
  nodes of a tree form a tree. Verifying request b under budget n means verifying that
  truncated tree: rows, tokens and parents of nodes 0..n-1, the child uniform slots 1..n-1 and
  the bonus uniform, which stays in slot N of the full [N+1] layout.
* Acceptance ratio of a step: sum over the usable requests (status 0, budget in [1, N], valid
  parents) of the accepted length, divided by the sum of the deepest node depth within each
  request's budget (the most that request could accept; k for a chain of k drafts).
* Moving average: ema <- (1 - alpha) * ema + alpha * ratio, only when that denominator is > 0.
* Budget: clamped to [n_min, n_max], then + step (capped at n_max) if ema > target + band,
  - step (floored at n_min) if ema < target - band, else unchanged.

The float64 expressions are evaluated in exactly this order, so a device implementation that
rounds each operation the same way reproduces the state bit for bit.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class Params:
    target: float
    alpha: float
    band: float
    n_min: int
    n_max: int
    step: int = 1


@dataclass
class State:
    ema: float
    budget: int
    steps: int = 0


def node_depth(parent_row, i: int):
    """Edges from node i up to the root, counted by walking the parent links (None if the
    chain leaves [0, i) or does not end at a root marked -1)."""
    d, node = 0, i
    while node != 0:
        p = int(parent_row[node])
        if p < 0 or p >= node:
            return None
        node, d = p, d + 1
    return d if int(parent_row[0]) == -1 else None


def max_depth(parent_row, n: int):
    """Deepest node among nodes 0..n-1 (None if a parent link there is invalid)."""
    best = 0
    for i in range(n):
        d = node_depth(parent_row, i)
        if d is None:
            return None
        best = max(best, d)
    return best


def truncate(logits, tokens, parent, uniforms, n: int, draft=None):
    """The inputs of one request verified under budget n (arrays of that request only):
    rows, tokens and parents of nodes 0..n-1, uniforms of slots 0..n-1 and the bonus slot N."""
    N = parent.shape[-1]
    u = None
    if uniforms is not None:
        u = np.concatenate([uniforms[:n], uniforms[N:N + 1]])
    d = None if draft is None else draft[:n]
    return logits[:n], tokens[:n], parent[:n], u, d


def update(params: Params, state: State, accept_len, status, parent, n_active) -> State:
    """One controller step; returns the new state (the caller writes state.budget to every
    request's n_active)."""
    A = 0
    D = 0
    N = parent.shape[1]
    for b in range(len(accept_len)):
        if int(status[b]) != 0:
            continue
        n = int(n_active[b])
        if n < 1 or n > N:
            continue
        dm = max_depth(parent[b], n)
        if dm is None:
            continue
        A += int(accept_len[b])
        D += dm
    k = min(max(int(state.budget), params.n_min), params.n_max)
    ema, steps = float(state.ema), int(state.steps)
    if D > 0:
        ratio = float(A) / float(D)
        ema = (1.0 - params.alpha) * ema + params.alpha * ratio
        steps += 1
        if ema > params.target + params.band:
            k = min(k + params.step, params.n_max)
        elif ema < params.target - params.band:
            k = max(k - params.step, params.n_min)
    return State(ema=ema, budget=k, steps=steps)
