"""Losslessness pins of the oracle (CPU only).

EmbodiInfer PR #11 "perf(activevln): grammar-trie speculation and lossless throughput", commit
4b728e2, claims that greedy keeps the argmax path and that sampling with standard rejection
sampling against the draft leaves the output distribution unchanged. These tests check that
claim as mathematics on vocabularies of at most 8 tokens:

* the exact law of the emitted tokens under the verify procedure (uniforms integrated
  analytically) equals target autoregressive sampling (to 1e-12);
* the C oracle, driven by seeded uniforms, reproduces that law (chi-square on 2e5 draws).
"""
import itertools

import numpy as np
import pytest
from scipy import stats

from oracle import enumerate as E
from oracle import oracle as O

TREES = [
    # (parent, tokens) -- tokens of siblings distinct unless noted
    ([-1, 0, 0, 1], [0, 1, 2, 3]),
    ([-1, 0, 0, 0, 1, 2], [0, 2, 0, 3, 1, 1]),
    ([-1, 0, 1, 2], [0, 1, 1, 2]),                # chain
    ([-1, 0, 0, 1, 1], [0, 3, 3, 0, 2]),          # duplicate sibling tokens at the root
    ([-1, 0, 0, 0, 0], [0, 0, 1, 2, 3]),          # every token of V=4 drafted at the root
]


@pytest.mark.parametrize("T", [0.6, 1.0, 1.7])
@pytest.mark.parametrize("case", range(len(TREES)))
def test_point_mass_exact_law_equals_target(case, T):
    parent, tokens = TREES[case]
    V = 4 if case != 1 else 5
    model = E.SyntheticLM(V, seed=100 + case, scale=1.3)
    got = E.verify_point_dist(model, tokens, parent, T)
    assert abs(sum(got.values()) - 1.0) < 1e-12
    assert E.max_abs_diff(got, E.target_stopped_dist(model, tokens, parent, T)) < 1e-12
    depth = max(len(p) for p in E.prefixes(tokens, parent))
    ext = E.extend(got, model, T, depth + 1)
    assert E.max_abs_diff(ext, E.target_joint(model, T, depth + 1)) < 1e-12


@pytest.mark.parametrize("k,V,T", [(1, 4, 1.0), (2, 4, 0.8), (3, 3, 1.3), (2, 5, 1.0)])
def test_dense_chain_exact_law_equals_target(k, V, T):
    model = E.SyntheticLM(V, seed=7, scale=1.5)
    draft = E.SyntheticLM(V, seed=8, scale=1.5)
    law = E.dense_chain_mixture(model, draft, k, T)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    ext = E.extend(law, model, T, k + 1)
    assert E.max_abs_diff(ext, E.target_joint(model, T, k + 1)) < 1e-12


@pytest.mark.parametrize("parent", [[-1, 0, 0], [-1, 0, 0, 1], [-1, 0, 0, 0]])
def test_dense_tree_iid_siblings_exact_law_equals_target(parent):
    """SpecInfer's multi-step form on trees: siblings drawn i.i.d. from the parent's draft
    row, residual carried across siblings."""
    V, T = 3, 1.0
    model = E.SyntheticLM(V, seed=21, scale=1.4)
    draft = E.SyntheticLM(V, seed=22, scale=1.4)
    law = E.dense_tree_mixture(model, draft, parent, T)
    depth = max(len(p) for p in E.prefixes([0] * len(parent), parent))
    ext = E.extend(law, model, T, depth + 1)
    assert E.max_abs_diff(ext, E.target_joint(model, T, depth + 1)) < 1e-12


def test_greedy_limit_is_argmax_path():
    """With a vanishing temperature the exact law collapses onto the greedy output."""
    parent, tokens = TREES[0]
    model = E.SyntheticLM(4, seed=3, scale=2.0)
    law = E.verify_point_dist(model, tokens, parent, 1e-3)
    rows = E.tree_rows(model, tokens, parent)
    g = O.default().verify_greedy(rows[None], np.array([tokens]), np.array([parent]))
    L = int(g["accept_len"][0])
    seq = tuple(int(x) for x in g["out_tokens"][0, :L + 1])
    assert law[seq] > 1 - 1e-12


# ---- the C oracle, driven by uniforms ---------------------------------------------------------

def _sequences(res):
    L = res["accept_len"]
    toks = res["out_tokens"]
    return [tuple(int(x) for x in toks[i, :L[i] + 1]) for i in range(len(L))]


def _chi2_pvalue(samples, law):
    keys = sorted(set(law) | set(samples))
    n = len(samples)
    counts = {}
    for s in samples:
        counts[s] = counts.get(s, 0) + 1
    obs, exp = [], []
    rest_o, rest_e = 0.0, 0.0
    for k in keys:
        e = law.get(k, 0.0) * n
        o = counts.get(k, 0)
        if e == 0.0:
            assert o == 0, f"sequence {k} has zero probability but was drawn {o} times"
            continue
        if e < 5:
            rest_o += o
            rest_e += e
        else:
            obs.append(o)
            exp.append(e)
    if rest_e > 0:
        obs.append(rest_o)
        exp.append(rest_e)
    exp = np.array(exp)
    exp *= n / exp.sum()
    return stats.chisquare(np.array(obs, float), exp).pvalue


NDRAW = 200_000


@pytest.mark.parametrize("case", [0, 1, 3, 4])
def test_c_oracle_point_mass_matches_exact_law(orc, case):
    parent, tokens = TREES[case]
    V = 4 if case != 1 else 5
    T = 0.9
    model = E.SyntheticLM(V, seed=100 + case, scale=1.3)
    rows = E.tree_rows(model, tokens, parent)
    N = len(parent)
    rng = np.random.default_rng(555 + case)
    logits = np.broadcast_to(rows, (NDRAW, N, V)).copy()
    u = rng.random((NDRAW, N + 1), dtype=np.float32)
    res = orc.verify_sample(logits, np.tile(tokens, (NDRAW, 1)), np.tile(parent, (NDRAW, 1)),
                            T, u, nthreads=8)
    assert (res["status"] == 0).all()
    law = E.verify_point_dist(model, tokens, parent, T)
    assert _chi2_pvalue(_sequences(res), law) > 1e-5


def _dense_chain_batch(model, draft, k, V, T, n, rng):
    parent = [-1] + list(range(k))
    chains = list(itertools.product(range(V), repeat=k))
    weights = []
    for xs in chains:
        w, pre = 1.0, ()
        for x in xs:
            w *= draft.probs(pre, T)[x]
            pre = pre + (x,)
        weights.append(w)
    weights = np.array(weights) / sum(weights)
    pick = rng.choice(len(chains), size=n, p=weights)
    rows = np.stack([E.tree_rows(model, (0,) + xs, parent) for xs in chains])
    drows = np.stack([E.tree_rows(draft, (0,) + xs, parent) for xs in chains])
    toks = np.array([(0,) + xs for xs in chains], np.int32)
    return (rows[pick], drows[pick], toks[pick], np.tile(parent, (n, 1)).astype(np.int32))


@pytest.mark.parametrize("k,V,T", [(2, 4, 1.0), (3, 3, 0.7)])
def test_c_oracle_dense_chain_matches_exact_law(orc, k, V, T):
    model = E.SyntheticLM(V, seed=31, scale=1.5)
    draft = E.SyntheticLM(V, seed=32, scale=1.5)
    rng = np.random.default_rng(77)
    logits, dlogits, toks, par = _dense_chain_batch(model, draft, k, V, T, NDRAW, rng)
    u = rng.random((NDRAW, k + 2), dtype=np.float32)
    res = orc.verify_sample(logits, toks, par, T, u, draft=dlogits, draft_kind=O.DRAFT_LOGITS,
                            nthreads=8)
    assert (res["status"] == 0).all()
    law = E.dense_chain_mixture(model, draft, k, T)
    assert _chi2_pvalue(_sequences(res), law) > 1e-5


def test_c_oracle_dense_tree_matches_exact_law(orc):
    parent = [-1, 0, 0, 1]
    V, T, n = 3, 1.0, NDRAW
    model = E.SyntheticLM(V, seed=41, scale=1.4)
    draft = E.SyntheticLM(V, seed=42, scale=1.4)
    rng = np.random.default_rng(99)
    assigns = list(itertools.product(range(V), repeat=len(parent) - 1))
    weights, rows, drows = [], [], []
    for xs in assigns:
        tokens = (0,) + xs
        pre = E.prefixes(tokens, parent)
        w = 1.0
        for i in range(1, len(parent)):
            w *= draft.probs(pre[parent[i]], T)[tokens[i]]
        weights.append(w)
        rows.append(E.tree_rows(model, tokens, parent))
        drows.append(E.tree_rows(draft, tokens, parent))
    weights = np.array(weights) / sum(weights)
    pick = rng.choice(len(assigns), size=n, p=weights)
    toks = np.array([(0,) + xs for xs in assigns], np.int32)[pick]
    u = rng.random((n, len(parent) + 1), dtype=np.float32)
    res = orc.verify_sample(np.stack(rows)[pick], toks, np.tile(parent, (n, 1)), T, u,
                            draft=np.stack(drows)[pick], draft_kind=O.DRAFT_LOGITS, nthreads=8)
    law = E.dense_tree_mixture(model, draft, parent, T)
    assert _chi2_pvalue(_sequences(res), law) > 1e-5
