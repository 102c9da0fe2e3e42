"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case copies ``oracle/oracle.c``, plants one plausible mistake by text substitution (a
wrong comparison, a dropped term, a wrong index, a swapped operand), compiles the copy and runs
a battery built from the same pins as the other oracle tests: the hand-worked goldens, exact
and Monte-Carlo losslessness, the two-token closed form, a hand-worked inverse-CDF draw window
and the graph-ancestor mask check. The
battery must fail for every mutant and pass for the unmodified source.
"""
import itertools
import math
import os

import networkx as nx
import numpy as np
import pytest

import golden_io
from oracle import enumerate as E
from oracle import oracle as O
from test_oracle_golden import run_oracle

MUTANTS = {
    "accept_not_strict": ("if (uc < rhat)", "if (uc <= rhat)"),
    "no_renormalisation": ("rhat = p[t] / S;", "rhat = p[t];"),
    "argmax_last_tie": ("if (z > best) {", "if (z >= best) {"),
    "bonus_keeps_rejected": ("r[v] = inR[v] ? 0.0 : p[v];", "r[v] = p[v];"),
    "residual_sign": ("double d = r[v] - q[v];", "double d = q[v] - r[v];"),
    "cdf_not_strict": ("if (C > tau) {", "if (C >= tau) {"),
    "uniform_index": ("double uc = (double)u[c];", "double uc = (double)u[c - 1];"),
    "kv_commit_drops_root": ("o.kv_commit[(size_t)b * N + j + 1] = path[j];",
                             "o.kv_commit[(size_t)b * N + j] = path[j];"),
    "mask_without_self": ("m |= (uint64_t)1 << j;", "if (j != i) m |= (uint64_t)1 << j;"),
    "depth_off_by_one": ("int d = -1;", "int d = 0;"),
    "dense_accept_against_p": ("if (lhs < r[x]) {", "if (lhs < p[x]) {"),
    "temperature_dropped": ("p[v] = exp((elem(row, dtype, v) - m) / T);",
                            "p[v] = exp((elem(row, dtype, v) - m));"),
    "bonus_uniform_slot": ("for (int64_t v = 0; v < V; v++) r[v] = inR[v] ? 0.0 : p[v];\n    double cm;\n    int64_t alt, win[2];\n    int64_t bonus = inv_cdf(r, V, (double)u[N], &cm, &alt, win);",
                           "for (int64_t v = 0; v < V; v++) r[v] = inR[v] ? 0.0 : p[v];\n    double cm;\n    int64_t alt, win[2];\n    int64_t bonus = inv_cdf(r, V, (double)u[N - 1], &cm, &alt, win);"),
    "draft_row_of_child": ("draft_row(draft, draft_kind, draft_dtype, grow, V, T, q)",
                           "draft_row(draft, draft_kind, draft_dtype, grow + 1, V, T, q)"),
    "greedy_ignores_token": ("if (par[c] == node && tok[c] == a) {", "if (par[c] == node) {"),
    "window_low_end_at_tau": ("if (win[0] < 0 && C > tau - delta) win[0] = v;",
                              "if (win[0] < 0 && C > tau) win[0] = v;"),
    "window_high_end_at_tau": ("if (Cprev >= tau + delta) break;", "if (Cprev >= tau) break;"),
}


def _battery(orc) -> list:
    """Returns the names of the pins that fail."""
    failed = []
    for name in golden_io.names():
        g = golden_io.load(name)
        try:
            if golden_io.mismatches(g, run_oracle(orc, g)):
                failed.append("golden:" + name)
        except Exception:
            failed.append("golden-error:" + name)
    # Monte-Carlo losslessness, point-mass trie with a duplicate-free root of 3 children
    from test_oracle_lossless import _chi2_pvalue, _sequences
    parent, tokens, V, T, n = [-1, 0, 0, 0, 1, 2], [0, 2, 0, 3, 1, 1], 5, 0.9, 50_000
    model = E.SyntheticLM(V, seed=101, scale=1.3)
    rows = E.tree_rows(model, tokens, parent)
    rng = np.random.default_rng(9)
    res = orc.verify_sample(np.broadcast_to(rows, (n, 6, V)).copy(), np.tile(tokens, (n, 1)),
                            np.tile(parent, (n, 1)), T,
                            rng.random((n, 7), dtype=np.float32), nthreads=8)
    try:
        if _chi2_pvalue(_sequences(res), E.verify_point_dist(model, tokens, parent, T)) < 1e-5:
            failed.append("mc:point")
    except AssertionError:
        failed.append("mc:point-impossible")
    # Monte-Carlo losslessness, dense tree with i.i.d. siblings
    parent, V, T = [-1, 0, 0, 1], 3, 1.0
    model, draft = E.SyntheticLM(V, seed=41, scale=1.4), E.SyntheticLM(V, seed=42, scale=1.4)
    assigns = list(itertools.product(range(V), repeat=3))
    w, rows, drows = [], [], []
    for xs in assigns:
        toks = (0,) + xs
        pre = E.prefixes(toks, parent)
        pw = 1.0
        for i in range(1, 4):
            pw *= draft.probs(pre[parent[i]], T)[toks[i]]
        w.append(pw)
        rows.append(E.tree_rows(model, toks, parent))
        drows.append(E.tree_rows(draft, toks, parent))
    pick = rng.choice(len(assigns), size=n, p=np.array(w) / sum(w))
    toks = np.array([(0,) + xs for xs in assigns], np.int32)[pick]
    res = orc.verify_sample(np.stack(rows)[pick], toks, np.tile(parent, (n, 1)), T,
                            rng.random((n, 5), dtype=np.float32), draft=np.stack(drows)[pick],
                            draft_kind=O.DRAFT_LOGITS, nthreads=8)
    try:
        if _chi2_pvalue(_sequences(res), E.dense_tree_mixture(model, draft, parent, T)) < 1e-5:
            failed.append("mc:dense-tree")
    except AssertionError:
        failed.append("mc:dense-impossible")
    # V = 2 closed form at T = 0.5
    z = np.array([0.7, -0.4], np.float32)
    p0 = 1.0 / (1.0 + math.exp(-(0.7 - (-0.4)) / 0.5))
    for u1, want in [(p0 * 0.999, 1), (p0 * 1.001, 0)]:
        r = orc.verify_sample(np.stack([z, z])[None], np.array([[0, 0]], np.int32),
                              np.array([[-1, 0]], np.int32), 0.5,
                              np.array([[0.0, u1, 0.3]], np.float32))
        if r["accept_len"][0] != want:
            failed.append("closed-form")
    # the draw window of a hand-worked inverse CDF (tokens 1 and 2 have tiny mass)
    _, _, win = orc.inv_cdf(np.array([0.5, 1e-9, 2e-9, 0.5 - 3e-9]), 0.5 + 5e-10, window=True)
    if win != (0, 3):
        failed.append("window")
    # mask against graph ancestors
    par = np.array([[-1, 0, 0, 1, 3, 2, 5, 5]], np.int32)
    anc, depth, _ = orc.build_mask(par)
    g = nx.DiGraph([(int(par[0, i]), i) for i in range(1, 8)])
    for i in range(8):
        want = {i} | nx.ancestors(g, i)
        if {j for j in range(8) if (int(anc[0, i]) >> j) & 1} != want or \
                depth[0, i] != len(want) - 1:
            failed.append("mask")
            break
    return failed


def _build_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    with open(O.SOURCE) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation site of {name} not found in oracle.c"
    src = src.replace(old, new)
    path = tmp_path / f"{name}.c"
    path.write_text(src)
    return O.Oracle(O.compile_oracle(str(path), str(tmp_path / f"lib{name}.so"), force=True))


def test_battery_passes_on_the_oracle(orc):
    assert _battery(orc) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    mutant = _build_mutant(tmp_path, name)
    assert _battery(mutant), f"no pin catches the planted mistake {name}"
