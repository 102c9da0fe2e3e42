"""Pins of the node-budget oracle and the adaptive budget controller (CPU only).

The controller is a reading of IluvatarLabs/vllm PR #3's adaptive mode (the page states the
goal, a target acceptance ratio held by changing the number of speculative tokens, and no
formula), so the pins are what that reading fixes: the moving average's closed form, the
dead band, the limits, which requests count, the depth bound taken from the graph, and the
meaning of a truncated tree. Planted mistakes in a copy of the module must fail them.
"""
import math

import networkx as nx
import numpy as np
import pytest

from oracle import budget as BU
from speculative_decoding_tree_mask_gb300 import workloads as W


def _chains(B, k):
    return np.stack([W.chain(k + 1) for _ in range(B)])


# ---- depth bound ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(5))
def test_max_depth_matches_graph(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 65))
    par = W.random_trie(rng, N, 10, 6)
    g = nx.DiGraph([(int(par[i]), i) for i in range(1, N)])
    g.add_node(0)
    lengths = nx.single_source_shortest_path_length(g, 0)
    for n in range(1, N + 1):
        assert BU.max_depth(par, n) == max(lengths[i] for i in range(n))


def test_max_depth_rejects_bad_parents():
    assert BU.max_depth(np.array([-1, 0, 2]), 3) is None
    assert BU.max_depth(np.array([-1, 0, 2]), 2) == 1   # the bad node lies beyond the budget
    assert BU.max_depth(np.array([0, 0]), 1) is None


# ---- moving average and budget rule --------------------------------------------------------

def test_constant_ratio_closed_form():
    """Ratio 0.5 every step: ema_t = r + (ema_0 - r) (1 - alpha)^t."""
    prm = BU.Params(target=0.9, alpha=0.25, band=0.0, n_min=2, n_max=5)
    par = _chains(4, 4)
    acc = np.array([4, 2, 0, 2])
    st = BU.State(ema=1.0, budget=5)
    for t in range(1, 30):
        st = BU.update(prm, st, acc, np.zeros(4), par, np.full(4, 5))
        assert math.isclose(st.ema, 0.5 + 0.5 * 0.75 ** t, rel_tol=0, abs_tol=1e-14)
        assert st.steps == t
    assert st.budget == 2   # the average stays below the target: the budget falls to n_min


def test_budget_climbs_and_falls_within_limits():
    prm = BU.Params(target=0.6, alpha=1.0, band=0.1, n_min=3, n_max=9, step=2)
    par = _chains(2, 8)
    st = BU.State(ema=0.6, budget=4)
    seen = []
    for _ in range(5):   # everything accepted: ratio 1 > 0.7
        n = np.full(2, st.budget)
        st = BU.update(prm, st, n - 1, np.zeros(2), par, n)
        seen.append(st.budget)
    assert seen == [6, 8, 9, 9, 9]
    for _ in range(5):   # nothing accepted: ratio 0 < 0.5
        st = BU.update(prm, st, np.zeros(2), np.zeros(2), par, np.full(2, st.budget))
        seen.append(st.budget)
    assert seen[5:] == [7, 5, 3, 3, 3]


def test_dead_band_holds_the_budget():
    prm = BU.Params(target=0.5, alpha=1.0, band=0.2, n_min=1, n_max=9)
    par = _chains(1, 8)
    for acc, want in [(3, 5), (4, 5), (5, 5), (6, 6), (1, 4)]:   # ratios 3/8 .. 6/8, 1/8
        st = BU.update(prm, BU.State(ema=0.5, budget=5), np.array([acc]), np.zeros(1), par,
                       np.array([9]))
        assert st.budget == want, (acc, st)


def test_unusable_requests_do_not_count():
    prm = BU.Params(target=0.5, alpha=0.5, band=0.0, n_min=1, n_max=9)
    par = _chains(4, 8)
    acc = np.array([8, 0, 7, 1])
    status = np.array([0, 3, 0, 0])
    n_act = np.array([9, 9, 9, 0])   # request 3: budget outside [1, N]
    a = BU.update(prm, BU.State(0.5, 5), acc, status, par, n_act)
    b = BU.update(prm, BU.State(0.5, 5), acc[[0, 2]], status[[0, 2]], par[[0, 2]], n_act[[0, 2]])
    assert a == b
    assert a.ema == 0.5 * 0.5 + 0.5 * (15 / 16)


def test_no_depth_leaves_the_average():
    prm = BU.Params(target=0.5, alpha=0.5, band=0.0, n_min=2, n_max=4)
    st = BU.update(prm, BU.State(0.3, 7, steps=4), np.zeros(3), np.zeros(3), _chains(3, 5),
                   np.ones(3))   # budget 1: the root alone, nothing could be accepted
    assert st == BU.State(0.3, 4, 4)   # only the clamp to [n_min, n_max] applies


def test_depth_counts_only_the_budgeted_prefix():
    prm = BU.Params(target=0.5, alpha=1.0, band=0.0, n_min=1, n_max=9)
    par = np.array([[-1, 0, 0, 1, 3, 4]])   # depths 0 1 1 2 3 4
    for n, D in [(3, 1), (4, 2), (6, 4)]:
        st = BU.update(prm, BU.State(0.5, 5), np.array([1]), np.zeros(1), par, np.array([n]))
        assert st.ema == 1 / D


# ---- truncated trees -----------------------------------------------------------------------

def test_truncation_keeps_the_bonus_slot(orc):
    """Budget 1 keeps the root alone: the bonus is drawn from the root row with the uniform in
    slot N. p = softmax([0, ln 2, ln 3]) = (1/6, 2/6, 3/6): u = 0.9 -> token 2, u = 0.1 -> 0."""
    z = np.array([0.0, math.log(2.0), math.log(3.0)], np.float32)
    logits = np.stack([z, z, z])[None]
    tok, par = np.array([[0, 1, 2]], np.int32), np.array([[-1, 0, 0]], np.int32)
    u = np.array([[0.0, 0.1, 0.1, 0.9]], np.float32)
    lg, tk, pr, uu, _ = BU.truncate(logits[0], tok[0], par[0], u[0], 1)
    r = orc.verify_sample(lg[None], tk[None], pr[None], 1.0, uu[None])
    assert r["accept_len"][0] == 0 and r["bonus"][0] == 2
    assert uu.tolist() == pytest.approx([0.0, 0.9])


@pytest.mark.parametrize("seed", range(4))
def test_greedy_budget_covering_the_path_changes_nothing(orc, seed):
    """The greedy walk takes the first matching child in node order, so a budget larger than
    every node on the full tree's accepted path reproduces the full result, and a budget that
    cuts the path stops the walk at the last kept path node."""
    w = W.WORKLOADS["greedy_trie"].scaled(V=512, B=6)
    par, tok = W.make_trees(w, seed=seed)
    logits = W.host_logits(W.make_logits(w, par, tok, seed=seed))
    full = orc.verify_greedy(logits, tok, par)
    for b in range(w.B):
        L = int(full["accept_len"][b])
        path = [int(x) for x in full["kv_commit"][b, 1:L + 1]]
        for n in range(1, w.N + 1):
            lg, tk, pr, _, _ = BU.truncate(logits[b], tok[b], par[b], None, n)
            r = orc.verify_greedy(lg[None], tk[None], pr[None])
            kept = [x for x in path if x < n]
            if len(kept) == L:
                assert r["accept_len"][0] == L and r["bonus"][0] == full["bonus"][b]
            else:
                cut = next(j for j, x in enumerate(path) if x >= n)
                assert r["accept_len"][0] == cut
                assert list(r["kv_commit"][0, 1:cut + 1]) == path[:cut]


# ---- planted mistakes ----------------------------------------------------------------------

MUTANTS = {
    "alpha_swapped": ("ema = (1.0 - params.alpha) * ema + params.alpha * ratio",
                      "ema = params.alpha * ema + (1.0 - params.alpha) * ratio"),
    "band_sign": ("if ema > params.target + params.band:", "if ema > params.target - params.band:"),
    "depth_of_full_tree": ("dm = max_depth(parent[b], n)", "dm = max_depth(parent[b], N)"),
    "status_ignored": ("if int(status[b]) != 0:", "if False:"),
    "depth_off_by_one": ("d, node = 0, i", "d, node = 1, i"),
    "bonus_slot_moves": ("uniforms[N:N + 1]", "uniforms[n:n + 1]"),
    "no_clamp": ("k = min(max(int(state.budget), params.n_min), params.n_max)",
                 "k = int(state.budget)"),
    "steps_not_counted": ("        steps += 1\n", ""),
}


def _mutant_module(name):
    import sys
    import types
    old, new = MUTANTS[name]
    src = open(BU.__file__).read()
    assert src.count(old) == 1, name
    mod = types.ModuleType("budget_" + name)
    sys.modules[mod.__name__] = mod   # dataclasses look their module up while decorating
    try:
        exec(compile(src.replace(old, new), BU.__file__, "exec"), mod.__dict__)
    finally:
        del sys.modules[mod.__name__]
    return mod


PINS = [test_max_depth_matches_graph, test_constant_ratio_closed_form,
        test_budget_climbs_and_falls_within_limits, test_dead_band_holds_the_budget,
        test_unusable_requests_do_not_count, test_no_depth_leaves_the_average,
        test_depth_counts_only_the_budgeted_prefix, test_truncation_keeps_the_bonus_slot]


def _battery(orc):
    failed = []
    for pin in PINS:
        try:
            if pin is test_max_depth_matches_graph:
                pin(0)
            elif pin is test_truncation_keeps_the_bonus_slot:
                pin(orc)
            else:
                pin()
        except Exception:
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(orc, monkeypatch, name):
    monkeypatch.setitem(globals(), "BU", _mutant_module(name))
    assert _battery(orc), f"no pin catches the planted mistake {name}"


def test_battery_passes_on_the_oracle(orc):
    assert _battery(orc) == []
