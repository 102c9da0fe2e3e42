"""Invariants, closed forms and library special cases that pin the oracle (CPU only)."""
import math

import networkx as nx
import numpy as np
import pytest
from scipy import special

from oracle import oracle as O
from speculative_decoding_tree_mask_gb300 import workloads as W


def _small(name, **kw):
    return W.WORKLOADS[name].scaled(**kw)


def _path_ok(parent, kv, L):
    if kv[0] != 0:
        return False
    return all(parent[kv[j + 1]] == kv[j] for j in range(L))


# ---- tree mask ----------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
def test_mask_matches_graph_ancestors(orc, seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 65))
    parent = np.stack([W.random_trie(rng, N, 10, 6) for _ in range(4)])
    anc, depth, status = orc.build_mask(parent)
    assert (status == 0).all()
    for b in range(parent.shape[0]):
        g = nx.DiGraph()
        g.add_nodes_from(range(N))
        g.add_edges_from((int(parent[b, i]), i) for i in range(1, N))
        for i in range(N):
            want = {i} | nx.ancestors(g, i)
            got = {j for j in range(N) if (int(anc[b, i]) >> j) & 1}
            assert got == want
            assert depth[b, i] == nx.shortest_path_length(g, 0, i)
            assert bin(int(anc[b, i])).count("1") == depth[b, i] + 1
            if i:
                p = parent[b, i]
                assert int(anc[b, p]) & ~int(anc[b, i]) == 0


def test_mask_full_width_chain(orc):
    anc, depth, status = orc.build_mask(W.chain(64)[None])
    assert status[0] == 0
    assert [int(a) for a in anc[0]] == [(1 << (i + 1)) - 1 for i in range(64)]
    assert depth[0].tolist() == list(range(64))


# ---- greedy --------------------------------------------------------------------------------

def _brute_greedy(logits, parent, tok):
    """Longest root path whose every edge token equals the parent row's first argmax
    (numpy's argmax returns the first maximum)."""
    N = len(parent)
    am = logits.astype(np.float64).argmax(axis=-1)
    best = 0
    for i in range(N):
        j, ok, d = i, True, 0
        while j != 0:
            if tok[j] != am[parent[j]]:
                ok = False
                break
            j = parent[j]
            d += 1
        if ok and d > best:
            best, node = d, i
    return best


@pytest.mark.parametrize("boost", [0.0, 6.0, 40.0])
def test_greedy_equals_longest_argmax_path(orc, boost):
    w = _small("greedy_trie", B=24, V=97, dtype="f32", boost=boost, seed=5)
    x = W.make(w)
    logits = W.host_logits(x["logits"])
    res = orc.verify_greedy(logits, x["tok_np"], x["parent_np"])
    _, depth, _ = orc.build_mask(x["parent_np"])
    for b in range(w.B):
        par, tok = x["parent_np"][b], x["tok_np"][b]
        L = int(res["accept_len"][b])
        assert res["status"][b] == 0
        assert L == _brute_greedy(logits[b], par, tok)
        assert L <= depth[b].max()
        kv = res["kv_commit"][b]
        assert _path_ok(par, kv, L)
        assert (res["out_tokens"][b, :L] == tok[kv[1:L + 1]]).all()
        stop = kv[L]
        kids = [c for c in range(w.N) if par[c] == stop]
        assert res["bonus"][b] not in [tok[c] for c in kids]
        assert res["bonus"][b] == np.argmax(logits[b, stop].astype(np.float64))
        assert res["out_tokens"][b, L] == res["bonus"][b]
        assert (res["out_tokens"][b, L + 1:] == -1).all()
        assert (res["kv_commit"][b, L + 1:] == -1).all()
    if boost == 40.0:
        assert res["accept_len"].max() >= 3   # the walk goes deep somewhere


def test_greedy_planted_ties_take_lowest_index(orc):
    rng = np.random.default_rng(1)
    B, N, V = 16, 3, 50
    logits = rng.standard_normal((B, N, V)).astype(np.float32)
    parent = np.tile(W.chain(N), (B, 1))
    tok = np.zeros((B, N), np.int32)
    for b in range(B):
        for i in range(N):
            idx = np.sort(rng.choice(V, size=3, replace=False))
            logits[b, i, idx] = 10.0
        tok[b, 1] = np.flatnonzero(logits[b, 0] == 10.0)[0]
        tok[b, 2] = np.flatnonzero(logits[b, 1] == 10.0)[1]   # second tie: never accepted
    res = orc.verify_greedy(logits, tok, parent)
    assert (res["accept_len"] == 1).all()
    assert (res["bonus"] == [np.flatnonzero(logits[b, 1] == 10.0)[0] for b in range(B)]).all()


def test_greedy_bf16_equals_f32_on_same_values(orc):
    import torch
    w = _small("greedy_trie", B=6, V=300, boost=20.0, seed=9)
    x = W.make(w)
    r16 = orc.verify_greedy(W.host_logits(x["logits"]), x["tok_np"], x["parent_np"])
    r32 = orc.verify_greedy(x["logits"].to(torch.float32).numpy(), x["tok_np"], x["parent_np"])
    for k in r16:
        assert np.array_equal(r16[k], r32[k])


# ---- rows ------------------------------------------------------------------------------------

@pytest.mark.parametrize("T", [0.3, 1.0, 2.5])
def test_row_softmax_matches_library(orc, T):
    rng = np.random.default_rng(2)
    row = (rng.standard_normal(3001) * 3).astype(np.float32)
    p = orc.row_softmax(row, T)
    ref = special.softmax(row.astype(np.float64) / T)
    assert np.allclose(p, ref, rtol=1e-12, atol=0)
    m, S, a, bad = orc.row_stats(row, T)
    assert m == row.max() and a == int(np.argmax(row)) and bad == 0
    assert math.isclose(math.log(S) + m / T, special.logsumexp(row.astype(np.float64) / T),
                        rel_tol=1e-12)


def test_row_stats_bad_rows(orc):
    assert orc.row_stats(np.array([0, np.nan, 1], np.float32), 1.0)[3] == 1
    assert orc.row_stats(np.array([0, np.inf, 1], np.float32), 1.0)[3] == 1
    assert orc.row_stats(np.full(4, -np.inf, np.float32), 1.0)[3] == 1
    assert orc.row_stats(np.array([-np.inf, 0.0, -np.inf], np.float32), 1.0)[3] == 0


def test_inv_cdf_is_searchsorted(orc):
    rng = np.random.default_rng(3)
    for _ in range(200):
        V = int(rng.integers(1, 40))
        r = rng.random(V) * (rng.random(V) < 0.7)
        if r.sum() == 0:
            r[rng.integers(V)] = 1.0
        u = float(rng.random())
        v, margin = orc.inv_cdf(r, u)
        c = np.cumsum(r)      # sequential running sums, the order the oracle adds in
        tau = u * c[-1]
        assert v == int(np.searchsorted(c, tau, side="right"))
        assert r[v] > 0
        assert margin >= 0


def test_inv_cdf_fallback_and_zero_mass_entries(orc):
    v, m = orc.inv_cdf(np.array([0.0, 0.5, 0.0, 0.5, 0.0]), np.nextafter(1.0, 0.0))
    assert v == 3
    v, m = orc.inv_cdf(np.array([0.0, 0.0, 1.0]), 0.0)
    assert v == 2


# ---- sampling special cases -----------------------------------------------------------------

def test_small_temperature_sampling_equals_greedy(orc):
    rng = np.random.default_rng(4)
    B, N, V = 64, 12, 40
    # well separated logits: distinct multiples of 0.5
    logits = np.stack([np.stack([rng.permutation(V) * 0.5 for _ in range(N)])
                       for _ in range(B)]).astype(np.float32)
    parent = np.stack([W.random_trie(rng, N, 4, 3) for _ in range(B)])
    tok = np.stack([W.child_tokens(rng, parent[b], V) for b in range(B)])
    am = logits.argmax(-1)
    for b in range(B):       # make some paths acceptable
        for c in range(1, N):
            if rng.random() < 0.6:
                sib = [s for s in range(1, N) if parent[b, s] == parent[b, c] and s != c]
                if all(tok[b, s] != am[b, parent[b, c]] for s in sib):
                    tok[b, c] = am[b, parent[b, c]]
    u = rng.uniform(0.001, 0.999, (B, N + 1)).astype(np.float32)
    g = orc.verify_greedy(logits, tok, parent)
    s = orc.verify_sample(logits, tok, parent, 1e-3, u)
    for k in ("accept_len", "out_tokens", "kv_commit", "bonus", "status"):
        assert np.array_equal(g[k], s[k]), k
    assert g["accept_len"].max() >= 2


def test_temperature_zero_is_greedy(orc):
    w = _small("sampling_trie", B=8, V=200, dtype="f32", boost=30.0, seed=12)
    x = W.make(w)
    logits = W.host_logits(x["logits"])
    g = orc.verify_greedy(logits, x["tok_np"], x["parent_np"])
    s = orc.verify_sample(logits, x["tok_np"], x["parent_np"], 0.0, x["uniforms"].numpy())
    for k in ("accept_len", "out_tokens", "kv_commit", "bonus", "status"):
        assert np.array_equal(g[k], s[k])


def test_dense_draft_equal_to_target_accepts_everything(orc):
    w = _small("dense_chain", B=16, V=64, dtype="f32", seed=13)
    x = W.make(w)
    logits = W.host_logits(x["logits"])
    u = np.minimum(x["uniforms"].numpy(), np.float32(0.999999))
    res = orc.verify_sample(logits, x["tok_np"], x["parent_np"], 1.0, u, draft=logits,
                            draft_kind=O.DRAFT_LOGITS)
    assert (res["accept_len"] == w.N - 1).all()


def test_zero_and_one_probability_children(orc):
    V = 6
    logits = np.zeros((2, 2, V), np.float32)
    logits[0, 0, 3] = -np.inf                   # p(3) = 0
    logits[1, 0, :] = -np.inf
    logits[1, 0, 4] = 0.0                       # p(4) = 1
    parent = np.tile([-1, 0], (2, 1)).astype(np.int32)
    tok = np.array([[0, 3], [0, 4]], np.int32)
    for u1 in [0.0, 1e-7, 0.5, 0.9999999]:
        u = np.array([[0.0, u1, 0.5], [0.0, u1, 0.5]], np.float32)
        res = orc.verify_sample(logits, tok, parent, 1.0, u)
        assert res["accept_len"].tolist() == [0, 1]
        assert res["bonus"][0] != 3


@pytest.mark.parametrize("T", [0.5, 1.0, 3.0])
def test_two_token_closed_form(orc, T):
    """V = 2, one child with token 0: accepted iff u < sigmoid((z0 - z1)/T)."""
    rng = np.random.default_rng(5)
    for _ in range(50):
        z = (rng.standard_normal(2) * 2).astype(np.float32)
        p0 = 1.0 / (1.0 + math.exp(-(float(z[0]) - float(z[1])) / T))
        for u1, want in [(p0 * (1 - 1e-6), 1), (min(p0 * (1 + 1e-6), 0.9999999), 0)]:
            if not (0.0 <= np.float32(u1) < 1.0):
                continue
            u = np.array([[0.0, u1, 0.3]], np.float32)
            if abs(float(np.float32(u1)) - p0) < 1e-9:
                continue
            res = orc.verify_sample(np.stack([z, z])[None], np.array([[0, 0]], np.int32),
                                    np.array([[-1, 0]], np.int32), T, u)
            assert res["accept_len"][0] == want
            if want == 0:
                assert res["bonus"][0] == 1     # token 0 removed from the residual


def test_cdf_alt_is_the_token_across_the_nearer_boundary(orc):
    """Root only, V = 4 equal logits: p = 1/4 each, boundaries at 1/4, 1/2, 3/4."""
    logits = np.zeros((3, 1, 4), np.float32)
    tok = np.zeros((3, 1), np.int32)
    par = np.full((3, 1), -1, np.int32)
    u = np.array([[0.0, np.float32(0.5) + np.float32(6e-8)],      # just above 1/2: token 2, alt 1
                  [0.0, np.float32(0.75) - np.float32(6e-8)],     # just below 3/4: token 2, alt 3
                  [0.0, 0.6]], np.float32)                        # mid-interval: alt 2 only if
    r = orc.verify_sample(logits, tok, par, 1.0, u)               # it is the nearer side
    assert r["bonus"].tolist() == [2, 2, 2]
    assert r["cdf_alt"][:2].tolist() == [1, 3]
    assert (r["cdf_margin"][:2] < 1e-6).all() and r["cdf_margin"][2] > 1e-2


def test_cdf_window_spans_tokens_within_the_tolerance(orc):
    """The draw window: tokens with mass whose CDF interval comes within 1e-6 * S of tau.
    r = (0.5, 1e-9, 2e-9, 0.5 - 3e-9), S = 1: tau = 0.5 + 5e-10 lies inside token 1's
    interval [0.5, 0.5 + 1e-9), and every interval touches (tau - 1e-6, tau + 1e-6), so the
    window is tokens 0..3; tau = 0.25 is deep inside token 0 (window 0..0); with a zero-mass
    token between two halves, tau = 0.5 - 1e-7 gives 0..2 (token 1 has no mass but lies
    inside, tokens 0 and 2 are the ends)."""
    v, m, win = orc.inv_cdf(np.array([0.5, 1e-9, 2e-9, 0.5 - 3e-9]), 0.5 + 5e-10, window=True)
    assert v == 1 and m < 1e-9 and win == (0, 3)
    v, m, win = orc.inv_cdf(np.array([0.5, 1e-9, 2e-9, 0.5 - 3e-9]), 0.25, window=True)
    assert v == 0 and win == (0, 0)
    v, m, win = orc.inv_cdf(np.array([0.5, 0.0, 0.5]), 0.5 - 1e-7, window=True)
    assert v == 0 and win == (0, 2)
    v, m, win = orc.inv_cdf(np.array([0.25, 0.25, 0.25, 0.25]), 0.6, window=True)
    assert v == 2 and win == (2, 2)
    # brute force on random rows: the window is exactly the tokens with mass whose interval
    # meets [tau - 1e-6 S, tau + 1e-6 S)
    rng = np.random.default_rng(5)
    for _ in range(200):
        r = rng.random(12) ** 8 * (rng.random(12) < 0.8)
        u = rng.random()
        v, m, win = orc.inv_cdf(r, u, window=True)
        S = r.sum()
        C = np.cumsum(r)
        lo, hi = u * S - 1e-6 * S, u * S + 1e-6 * S
        want = [w for w in range(12) if r[w] > 0 and C[w] > lo and C[w] - r[w] < hi]
        assert win == (min(want + [v]), max(want + [v])), (r, u, win, want)
