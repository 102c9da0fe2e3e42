"""Node budgets and the adaptive budget controller on the GPU, through the C ABI.

A request verified under budget n must give the oracle's result on its truncated tree (nodes
0..n-1, bonus uniform still in slot N), for every verify entry point; rows beyond the budget
are never read; a bad budget is refused per request; the device controller reproduces the
oracle controller's float64 state bit for bit; and a captured graph of verify + update
follows the budget from step to step (IluvatarLabs/vllm PR #3, adaptive mode under CUDA
graphs).
"""
import numpy as np
import pytest
import torch

import parity as PY
from oracle import budget as BU
from speculative_decoding_tree_mask_gb300 import binding as G
from speculative_decoding_tree_mask_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
KEYS = PY.KEYS


@pytest.fixture(scope="module")
def h():
    G.load()
    with G.Handle(256, 64, 1 << 21, 0) as handle:
        yield handle


@pytest.fixture(autouse=True)
def _no_budget_after(h):
    yield
    G.spec_set_node_budget(h, None)


def _budgets(rng, B, N):
    n = rng.integers(1, N + 1, size=B)
    n[0], n[-1] = 1, N
    return n.astype(np.int32)


def _pad(a, N, fill=-1):
    out = np.full((a.shape[0], N), fill, a.dtype)
    out[:, :a.shape[1]] = a
    return out


def oracle_budgeted(orc, x, n_active, mode, T=None, kind=G.SPEC_DRAFT_POINT):
    """The oracle on each request's truncated tree, assembled into [B, N] outputs."""
    logits = W.host_logits(x["logits"])
    draft = W.host_logits(x["draft"]) if "draft" in x else None
    tok, par = x["draft_token"].cpu().numpy(), x["parent"].cpu().numpy()
    u = x["uniforms"].cpu().numpy()
    B, N = par.shape
    res = {k: [] for k in KEYS + ("decision_margin", "cdf_margin", "cdf_alt", "cdf_lo",
                                  "cdf_hi")}
    for b in range(B):
        lg, tk, pr, uu, dr = BU.truncate(logits[b], tok[b], par[b], u[b], int(n_active[b]),
                                         None if draft is None else draft[b])
        if mode == "greedy":
            r = orc.verify_greedy(lg[None], tk[None], pr[None])
        else:
            r = orc.verify_sample(lg[None], tk[None], pr[None], T, uu[None],
                                  draft=None if dr is None else dr[None],
                                  draft_kind=PY.ORACLE_KIND[kind])
        for k in res:
            if k in r:
                v = r[k]
                res[k].append(_pad(v, N)[0] if k in ("out_tokens", "kv_commit") else v[0])
    return {k: np.stack(v) for k, v in res.items() if v}


def _set(h, n_active):
    t = torch.as_tensor(n_active, dtype=torch.int32).to(DEV)
    G.spec_set_node_budget(h, t)
    return t


def _run(fn, *a, **kw):
    out = fn(*a, **kw)
    torch.cuda.synchronize()
    return PY.to_np(out)


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("lazy", [False, True])
def test_greedy_under_budget(h, orc, seed, lazy):
    w = W.WORKLOADS["greedy_trie"].scaled(B=12, V=30011)
    x = W.make(w, device=DEV, seed=seed)
    n_active = _budgets(np.random.default_rng(seed), w.B, w.N)
    _set(h, n_active)
    fn = G.verify_greedy_lazy if lazy else G.verify_greedy
    got = _run(fn, h, x["logits"], x["draft_token"], x["parent"])
    ref = oracle_budgeted(orc, x, n_active, "greedy")
    PY.assert_exact(got, ref)


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("lazy", [False, True])
def test_point_sampling_under_budget(h, orc, seed, lazy):
    w = W.WORKLOADS["sampling_trie"].scaled(B=16, V=40000)
    x = W.make(w, device=DEV, seed=seed)
    n_active = _budgets(np.random.default_rng(100 + seed), w.B, w.N)
    _set(h, n_active)
    fn = G.verify_sample_lazy if lazy else G.verify_sample
    got = _run(fn, h, x["logits"], x["draft_token"], x["parent"], w.temperature, x["uniforms"])
    ref = oracle_budgeted(orc, x, n_active, "sample", T=w.temperature)
    PY.compare_sample(got, ref)


@pytest.mark.parametrize("lazy", [False, True])
def test_dense_chain_under_budget(h, orc, lazy):
    w = W.WORKLOADS["dense_chain"].scaled(B=16, V=20000)
    x = W.make(w, device=DEV, seed=5)
    n_active = _budgets(np.random.default_rng(7), w.B, w.N)
    _set(h, n_active)
    fn = G.verify_sample_lazy if lazy else G.verify_sample
    got = _run(fn, h, x["logits"], x["draft_token"], x["parent"], w.temperature, x["uniforms"],
               draft=x["draft"], draft_kind=G.SPEC_DRAFT_LOGITS)
    ref = oracle_budgeted(orc, x, n_active, "sample", T=w.temperature, kind=G.SPEC_DRAFT_LOGITS)
    PY.compare_sample(got, ref)


@pytest.mark.parametrize("mode", ["greedy", "sample", "greedy_lazy", "sample_lazy"])
def test_rows_beyond_the_budget_are_not_read(h, orc, mode):
    """NaN in every row, token and uniform slot beyond the budget changes nothing."""
    w = W.WORKLOADS["sampling_trie"].scaled(B=8, V=12345)
    x = W.make(w, device=DEV, seed=11)
    n_active = _budgets(np.random.default_rng(11), w.B, w.N)
    ref_in = dict(x)
    poisoned = dict(x)
    poisoned["logits"] = x["logits"].clone()
    poisoned["draft_token"] = x["draft_token"].clone()
    poisoned["parent"] = x["parent"].clone()
    poisoned["uniforms"] = x["uniforms"].clone()
    for b, n in enumerate(n_active):
        poisoned["logits"][b, n:] = float("nan")
        poisoned["draft_token"][b, n:] = -7
        poisoned["parent"][b, n:] = 1000
        poisoned["uniforms"][b, n:w.N] = 5.0
    _set(h, n_active)
    greedy = mode.startswith("greedy")
    fn = {"greedy": G.verify_greedy, "sample": G.verify_sample,
          "greedy_lazy": G.verify_greedy_lazy, "sample_lazy": G.verify_sample_lazy}[mode]
    args = () if greedy else (w.temperature, poisoned["uniforms"])
    got = _run(fn, h, poisoned["logits"], poisoned["draft_token"], poisoned["parent"], *args)
    assert (got["status"] == 0).all()
    ref = oracle_budgeted(orc, ref_in, n_active, "greedy" if greedy else "sample",
                          T=w.temperature)
    if greedy:
        PY.assert_exact(got, ref)
    else:
        PY.compare_sample(got, ref)


def test_bad_budget_is_refused_per_request(h):
    w = W.WORKLOADS["sampling_trie"].scaled(B=6, V=5000)
    x = W.make(w, device=DEV, seed=2)
    n_active = np.array([0, w.N + 1, -5, 1, w.N, 3], np.int32)
    _set(h, n_active)
    for fn, args in [(G.verify_greedy, ()), (G.verify_greedy_lazy, ()),
                     (G.verify_sample, (w.temperature, x["uniforms"])),
                     (G.verify_sample_lazy, (w.temperature, x["uniforms"]))]:
        got = _run(fn, h, x["logits"], x["draft_token"], x["parent"], *args)
        assert got["status"][:3].tolist() == [G.SPEC_REQ_BAD_BUDGET] * 3
        assert (got["accept_len"][:3] == 0).all() and (got["bonus"][:3] == -1).all()
        assert (got["out_tokens"][:3] == -1).all() and (got["kv_commit"][:3] == -1).all()
        assert (got["status"][3:] == 0).all()


def test_clearing_the_budget_verifies_every_node(h):
    w = W.WORKLOADS["greedy_trie"].scaled(B=8, V=8000)
    x = W.make(w, device=DEV, seed=4)
    full = _run(G.verify_greedy, h, x["logits"], x["draft_token"], x["parent"])
    _set(h, np.full(w.B, 1, np.int32))
    root = _run(G.verify_greedy, h, x["logits"], x["draft_token"], x["parent"])
    assert (root["accept_len"] == 0).all()
    G.spec_set_node_budget(h, None)
    again = _run(G.verify_greedy, h, x["logits"], x["draft_token"], x["parent"])
    for k in KEYS:
        assert np.array_equal(full[k], again[k]), k
    _set(h, np.full(w.B, w.N, np.int32))
    same = _run(G.verify_greedy, h, x["logits"], x["draft_token"], x["parent"])
    for k in KEYS:
        assert np.array_equal(full[k], same[k]), k


# ---- controller ----------------------------------------------------------------------------

def _gpu_update(h, prm, state, acc, status, parent, n_active_t):
    G.spec_budget_update(h, G.BudgetParams(prm.target, prm.alpha, prm.band, prm.n_min,
                                           prm.n_max, prm.step),
                         torch.as_tensor(acc, dtype=torch.int32).to(DEV),
                         torch.as_tensor(status, dtype=torch.int32).to(DEV),
                         torch.as_tensor(parent, dtype=torch.int32).to(DEV), state, n_active_t)


@pytest.mark.parametrize("seed", range(3))
def test_controller_matches_the_oracle_bit_for_bit(h, seed):
    rng = np.random.default_rng(seed)
    B, N = 200, 64
    prm = BU.Params(target=float(rng.uniform(0.2, 0.8)), alpha=float(rng.uniform(0.05, 1.0)),
                    band=float(rng.uniform(0.0, 0.1)), n_min=int(rng.integers(1, 8)),
                    n_max=int(rng.integers(20, 65)), step=int(rng.integers(1, 5)))
    ref = BU.State(ema=float(rng.uniform()), budget=int(rng.integers(1, 65)))
    state = G.budget_state(ref.ema, ref.budget, DEV)
    n_t = torch.empty(B, dtype=torch.int32, device=DEV)
    n_ref = np.full(B, ref.budget, np.int32)
    for step in range(25):
        par = np.stack([W.random_trie(rng, N, 10, 6) for _ in range(B)])
        if step % 7 == 3:   # a few budgets outside [1, N]: those requests must not count
            n_ref[::5] = rng.integers(-2, N + 3, size=len(n_ref[::5]))
        n_t.copy_(torch.as_tensor(n_ref))
        depth_cap = np.array([BU.max_depth(par[b], min(max(int(n_ref[b]), 1), N))
                              for b in range(B)])
        acc = rng.integers(0, depth_cap + 1)
        status = np.where(rng.random(B) < 0.1, 3, 0)
        _gpu_update(h, prm, state, acc, status, par, n_t)
        ref = BU.update(prm, ref, acc, status, par, n_ref)
        ema, budget, steps = G.read_budget_state(state)
        assert (ema, budget, steps) == (ref.ema, ref.budget, ref.steps), (step, ema, ref)
        assert (n_t.cpu().numpy() == ref.budget).all()
        n_ref = np.full(B, ref.budget, np.int32)


def test_controller_argument_checks(h):
    par = torch.as_tensor(np.stack([W.chain(8)] * 2), dtype=torch.int32).to(DEV)
    z = torch.zeros(2, dtype=torch.int32, device=DEV)
    st = G.budget_state(0.5, 4, DEV)
    for bad in [G.BudgetParams(0.0, 0.5, 0.0, 1, 8, 1), G.BudgetParams(0.5, 1.5, 0.0, 1, 8, 1),
                G.BudgetParams(0.5, 0.5, -0.1, 1, 8, 1), G.BudgetParams(0.5, 0.5, 0.0, 0, 8, 1),
                G.BudgetParams(0.5, 0.5, 0.0, 5, 4, 1), G.BudgetParams(0.5, 0.5, 0.0, 1, 9, 1),
                G.BudgetParams(0.5, 0.5, 0.0, 1, 8, 0),
                G.BudgetParams(0.5, 0.5, float("inf"), 1, 8, 1)]:
        with pytest.raises(G.SpecError):
            G.spec_budget_update(h, bad, z, z, par, st, z.clone())
    assert G.read_budget_state(st) == (0.5, 4, 0)


def test_adaptive_step_replays_from_a_cuda_graph(h, orc):
    """verify (under the device budget) + controller update, captured once and replayed on new
    inputs: every replay uses the budget the previous replay wrote, like the oracle loop."""
    # boost 24: acceptance ratios of ~0.3-0.7 that fall as the budget grows, so the budget
    # moves both ways around the target
    w = W.WORKLOADS["sampling_trie"].scaled(B=8, V=9000, boost=24.0)
    prm = BU.Params(target=0.45, alpha=0.5, band=0.02, n_min=4, n_max=w.N, step=6)
    x = W.make(w, device=DEV, seed=20)
    static = {k: x[k].clone() for k in ("logits", "draft_token", "parent", "uniforms")}
    n_t = torch.full((w.B,), 10, dtype=torch.int32, device=DEV)
    state = G.budget_state(0.45, 10, DEV)
    out = G.alloc_outputs(w.B, w.N, DEV)
    G.spec_set_node_budget(h, n_t)
    bp = G.BudgetParams(prm.target, prm.alpha, prm.band, prm.n_min, prm.n_max, prm.step)

    def step():
        G.verify_sample(h, static["logits"], static["draft_token"], static["parent"],
                        w.temperature, static["uniforms"], out=out)
        G.spec_budget_update(h, bp, out["accept_len"], out["status"], static["parent"], state,
                             n_t)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()   # warm-up outside capture; restore the initial state afterwards
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    state.copy_(G.budget_state(0.45, 10, DEV))
    n_t.fill_(10)
    torch.cuda.synchronize()

    ref = BU.State(ema=0.45, budget=10)
    budgets = []
    for seed in range(21, 29):
        y = W.make(w, device=DEV, seed=seed)
        for k in static:
            static[k].copy_(y[k])
        n_ref = np.full(w.B, ref.budget, np.int32)
        assert (n_t.cpu().numpy() == n_ref).all()
        graph.replay()
        torch.cuda.synchronize()
        got = PY.to_np(out)
        want = oracle_budgeted(orc, y, n_ref, "sample", T=w.temperature)
        PY.compare_sample(got, want, max_excluded=0)   # the controller needs exact lengths
        assert np.array_equal(got["accept_len"], want["accept_len"])
        ref = BU.update(prm, ref, want["accept_len"], want["status"], y["parent_np"], n_ref)
        assert G.read_budget_state(state) == (ref.ema, ref.budget, ref.steps)
        budgets.append(ref.budget)
    assert len(set(budgets)) >= 3, budgets   # the budget moved both ways
