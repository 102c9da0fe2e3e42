"""Randomised parity sweep: many small seeded configurations (tree shapes, vocabulary sizes
around the vector and sub-tile boundaries, element types, temperatures, boosts, draft kinds,
node budgets, eager and lazy calls) against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import parity as PY
from oracle import budget as BU
from speculative_decoding_tree_mask_gb300 import binding as G
from speculative_decoding_tree_mask_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
CASES = 48


@pytest.fixture(scope="module")
def h():
    G.load()
    with G.Handle(64, 64, 1 << 16, 0) as handle:
        yield handle


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 33))
    N = int(rng.choice([1, 2, 3, 7, 16, 31, 32, 33, 63, 64]))
    V = int(rng.choice([1, 2, 7, 8, 9, 255, 256, 257, 1000, 2048, 4097, 9001, 40000]))
    dtype = str(rng.choice(["bf16", "f32"]))
    mode = str(rng.choice(["greedy", "point", "point", "logits", "probs"]))
    T = float(rng.choice([0.3, 0.7, 1.0, 1.6]))
    boost = float(rng.choice([0.0, 4.0, 12.0, 30.0]))
    sigma = float(rng.choice([1.0, 3.0]))
    lazy = bool(rng.integers(0, 2))
    budget = bool(rng.integers(0, 4) == 0)
    chain = mode in ("logits", "probs") and bool(rng.integers(0, 2))
    return dict(B=B, N=N, V=V, dtype=dtype, mode=mode, T=T, boost=boost, sigma=sigma,
                lazy=lazy, budget=budget, chain=chain, seed=seed)


def _inputs(c):
    rng = np.random.default_rng(c["seed"])
    B, N, V = c["B"], c["N"], c["V"]
    if c["chain"]:
        parent = np.stack([W.chain(N) for _ in range(B)])
    else:
        parent = np.stack([W.random_trie(rng, N, int(rng.integers(1, 11)),
                                         int(rng.integers(1, 7))) for _ in range(B)])
    tok = np.stack([W.child_tokens(rng, parent[b], V) for b in range(B)])
    g = torch.Generator().manual_seed(c["seed"])
    z = torch.randn((B, N, V), generator=g) * c["sigma"]
    # boost the first child's token in each row, so walks go deep
    for b in range(B):
        for i in range(N):
            kids = np.nonzero(parent[b] == i)[0]
            kids = kids[kids > 0]
            if len(kids):
                z[b, i, int(tok[b, kids[0]])] += c["boost"]
    tdt = torch.bfloat16 if c["dtype"] == "bf16" else torch.float32
    logits = z.to(tdt)
    draft = None
    if c["mode"] in ("logits", "probs"):
        d = z + 0.6 * torch.randn((B, N, V), generator=g)
        draft = d.to(tdt) if c["mode"] == "logits" else torch.softmax(d / c["T"], -1).float()
        # dense drafts: child tokens drawn from the parent's draft row
        q = torch.softmax(draft.float() / (c["T"] if c["mode"] == "logits" else 1.0), -1) \
            if c["mode"] == "logits" else draft
        for b in range(B):
            for i in range(1, N):
                tok[b, i] = int(torch.multinomial(q[b, parent[b, i]], 1, generator=g))
    u = torch.rand((B, N + 1), generator=g)
    n_active = None
    if c["budget"]:
        n_active = rng.integers(1, N + 1, size=B).astype(np.int32)
    return parent.astype(np.int32), tok.astype(np.int32), logits, draft, u, n_active


@pytest.mark.parametrize("seed", range(CASES))
def test_fuzz_against_oracle(h, orc, seed):
    c = _case(seed)
    parent, tok, logits, draft, u, n_active = _inputs(c)
    B, N = parent.shape
    dl, dt, dp = logits.to(DEV), torch.from_numpy(tok).to(DEV), torch.from_numpy(parent).to(DEV)
    du = u.to(DEV)
    ddraft = None if draft is None else draft.to(DEV)
    kind = {"logits": G.SPEC_DRAFT_LOGITS, "probs": G.SPEC_DRAFT_PROBS_F32}.get(
        c["mode"], G.SPEC_DRAFT_POINT)
    na = None
    if n_active is not None:
        na = torch.from_numpy(n_active).to(DEV)
        G.spec_set_node_budget(h, na)
    try:
        if c["mode"] == "greedy":
            fn = G.verify_greedy_lazy if c["lazy"] else G.verify_greedy
            out = fn(h, dl, dt, dp)
        else:
            fn = G.verify_sample_lazy if c["lazy"] else G.verify_sample
            out = fn(h, dl, dt, dp, c["T"], du, draft=ddraft, draft_kind=kind)
        torch.cuda.synchronize()
    finally:
        G.spec_set_node_budget(h, None)
    got = PY.to_np(out)
    # the oracle, request by request on the (possibly truncated) tree
    hl = W.host_logits(logits)
    hd = None if draft is None else (W.host_logits(draft) if c["mode"] == "logits"
                                     else draft.numpy())
    keys = PY.KEYS + ("decision_margin", "cdf_margin", "cdf_alt", "cdf_lo", "cdf_hi")
    ref = {k: [] for k in keys}
    for b in range(B):
        n = N if n_active is None else int(n_active[b])
        lg, tk, pr, uu, dr = BU.truncate(hl[b], tok[b], parent[b], u[b].numpy(), n,
                                         None if hd is None else hd[b])
        if c["mode"] == "greedy":
            r = orc.verify_greedy(lg[None], tk[None], pr[None])
        else:
            r = orc.verify_sample(lg[None], tk[None], pr[None], c["T"], uu[None],
                                  draft=None if dr is None else dr[None],
                                  draft_kind=PY.ORACLE_KIND[kind])
        for k in keys:
            if k in r:
                v = r[k][0]
                if k in ("out_tokens", "kv_commit"):
                    v = np.concatenate([v, np.full(N - n, -1, v.dtype)])
                ref[k].append(v)
    ref = {k: np.stack(v) for k, v in ref.items() if v}
    if c["mode"] == "greedy":
        PY.assert_exact(got, ref)
    else:
        PY.compare_sample(got, ref)
