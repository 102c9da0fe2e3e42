"""CUDA path against the oracle, through the C ABI (needs a GB300 and the built library).

Greedy results, masks and argmax are compared bit for bit; sampling results are identical
except requests whose oracle decision or inverse-CDF margin is below 1e-6 (counted).
"""
import itertools
import os

import numpy as np
import pytest
import torch

import golden_io
import parity as PY
from oracle import enumerate as E
from oracle import oracle as O
from speculative_decoding_tree_mask_gb300 import binding as G
from speculative_decoding_tree_mask_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def h():
    G.load()
    with G.Handle(256, 64, 1 << 21, 0) as handle:
        yield handle


def _to(x, dtype=None):
    t = torch.as_tensor(x)
    if dtype is not None:
        t = t.to(dtype)
    return t.to(DEV).contiguous()


# ---- tree mask ---------------------------------------------------------------------------------

@pytest.mark.parametrize("N", [1, 2, 5, 32, 33, 64])
def test_tree_mask_bit_exact(h, orc, N):
    rng = np.random.default_rng(N)
    B = 37
    parents = [W.random_trie(rng, N, 10, 6) for _ in range(B - 3)]
    parents.append(W.chain(N))
    parents.append(np.array([-1] + [0] * (N - 1), np.int32))   # star
    bad = W.random_trie(rng, N, 10, 6)
    if N > 1:
        bad[N - 1] = N - 1                                         # parent not before child
    else:
        bad[0] = 0
    parents.append(bad)
    parent = np.stack(parents).astype(np.int32)
    out = G.build_tree_mask(h, _to(parent))
    torch.cuda.synchronize()
    anc, depth, status = orc.build_mask(parent)
    assert np.array_equal(out["anc_mask"].cpu().numpy().view(np.uint64), anc)
    assert np.array_equal(out["depth"].cpu().numpy(), depth)
    assert np.array_equal(out["status"].cpu().numpy(), status)
    assert status[-1] == 1 and (status[:-1] == 0).all()


# ---- hand-worked goldens through the GPU --------------------------------------------------------

@pytest.mark.parametrize("name", golden_io.names())
def test_golden_on_gpu(h, name):
    g = golden_io.load(name)
    if g["op"] == "mask":
        out = G.build_tree_mask(h, _to(g["parent"]))
        torch.cuda.synchronize()
        got = dict(anc=out["anc_mask"].cpu().numpy().view(np.uint64),
                   depth=out["depth"].cpu().numpy(), status=out["status"].cpu().numpy())
    elif g["op"] == "greedy":
        got = PY.gpu_greedy(h, _to(g["logits"]), _to(g["draft_token"]), _to(g["parent"]))
    else:
        kind = {"probs_f32": G.SPEC_DRAFT_PROBS_F32, "logits": G.SPEC_DRAFT_LOGITS}.get(
            g.get("draft_kind"), G.SPEC_DRAFT_POINT)
        draft = _to(g["draft"]) if "draft" in g else None
        got = PY.gpu_sample(h, _to(g["logits"]), _to(g["draft_token"]), _to(g["parent"]),
                            g["temperature"], _to(g["uniforms"]), draft, kind)
    assert golden_io.mismatches(g, got) == []


# ---- greedy -------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny_chain", "greedy_trie"])
def test_greedy_workloads_bit_exact(h, orc, name):
    w = W.WORKLOADS[name]
    x = W.make(w, device=DEV)
    gpu = PY.gpu_greedy(h, x["logits"], x["draft_token"], x["parent"])
    ref = orc.verify_greedy(PY.host(x["logits"]), x["tok_np"], x["parent_np"])
    PY.assert_exact(gpu, ref)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [1, 3, 8, 9, 255, 256, 257, 1000, 4097, 151936])
@pytest.mark.parametrize("offset", [0, 1])
def test_greedy_ragged_vocab_and_misaligned_rows(h, orc, dtype, V, offset):
    w = W.WORKLOADS["greedy_trie"].scaled(B=5, N=9, V=V, dtype=dtype, boost=15.0, seed=V + offset)
    x = W.make(w, device=DEV)
    flat = torch.empty(w.B * w.N * V + offset, dtype=w.torch_dtype, device=DEV)
    logits = flat[offset:].view(w.B, w.N, V)
    logits.copy_(x["logits"])
    gpu = PY.gpu_greedy(h, logits, x["draft_token"], x["parent"])
    ref = orc.verify_greedy(PY.host(x["logits"]), x["tok_np"], x["parent_np"])
    PY.assert_exact(gpu, ref)


def test_greedy_planted_ties_lowest_index(h, orc):
    B, N, V = 8, 4, 152064
    rng = np.random.default_rng(3)
    logits = torch.randn((B, N, V), device=DEV).to(torch.bfloat16)
    parent = np.tile(W.chain(N), (B, 1))
    tok = np.zeros((B, N), np.int32)
    for b in range(B):
        for i in range(N):
            pos = np.sort(rng.choice(V, size=4, replace=False))
            logits[b, i, torch.as_tensor(pos, device=DEV)] = 9.0
            if i + 1 < N:
                tok[b, i + 1] = pos[0]
    gpu = PY.gpu_greedy(h, logits, _to(tok), _to(parent))
    ref = orc.verify_greedy(PY.host(logits), tok, parent)
    PY.assert_exact(gpu, ref)
    assert (gpu["accept_len"] == N - 1).all()


def test_off_path_rows_may_hold_nan(h, orc):
    w = W.WORKLOADS["greedy_trie"].scaled(B=16, V=5000, boost=30.0, seed=77)
    x = W.make(w, device=DEV)
    ref = orc.verify_greedy(PY.host(x["logits"]), x["tok_np"], x["parent_np"])
    logits = x["logits"].clone()
    for b in range(w.B):
        on_path = set(ref["kv_commit"][b][ref["kv_commit"][b] >= 0].tolist())
        for i in range(w.N):
            if i not in on_path:
                logits[b, i] = float("nan")
    gpu = PY.gpu_greedy(h, logits, x["draft_token"], x["parent"])
    PY.assert_exact(gpu, ref)
    assert (gpu["status"] == 0).all()


# ---- row statistics -----------------------------------------------------------------------------

@pytest.mark.parametrize("T", [0.7, 1.0, 2.0])
@pytest.mark.parametrize("dtype,V", [("bf16", 151936), ("f32", 4099), ("bf16", 77)])
def test_row_stats_against_oracle(h, orc, T, dtype, V):
    w = W.WORKLOADS["sampling_trie"].scaled(B=6, N=16, V=V, dtype=dtype, seed=V)
    x = W.make(w, device=DEV)
    logits = x["logits"]
    logits[0, 3] = float("-inf")                       # all -inf row
    logits[1, 2, V // 2] = float("nan")                # NaN row
    logits[2, 5, V - 1] = float("inf")                 # +inf row
    logits[3, 1, : V // 2] = float("-inf")             # partly -inf
    rows = w.B * w.N
    m = torch.empty(rows, device=DEV)
    s = torch.empty(rows, device=DEV)
    a = torch.empty(rows, dtype=torch.int32, device=DEV)
    f = torch.empty(rows, dtype=torch.int32, device=DEV)
    pc = torch.full((w.B, w.N), -1.0, device=DEV)
    G.spec_row_stats(h, logits, w.N, T, m, s, a, f, x["draft_token"], x["parent"], pc)
    torch.cuda.synchronize()
    hl = PY.host(logits).reshape(rows, V)
    m, s, a, f, pc = (t.cpu().numpy() for t in (m, s, a, f, pc))
    for r in range(rows):
        om, oS, oa, obad = orc.row_stats(hl[r], T)
        assert (f[r] != 0) == bool(obad), r
        if obad:
            continue
        assert m[r] == om and a[r] == oa, r
        assert abs(s[r] - oS) <= 1e-5 * oS, (r, s[r], oS)
    for b in range(w.B):
        for c in range(1, w.N):
            par = x["parent_np"][b, c]
            r = b * w.N + par
            if orc.row_stats(hl[r], T)[3]:
                continue
            p = orc.row_softmax(hl[r], T)[x["tok_np"][b, c]]
            assert abs(pc[b, c] - p) <= 1e-5 * p + 1e-30, (b, c, pc[b, c], p)



@pytest.mark.parametrize("B", [1, 6, 12, 24, 60])
@pytest.mark.parametrize("dtype,V", [("bf16", 151936), ("f32", 4099)])
def test_row_stats_every_row_split(h, orc, B, dtype, V):
    """Few rows are streamed by several CTAs each (8, 4 or 2 pieces, merged by the last CTA to
    finish): 16-node requests give 16 to 960 rows, across every split of a 152-SM GPU and the
    unsplit kernel. Repeated calls check that the per-row arrival counters start from zero."""
    w = W.WORKLOADS["sampling_trie"].scaled(B=B, N=16, V=V, dtype=dtype, seed=B * 7 + V)
    x = W.make(w, device=DEV)
    rows = w.B * w.N
    hl = PY.host(x["logits"]).reshape(rows, V)
    ref = [orc.row_stats(hl[r], 1.0) for r in range(rows)]
    for T, rep in ((1.0, 0), (1.0, 1), (0.0, 0)):
        m = torch.empty(rows, device=DEV)
        s = torch.empty(rows, device=DEV)
        a = torch.empty(rows, dtype=torch.int32, device=DEV)
        f = torch.empty(rows, dtype=torch.int32, device=DEV)
        G.spec_row_stats(h, x["logits"], w.N, T, m, s, a, f)
        torch.cuda.synchronize()
        m, s, a, f = (t.cpu().numpy() for t in (m, s, a, f))
        assert not f.any()
        for r in range(rows):
            om, oS, oa, _ = ref[r]
            assert m[r] == om and a[r] == oa, (T, rep, r)
            if T > 0:
                assert abs(s[r] - oS) <= 1e-5 * oS, (rep, r, s[r], oS)
            else:
                assert s[r] == 0.0, r

# ---- sampling, point-mass drafts ----------------------------------------------------------------

@pytest.mark.parametrize("T,boost", [(0.7, 8.0), (0.7, 30.0), (1.0, 12.0), (1.8, 20.0)])
def test_sample_point_trie(h, orc, T, boost):
    w = W.WORKLOADS["sampling_trie"].scaled(temperature=T, boost=boost, seed=int(T * 100 + boost))
    x = W.make(w, device=DEV)
    gpu = PY.gpu_sample(h, x["logits"], x["draft_token"], x["parent"], T, x["uniforms"])
    ref = PY.oracle_sample(orc, x["logits"], x["draft_token"], x["parent"], T, x["uniforms"])
    PY.compare_sample(gpu, ref)


@pytest.mark.parametrize("lazy", [False, True])
@pytest.mark.parametrize("dtype,V", [("bf16", 20008), ("bf16", 151936), ("f32", 4100),
                                     ("bf16", 20001)])
def test_bonus_in_the_ragged_last_chunk(h, orc, dtype, V, lazy):
    """Bonus uniforms near 1 put tau in the row's last chunk, whose last 256-token sub-tile is
    ragged (V not a multiple of 256). The register draw takes it with the vectors past V
    masked when V is a multiple of the vector width (8 bf16, 4 f32); V = 20001 leaves the rows
    unaligned and takes the whole-row search instead."""
    w = W.WORKLOADS["sampling_trie"].scaled(B=24, N=16, V=V, dtype=dtype, boost=4.0,
                                            sigma=2.0, temperature=1.0, seed=V + 17 * lazy)
    x = W.make(w, device=DEV)
    u = x["uniforms"].clone()
    u[:, w.N] = torch.linspace(0.95, 0.99999, w.B, device=DEV)
    fn = G.verify_sample_lazy if lazy else G.verify_sample
    gpu = PY.to_np(fn(h, x["logits"], x["draft_token"], x["parent"], 1.0, u))
    torch.cuda.synchronize()
    ref = PY.oracle_sample(orc, x["logits"], x["draft_token"], x["parent"], 1.0, u)
    PY.compare_sample(gpu, ref)
    ok = gpu["status"] == 0
    assert ok.all()
    # the draws land in the last chunk's tokens (an eighth of the row's sub-tiles, a sixteenth
    # for the lazy walk's chunks)
    nsub, nc = (V + 255) // 256, 16 if lazy else 8
    last = nsub * (nc - 1) // nc * 256
    assert (gpu["bonus"][ok] >= last).mean() > 0.3


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("mode", ["greedy", "sample", "lazy"])
def test_maximum_vocabulary(h, orc, dtype, mode):
    """V = 2^21, the largest vocabulary a handle serves: 8192 sub-tile sums per row, bonus
    chunks of 1024 sub-tiles (more than the register draw holds, so the chunk is summed and
    searched), and the lazy walk's largest shared-memory request."""
    V = 1 << 21
    w = W.WORKLOADS["sampling_trie"].scaled(B=2, N=6, V=V, dtype=dtype, boost=10.0,
                                            sigma=2.0, temperature=1.0, seed=21 + len(mode))
    x = W.make(w, device=DEV)
    if mode == "greedy":
        got = PY.gpu_greedy(h, x["logits"], x["draft_token"], x["parent"])
        PY.assert_exact(got, orc.verify_greedy(PY.host(x["logits"]), x["tok_np"],
                                               x["parent_np"]))
        return
    fn = G.verify_sample_lazy if mode == "lazy" else G.verify_sample
    gpu = PY.to_np(fn(h, x["logits"], x["draft_token"], x["parent"], 1.0, x["uniforms"]))
    torch.cuda.synchronize()
    ref = PY.oracle_sample(orc, x["logits"], x["draft_token"], x["parent"], 1.0, x["uniforms"])
    PY.compare_sample(gpu, ref)
    assert (gpu["status"] == 0).all()


def test_sample_point_many_small_requests(h, orc):
    w = W.WORKLOADS["sampling_trie"].scaled(B=256, N=24, V=3001, dtype="f32", boost=6.0,
                                            sigma=1.5, temperature=1.0, seed=9)
    x = W.make(w, device=DEV)
    gpu = PY.gpu_sample(h, x["logits"], x["draft_token"], x["parent"], 1.0, x["uniforms"])
    ref = PY.oracle_sample(orc, x["logits"], x["draft_token"], x["parent"], 1.0, x["uniforms"])
    PY.compare_sample(gpu, ref)
    assert gpu["accept_len"].max() >= 2


def test_sample_rejected_mass_resummed(h, orc):
    """The first child holds almost all the mass and is rejected: the next sibling's
    denominator is re-summed over the row."""
    B, N, V = 8, 4, 151936
    g = torch.Generator(device=DEV)
    g.manual_seed(17)
    logits = (3.0 * torch.randn((B, N, V), device=DEV, generator=g)).to(torch.bfloat16)
    parent = np.tile(np.array([-1, 0, 0, 0], np.int32), (B, 1))
    tok = np.tile(np.array([0, 11, 22, 33], np.int32), (B, 1))
    logits[:, 0, 11] = 20.0
    logits[:, 0, 22] = 3.0
    u = torch.rand((B, N + 1), device=DEV, generator=g)
    u[:, 1] = 0.99999
    gpu = PY.gpu_sample(h, logits, _to(tok), _to(parent), 1.0, u)
    ref = PY.oracle_sample(orc, logits, _to(tok), _to(parent), 1.0, u)
    PY.compare_sample(gpu, ref)


@pytest.mark.parametrize("lazy", [False, True])
@pytest.mark.parametrize("chunks", [1, 2, 4])
def test_heavy_rejections_across_chunks(h, orc, lazy, chunks):
    """Four children of the root hold 99.6% of the row's mass and are rejected one after
    another. Before the fourth decision the residual is re-summed: the eager walk sums the
    chunks holding rejected tokens exactly and takes the rest from the chunk partials when
    there are at most two such chunks, else (and in the lazy walk) the whole row. The bonus
    after the last rejection sums the whole row. The rejected tokens lie in one, two or four
    of the row's chunks."""
    B, N, V = 16, 5, 151936
    g = torch.Generator(device=DEV)
    g.manual_seed(23 + chunks)
    logits = (3.0 * torch.randn((B, N, V), device=DEV, generator=g)).to(torch.bfloat16)
    toks = {1: [1000, 1010, 1020, 1030], 2: [1000, 1010, 150000, 150010],
            4: [1000, 150000, 70000, 40000]}[chunks]
    for t, v in zip(toks, [22.0, 21.0, 20.0, 19.0]):
        logits[:, 0, t] = v
    parent = _to(np.tile(np.array([-1, 0, 0, 0, 0], np.int32), (B, 1)))
    tok = _to(np.tile(np.array([0] + toks, np.int32), (B, 1)))
    u = torch.rand((B, N + 1), device=DEV, generator=g)
    u[:, 1:5] = 0.999999
    fn = G.verify_sample_lazy if lazy else G.verify_sample
    out = fn(h, logits, tok, parent, 1.0, u)
    torch.cuda.synchronize()
    gpu = PY.to_np(out)
    ref = PY.oracle_sample(orc, logits, tok, parent, 1.0, u)
    assert (ref["accept_len"] == 0).all()
    PY.compare_sample(gpu, ref)

@pytest.mark.parametrize("lazy", [False, True])
@pytest.mark.parametrize("top", [20.0, 16.5, 15.0, 12.0])
def test_bonus_after_a_heavy_rejection(h, orc, lazy, top):
    """The root's only child holds a large share of the row's mass (about 97%, 50%, 20% and 1%
    for these logits against N(0, 3) noise over 151936 tokens) and is rejected: the bonus is
    drawn from the residual without that token, whose mass is comparable to the rounding of
    the row sum when the share is large."""
    B, N, V = 64, 2, 151936
    g = torch.Generator(device=DEV)
    g.manual_seed(int(top * 10))
    logits = (3.0 * torch.randn((B, N, V), device=DEV, generator=g)).to(torch.bfloat16)
    tok = torch.randint(0, V, (B,), device=DEV, generator=g, dtype=torch.int32)
    logits[torch.arange(B, device=DEV), 0, tok.long()] = top
    draft_token = torch.stack([torch.zeros_like(tok), tok], dim=1).contiguous()
    parent = _to(np.tile(np.array([-1, 0], np.int32), (B, 1)))
    u = torch.rand((B, N + 1), device=DEV, generator=g)
    u[:, 1] = 0.999999
    fn = G.verify_sample_lazy if lazy else G.verify_sample
    out = fn(h, logits, draft_token, parent, 1.0, u)
    torch.cuda.synchronize()
    gpu = PY.to_np(out)
    ref = PY.oracle_sample(orc, logits, draft_token, parent, 1.0, u)
    assert (ref["accept_len"] == 0).all()
    PY.compare_sample(gpu, ref)


def test_temperature_zero_is_greedy(h):
    w = W.WORKLOADS["sampling_trie"].scaled(boost=25.0, seed=4)
    x = W.make(w, device=DEV)
    a = PY.gpu_greedy(h, x["logits"], x["draft_token"], x["parent"])
    b = PY.gpu_sample(h, x["logits"], x["draft_token"], x["parent"], 0.0, x["uniforms"])
    for k in PY.KEYS:
        assert np.array_equal(a[k], b[k])


def test_sampling_is_deterministic(h):
    w = W.WORKLOADS["sampling_trie"].scaled(boost=12.0, seed=5)
    x = W.make(w, device=DEV)
    a = PY.gpu_sample(h, x["logits"], x["draft_token"], x["parent"], 0.7, x["uniforms"])
    b = PY.gpu_sample(h, x["logits"], x["draft_token"], x["parent"], 0.7, x["uniforms"])
    for k in PY.KEYS:
        assert np.array_equal(a[k], b[k])


# ---- sampling, dense drafts --------------------------------------------------------------------

def test_dense_chain_logits(h, orc):
    w = W.WORKLOADS["dense_chain"]
    x = W.make(w, device=DEV)
    gpu = PY.gpu_sample(h, x["logits"], x["draft_token"], x["parent"], 1.0, x["uniforms"],
                        x["draft"], G.SPEC_DRAFT_LOGITS)
    ref = PY.oracle_sample(orc, x["logits"], x["draft_token"], x["parent"], 1.0, x["uniforms"],
                           x["draft"], G.SPEC_DRAFT_LOGITS)
    PY.compare_sample(gpu, ref)


@pytest.mark.parametrize("V", [1000, 4103])
def test_dense_chain_probs(h, orc, V):
    w = W.WORKLOADS["dense_chain"].scaled(B=32, V=V, dtype="f32", seed=V)
    x = W.make(w, device=DEV)
    probs = torch.softmax(x["draft"].float().cpu(), dim=-1).contiguous()
    probs[:, -1] = float("nan")            # the leaf's draft row is never read
    gpu = PY.gpu_sample(h, x["logits"], x["draft_token"], x["parent"], 1.0, x["uniforms"],
                        probs.to(DEV), G.SPEC_DRAFT_PROBS_F32)
    ref = PY.oracle_sample(orc, x["logits"], x["draft_token"], x["parent"], 1.0, x["uniforms"],
                           probs, G.SPEC_DRAFT_PROBS_F32)
    PY.compare_sample(gpu, ref)
    assert (gpu["status"] == 0).all()


def test_dense_tree_logits(h, orc):
    """Dense drafts on trees: siblings tested against successive residual levels."""
    rng = np.random.default_rng(8)
    B, N, V, T = 64, 12, 3000, 1.0
    parent = np.stack([W.random_trie(rng, N, 3, 4) for _ in range(B)])
    target = torch.randn((B, N, V), generator=torch.Generator().manual_seed(1)) * 1.0
    draft = target + 0.7 * torch.randn((B, N, V), generator=torch.Generator().manual_seed(2))
    probs = torch.softmax(draft / T, dim=-1)
    tok = np.zeros((B, N), np.int32)
    for b in range(B):
        for c in range(1, N):
            tok[b, c] = int(torch.multinomial(probs[b, parent[b, c]], 1,
                                              generator=torch.Generator().manual_seed(b * N + c)))
    u = torch.rand((B, N + 1), generator=torch.Generator().manual_seed(3))
    args = (_to(target), _to(tok), _to(parent), T, _to(u))
    gpu = PY.gpu_sample(h, *args, _to(draft), G.SPEC_DRAFT_LOGITS)
    ref = PY.oracle_sample(orc, *args, draft, G.SPEC_DRAFT_LOGITS)
    PY.compare_sample(gpu, ref)



@pytest.mark.parametrize("B", [3, 30, 60, 100, 200])
@pytest.mark.parametrize("kind", ["point", "dense"])
def test_walk_clusters(h, orc, B, kind):
    """With dense drafts, few requests run their walk on a thread-block cluster of 8, 4 or 2
    CTAs that share every vocabulary pass (sub-tile sums and totals exchanged through
    distributed shared memory): 3 to 200 requests span every cluster size of a 152-SM GPU (8
    CTAs up to 19 requests, 4 up to 38, 2 up to 76) and one CTA per request beyond. Point
    drafts, one CTA per request, run the same batch sizes. Odd V leaves a ragged last
    sub-tile and, for bf16 rows, rows that are not 16-byte aligned."""
    rng = np.random.default_rng(B * 31 + len(kind))
    N, T = 12, 1.0
    V = 20011 if kind == "point" else 9001
    parent = np.stack([W.random_trie(rng, N, 4, 3) for _ in range(B)])
    gen = torch.Generator().manual_seed(B)
    target = torch.randn((B, N, V), generator=gen) * (3.0 if kind == "point" else 1.0)
    tok = np.zeros((B, N), np.int32)
    draft = None
    if kind == "point":
        for b in range(B):
            tok[b] = W.child_tokens(rng, parent[b], V)
            for i in range(N):   # boost the first child (most nodes) so that walks go deep
                kids = np.nonzero(parent[b] == i)[0]
                if len(kids):
                    t = int(tok[b, kids[0]]) if rng.random() < 0.7 else int(rng.integers(V))
                    target[b, i, t] += 18.0
    else:
        draft = target + 0.7 * torch.randn((B, N, V), generator=gen)
        probs = torch.softmax(draft / T, dim=-1)
        for b in range(B):
            for c in range(1, N):
                tok[b, c] = int(torch.multinomial(probs[b, parent[b, c]], 1, generator=gen))
    logits = target.to(torch.bfloat16)
    u = torch.rand((B, N + 1), generator=gen)
    args = (_to(logits), _to(tok), _to(parent), T, _to(u))
    if kind == "point":
        gpu = PY.gpu_sample(h, *args)
        ref = PY.oracle_sample(orc, *args)
        assert gpu["accept_len"].max() >= 2
    else:
        dl = draft.to(torch.bfloat16)
        gpu = PY.gpu_sample(h, *args, _to(dl), G.SPEC_DRAFT_LOGITS)
        ref = PY.oracle_sample(orc, *args, dl, G.SPEC_DRAFT_LOGITS)
    PY.compare_sample(gpu, ref)
    # the same call twice gives the same outputs
    again = PY.gpu_sample(h, *args) if kind == "point" else \
        PY.gpu_sample(h, *args, _to(dl), G.SPEC_DRAFT_LOGITS)
    for k in PY.KEYS:
        assert np.array_equal(gpu[k], again[k]), k

# ---- full-size large-tree workload ----------------------------------------------------------------

def test_large_tree_full_size(h, orc):
    w = W.WORKLOADS["large_tree"]
    x = W.make(w, device=DEV)
    T = w.temperature
    gpu = PY.gpu_sample(h, x["logits"], x["draft_token"], x["parent"], T, x["uniforms"])
    # every request: structural properties of the result
    _, depth, _ = orc.build_mask(x["parent_np"])
    for b in range(w.B):
        par, tok = x["parent_np"][b], x["tok_np"][b]
        L = gpu["accept_len"][b]
        kv = gpu["kv_commit"][b]
        assert gpu["status"][b] == 0 and 0 <= L <= depth[b].max()
        assert kv[0] == 0 and all(par[kv[j + 1]] == kv[j] for j in range(L))
        assert (gpu["out_tokens"][b, :L] == tok[kv[1:L + 1]]).all()
        kids = [c for c in range(w.N) if par[c] == kv[L]]
        assert gpu["bonus"][b] not in tok[kids]       # rejected tokens leave the residual
    # every request against the oracle: sampling, then greedy on the same trees
    threads = os.cpu_count() or 8
    ref = PY.oracle_sample(orc, x["logits"], x["draft_token"], x["parent"], T, x["uniforms"],
                           nthreads=threads)
    PY.compare_sample(gpu, ref)
    gg = PY.gpu_greedy(h, x["logits"], x["draft_token"], x["parent"])
    gref = orc.verify_greedy(PY.host(x["logits"]), x["tok_np"], x["parent_np"], nthreads=threads)
    PY.assert_exact(gg, gref)


# ---- losslessness on the GPU (Monte Carlo against the exact law) --------------------------------

def _chi2(samples, law):
    from test_oracle_lossless import _chi2_pvalue
    return _chi2_pvalue(samples, law)


def test_gpu_point_mass_law(orc):
    parent, tokens = [-1, 0, 0, 0, 1, 2], [0, 2, 0, 3, 1, 1]
    V, T, n = 5, 0.9, 100_000
    model = E.SyntheticLM(V, seed=101, scale=1.3)
    rows = torch.as_tensor(E.tree_rows(model, tokens, parent))
    logits = rows.expand(n, -1, -1).contiguous().to(DEV)
    u = torch.rand((n, len(parent) + 1), generator=torch.Generator().manual_seed(5)).to(DEV)
    with G.Handle(n, 8, 64) as hh:
        out = PY.gpu_sample(hh, logits, _to(np.tile(tokens, (n, 1)).astype(np.int32)),
                            _to(np.tile(parent, (n, 1)).astype(np.int32)), T, u)
    seqs = [tuple(out["out_tokens"][i, :out["accept_len"][i] + 1]) for i in range(n)]
    assert _chi2(seqs, E.verify_point_dist(model, tokens, parent, T)) > 1e-5


def test_gpu_dense_chain_law(orc):
    k, V, T, n = 2, 4, 1.0, 100_000
    model, draft = E.SyntheticLM(V, seed=31, scale=1.5), E.SyntheticLM(V, seed=32, scale=1.5)
    parent = [-1] + list(range(k))
    chains = list(itertools.product(range(V), repeat=k))
    wts = []
    for xs in chains:
        pw, pre = 1.0, ()
        for t in xs:
            pw *= draft.probs(pre, T)[t]
            pre += (t,)
        wts.append(pw)
    rng = np.random.default_rng(6)
    pick = rng.choice(len(chains), size=n, p=np.array(wts) / sum(wts))
    rows = np.stack([E.tree_rows(model, (0,) + xs, parent) for xs in chains])[pick]
    drows = np.stack([E.tree_rows(draft, (0,) + xs, parent) for xs in chains])[pick]
    toks = np.array([(0,) + xs for xs in chains], np.int32)[pick]
    u = rng.random((n, k + 2), dtype=np.float32)
    with G.Handle(n, 8, 64) as hh:
        out = PY.gpu_sample(hh, _to(rows), _to(toks), _to(np.tile(parent, (n, 1)).astype(np.int32)),
                            T, _to(u), _to(drows), G.SPEC_DRAFT_LOGITS)
    seqs = [tuple(out["out_tokens"][i, :out["accept_len"][i] + 1]) for i in range(n)]
    assert _chi2(seqs, E.dense_chain_mixture(model, draft, k, T)) > 1e-5


# ---- API behaviour ---------------------------------------------------------------------------------

def test_host_argument_errors(h):
    w = W.WORKLOADS["sampling_trie"].scaled(B=2, N=4, V=100, seed=1)
    x = W.make(w, device=DEV)
    out = G.alloc_outputs(2, 4, DEV)
    with pytest.raises(G.SpecError) as e:
        G.verify_sample(h, x["logits"], x["draft_token"], x["parent"], -1.0, x["uniforms"])
    assert e.value.code == G.SPEC_ERR_ARG
    with pytest.raises(G.SpecError):
        G.verify_sample(h, x["logits"], x["draft_token"], x["parent"], float("nan"), x["uniforms"])
    with pytest.raises(G.SpecError):
        G.verify_sample(h, x["logits"], x["draft_token"], x["parent"], 1.0, x["uniforms"],
                        draft=None, draft_kind=G.SPEC_DRAFT_LOGITS)
    big = torch.zeros((257, 4, 100), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(G.SpecError):
        G.verify_greedy(h, big, torch.zeros((257, 4), dtype=torch.int32, device=DEV),
                        torch.zeros((257, 4), dtype=torch.int32, device=DEV))
    with pytest.raises(G.SpecError) as e:
        G.Handle(4, 65, 100)
    assert e.value.code == G.SPEC_ERR_UNSUPPORTED
    # B == 0 is a no-op for every call: nothing is launched or written
    e = {k: x[k][:0] for k in ("logits", "draft_token", "parent", "uniforms")}
    before = {k: v.clone() for k, v in out.items()}
    G.spec_verify_greedy(h, e["logits"], e["draft_token"], e["parent"], out["accept_len"],
                         out["out_tokens"], out["kv_commit"], out["bonus"], out["status"])
    G.spec_verify_sample(h, e["logits"], e["draft_token"], e["parent"], 1.0, e["uniforms"],
                         out["accept_len"], out["out_tokens"], out["kv_commit"], out["bonus"],
                         out["status"])
    G.spec_verify_greedy_lazy(h, e["logits"], e["draft_token"], e["parent"], out["accept_len"],
                              out["out_tokens"], out["kv_commit"], out["bonus"], out["status"])
    G.spec_verify_sample_lazy(h, e["logits"], e["draft_token"], e["parent"], 1.0, e["uniforms"],
                              out["accept_len"], out["out_tokens"], out["kv_commit"],
                              out["bonus"], out["status"])
    # (empty views of allocated tensors, so that every pointer is a valid one)
    mask = dict(anc=torch.zeros((1, 4), dtype=torch.int64, device=DEV)[:0],
                depth=torch.zeros((1, 4), dtype=torch.int32, device=DEV)[:0],
                status=torch.zeros(1, dtype=torch.int32, device=DEV)[:0])
    G.spec_build_tree_mask(h, e["parent"], mask["anc"], mask["depth"], mask["status"])
    kvsrc = torch.zeros((1, 4, 2, 16), dtype=torch.bfloat16, device=DEV)[:0]
    cache = torch.zeros((2, 8, 2, 16), dtype=torch.bfloat16, device=DEV)
    G.spec_kv_commit(h, kvsrc, kvsrc, e["parent"], out["accept_len"][:0], cache, cache.clone(),
                     G.SPEC_KV_NHD, torch.zeros((1, 1), dtype=torch.int32, device=DEV)[:0],
                     torch.zeros(1, dtype=torch.int32, device=DEV)[:0])
    torch.cuda.synchronize()
    for k, v in out.items():
        assert torch.equal(v, before[k]), k
    assert not cache.any()


def test_side_stream_and_profiling(h):
    w = W.WORKLOADS["sampling_trie"].scaled(B=4, N=8, V=20000, seed=2)
    x = W.make(w, device=DEV)
    s = torch.cuda.Stream()
    ref = PY.gpu_sample(h, x["logits"], x["draft_token"], x["parent"], 0.7, x["uniforms"])
    G.spec_profile_begin(h)
    with torch.cuda.stream(s):
        out = G.verify_sample(h, x["logits"], x["draft_token"], x["parent"], 0.7, x["uniforms"],
                              stream=s)
    s.synchronize()
    prof = G.spec_profile_end(h)
    assert prof["row_stats"][1] == 1 and prof["walk_sample"][1] == 1
    assert prof["row_stats"][0] > 0
    for k in PY.KEYS:
        assert np.array_equal(out[k].cpu().numpy(), ref[k])


def test_verify_waits_for_the_kernel_that_writes_the_logits(h, orc):
    """The stages are launched as programmatic dependents; each must still see everything the
    kernels before it in the stream wrote. Two inputs whose greedy results differ are copied
    alternately into one buffer by a device copy kernel, each copy followed at once (no
    synchronisation) by a verify call on the same stream."""
    w = W.WORKLOADS["greedy_trie"].scaled(B=16, V=40000)
    xa, xb = W.make(w, device=DEV, seed=31), W.make(w, device=DEV, seed=32)
    xb["draft_token"] = xa["draft_token"]
    xb["parent"] = xa["parent"]
    ref = {k: orc.verify_greedy(PY.host(x["logits"]), xa["tok_np"], xa["parent_np"])
           for k, x in (("a", xa), ("b", xb))}
    assert not np.array_equal(ref["a"]["bonus"], ref["b"]["bonus"])
    buf = torch.empty_like(xa["logits"])
    outs = []
    for i in range(12):
        buf.copy_((xa if i % 2 == 0 else xb)["logits"])
        o = G.verify_greedy(h, buf, xa["draft_token"], xa["parent"])
        outs.append({k: v.clone() for k, v in o.items()})
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        PY.assert_exact(PY.to_np(o), ref["a" if i % 2 == 0 else "b"])
