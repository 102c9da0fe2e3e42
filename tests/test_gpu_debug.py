"""The debug flavour (SPEC_DEBUG): the same kernels with their own consistency checks compiled
in, standing in for a memory checker on this pool. It must give the release results on a
parity subset (goldens, the small tries, the dense chain, lazy calls, fuzz cases, KV commit,
the no-allocation call), report data errors planted on the host with their usual codes, and
turn an arrival counter corrupted on the host into SPEC_REQ_INTERNAL for the affected request
only, with no trap, fault or wait on the GPU."""
import numpy as np
import pytest
import torch

import golden_io
import parity as PY
from speculative_decoding_tree_mask_gb300 import binding as G
from speculative_decoding_tree_mask_gb300 import build as Build
from speculative_decoding_tree_mask_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def dbg_lib():
    path = Build.build(debug=True)
    with G.use_library(path) as lib:
        yield lib


@pytest.fixture(scope="module")
def h(dbg_lib):
    with G.Handle(256, 64, 1 << 21, 0) as handle:
        yield handle


def _to(x):
    return torch.as_tensor(x).to(DEV).contiguous()


def _clean(h, B):
    words = G.spec_debug_words(h, B).cpu().numpy()
    assert (words == 0).all(), words


def test_the_debug_library_is_loaded(dbg_lib):
    assert G.spec_debug_build()


@pytest.mark.parametrize("name", golden_io.names())
def test_goldens(h, name):
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


@pytest.mark.parametrize("name,lazy", [("greedy_trie", False), ("greedy_trie", True),
                                       ("sampling_trie", False), ("sampling_trie", True),
                                       ("tiny_chain", False)])
def test_workloads_match_the_oracle(h, orc, name, lazy):
    """The small tries stream each row over several CTAs (the arrival counters are checked on
    every row); the lazy calls check their own row passes."""
    w = W.WORKLOADS[name].scaled(boost=20.0)
    x = W.make(w, device=DEV)
    if w.mode == "greedy":
        fn = G.verify_greedy_lazy if lazy else G.verify_greedy
        got = PY.to_np(fn(h, x["logits"], x["draft_token"], x["parent"]))
        torch.cuda.synchronize()
        PY.assert_exact(got, orc.verify_greedy(PY.host(x["logits"]), x["tok_np"],
                                               x["parent_np"]))
    else:
        fn = G.verify_sample_lazy if lazy else G.verify_sample
        got = PY.to_np(fn(h, x["logits"], x["draft_token"], x["parent"], w.temperature,
                          x["uniforms"]))
        torch.cuda.synchronize()
        PY.compare_sample(got, PY.oracle_sample(orc, x["logits"], x["draft_token"], x["parent"],
                                                w.temperature, x["uniforms"]))
    assert (got["status"] == 0).all()
    _clean(h, w.B)


@pytest.mark.parametrize("lazy", [False, True])
def test_dense_chain_matches_the_oracle(h, orc, lazy):
    """Dense drafts: the clustered eager walk (several CTAs per request) and the lazy walk."""
    w = W.WORKLOADS["dense_chain"].scaled(B=16, V=20000)
    x = W.make(w, device=DEV)
    fn = G.verify_sample_lazy if lazy else G.verify_sample
    got = PY.to_np(fn(h, x["logits"], x["draft_token"], x["parent"], w.temperature,
                      x["uniforms"], draft=x["draft"], draft_kind=G.SPEC_DRAFT_LOGITS))
    torch.cuda.synchronize()
    ref = PY.oracle_sample(orc, x["logits"], x["draft_token"], x["parent"], w.temperature,
                           x["uniforms"], x["draft"], G.SPEC_DRAFT_LOGITS)
    PY.compare_sample(got, ref)
    _clean(h, w.B)


@pytest.mark.parametrize("seed", [0, 1, 5, 17, 20, 28, 34, 45])
def test_fuzz_cases(h, orc, seed):
    import test_gpu_fuzz as F
    F.test_fuzz_against_oracle(h, orc, seed)


def test_kv_commit_case(h):
    import test_gpu_kv_commit as K
    from oracle import kv_commit as KO
    K.test_kv_commit_matches_oracle(h, "bf16", KO.FP8_E4M3, KO.HND, 128, "token")
    K.test_kv_commit_matches_oracle(h, "f32", KO.SAME, KO.NHD, 36, "tensor")
    K.test_kv_commit_fp8_quotients_at_rounding_boundaries(h, KO.FP8_E4M3)


def test_no_allocation_call(orc, dbg_lib):
    w = W.WORKLOADS["greedy_trie"].scaled(B=16, boost=20.0, seed=81)
    x = W.make(w, device=DEV)
    out = G.alloc_outputs(w.B, w.N, DEV)
    G.spec_verify_greedy_noalloc(x["logits"], x["draft_token"], x["parent"], out["accept_len"],
                                 out["out_tokens"], out["kv_commit"], out["bonus"],
                                 out["status"])
    torch.cuda.synchronize()
    PY.assert_exact(PY.to_np(out), orc.verify_greedy(PY.host(x["logits"]), x["tok_np"],
                                                     x["parent_np"]))


def test_inputs_corrupted_on_the_host_keep_their_codes(h, orc):
    """Data errors are not internal violations: a bad parent, an out-of-range token, a NaN
    row and a bad uniform give statuses 1-4 as in the release build, and the other requests
    match the oracle."""
    w = W.WORKLOADS["sampling_trie"].scaled(B=8, N=16, V=5000, boost=12.0, seed=83)
    x = W.make(w, device=DEV)
    par, tok = x["parent_np"].copy(), x["tok_np"].copy()
    par[1, 5] = 9                      # a parent after its child
    tok[2, 3] = w.V + 3                # a token outside the vocabulary
    logits = x["logits"].clone()
    logits[3, 0, 17] = float("nan")    # the root row, which every walk reads
    u = x["uniforms"].clone()
    u[4, 2] = 1.5                      # a uniform outside [0, 1)
    args = (logits, _to(tok), _to(par))
    g = PY.to_np(G.verify_greedy(h, *args))
    s = PY.to_np(G.verify_sample(h, *args, w.temperature, u))
    torch.cuda.synchronize()
    assert g["status"].tolist() == [0, 1, 2, 3, 0, 0, 0, 0]
    assert s["status"].tolist() == [0, 1, 2, 3, 4, 0, 0, 0]
    gref = orc.verify_greedy(PY.host(logits), tok, par)
    PY.assert_exact(g, gref)
    sref = orc.verify_sample(PY.host(logits), tok, par, w.temperature, u.cpu().numpy())
    PY.compare_sample(s, sref)
    _clean(h, w.B)


@pytest.mark.parametrize("value", [1, -3, 1000])
def test_corrupted_arrival_counter_is_reported(h, orc, value):
    """The greedy trie streams each row over 4 CTAs that count their arrivals. A counter
    that does not start at zero (set on the host before the launch) makes the row's pieces
    merge at the wrong arrival or never: the check turns exactly that request into
    SPEC_REQ_INTERNAL, the others match the oracle, and the next call is clean again."""
    w = W.WORKLOADS["greedy_trie"].scaled(boost=20.0, seed=84)
    with G.Handle(w.B, w.N, w.V, 0) as hs:
        x = W.make(w, device=DEV)
        ref = orc.verify_greedy(PY.host(x["logits"]), x["tok_np"], x["parent_np"])
        victim = 2
        G.spec_debug_inject_arrival(hs, victim * w.N + 0, value)
        got = PY.to_np(G.verify_greedy(hs, x["logits"], x["draft_token"], x["parent"]))
        words = G.spec_debug_words(hs, w.B).cpu().numpy()
        torch.cuda.synchronize()
        assert got["status"][victim] == G.SPEC_REQ_INTERNAL
        assert words[victim] & G.DBG_ARRIVAL
        assert got["accept_len"][victim] == 0 and got["bonus"][victim] == -1
        others = np.array([b for b in range(w.B) if b != victim])
        PY.assert_exact({k: v[others] for k, v in got.items()},
                        {k: v[others] for k, v in ref.items()})
        assert (np.delete(words, victim) == 0).all()
        again = PY.to_np(G.verify_greedy(hs, x["logits"], x["draft_token"], x["parent"]))
        torch.cuda.synchronize()
        PY.assert_exact(again, ref)
        _clean(hs, w.B)
