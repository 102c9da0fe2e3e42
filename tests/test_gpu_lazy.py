"""Lazy verification (only the rows the walk visits are read) against the oracle and against
the eager calls, through the C ABI (needs a GB300 and the built library)."""
import os

import numpy as np
import pytest
import torch

import golden_io
import parity as PY
from speculative_decoding_tree_mask_gb300 import binding as G
from speculative_decoding_tree_mask_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def h():
    G.load()
    with G.Handle(256, 64, 1 << 21, 0) as handle:
        yield handle


def _to(x):
    return torch.as_tensor(x).to(DEV).contiguous()


def lazy_greedy(h, logits, tok, parent):
    out = G.verify_greedy_lazy(h, logits, tok, parent)
    torch.cuda.synchronize()
    return PY.to_np(out)


def lazy_sample(h, logits, tok, parent, T, u, draft=None, kind=G.SPEC_DRAFT_POINT):
    out = G.verify_sample_lazy(h, logits, tok, parent, T, u, draft=draft, draft_kind=kind)
    torch.cuda.synchronize()
    return PY.to_np(out)


@pytest.mark.parametrize("name", golden_io.names())
def test_goldens_lazy(h, name):
    g = golden_io.load(name)
    if g["op"] == "mask":
        pytest.skip("the mask has no lazy form")
    if g["op"] == "greedy":
        got = lazy_greedy(h, _to(g["logits"]), _to(g["draft_token"]), _to(g["parent"]))
    else:
        kind = {"probs_f32": G.SPEC_DRAFT_PROBS_F32, "logits": G.SPEC_DRAFT_LOGITS}.get(
            g.get("draft_kind"), G.SPEC_DRAFT_POINT)
        draft = _to(g["draft"]) if "draft" in g else None
        got = lazy_sample(h, _to(g["logits"]), _to(g["draft_token"]), _to(g["parent"]),
                          g["temperature"], _to(g["uniforms"]), draft, kind)
    assert golden_io.mismatches(g, got) == []


@pytest.mark.parametrize("name,boost", [("tiny_chain", 0.0), ("greedy_trie", 8.0),
                                        ("greedy_trie", 40.0), ("large_tree", 30.0)])
def test_lazy_greedy_equals_eager_and_oracle(h, orc, name, boost):
    w = W.WORKLOADS[name].scaled(boost=boost) if boost else W.WORKLOADS[name]
    x = W.make(w, device=DEV)
    lz = lazy_greedy(h, x["logits"], x["draft_token"], x["parent"])
    eg = PY.gpu_greedy(h, x["logits"], x["draft_token"], x["parent"])
    for k in PY.KEYS:
        assert np.array_equal(lz[k], eg[k]), k
    ref = orc.verify_greedy(PY.host(x["logits"]), x["tok_np"], x["parent_np"],
                            nthreads=os.cpu_count() or 8)
    PY.assert_exact(lz, ref)


@pytest.mark.parametrize("dtype,V,offset", [("bf16", 9, 1), ("f32", 257, 1), ("bf16", 4097, 0),
                                            ("f32", 1000, 0)])
def test_lazy_greedy_ragged(h, orc, dtype, V, offset):
    w = W.WORKLOADS["greedy_trie"].scaled(B=5, N=9, V=V, dtype=dtype, boost=15.0, seed=V + offset)
    x = W.make(w, device=DEV)
    flat = torch.empty(w.B * w.N * V + offset, dtype=w.torch_dtype, device=DEV)
    logits = flat[offset:].view(w.B, w.N, V)
    logits.copy_(x["logits"])
    got = lazy_greedy(h, logits, x["draft_token"], x["parent"])
    ref = orc.verify_greedy(PY.host(x["logits"]), x["tok_np"], x["parent_np"])
    PY.assert_exact(got, ref)


def test_lazy_never_reads_rows_off_the_path(h, orc):
    w = W.WORKLOADS["greedy_trie"].scaled(B=16, V=5000, boost=30.0, seed=78)
    x = W.make(w, device=DEV)
    ref = orc.verify_greedy(PY.host(x["logits"]), x["tok_np"], x["parent_np"])
    logits = x["logits"].clone()
    u = x["uniforms"]
    for b in range(w.B):
        on_path = set(ref["kv_commit"][b][ref["kv_commit"][b] >= 0].tolist())
        for i in range(w.N):
            if i not in on_path:
                logits[b, i] = float("nan")
    got = lazy_greedy(h, logits, x["draft_token"], x["parent"])
    PY.assert_exact(got, ref)
    # sampling at a tiny temperature follows the same path and may not read other rows either
    s = lazy_sample(h, logits, x["draft_token"], x["parent"], 1e-4, u)
    assert (s["status"] == 0).all()


@pytest.mark.parametrize("T,boost", [(0.7, 8.0), (0.7, 30.0), (1.0, 12.0), (1.8, 20.0)])
def test_lazy_sample_point(h, orc, T, boost):
    w = W.WORKLOADS["sampling_trie"].scaled(temperature=T, boost=boost,
                                            seed=int(T * 100 + boost) + 1)
    x = W.make(w, device=DEV)
    got = lazy_sample(h, x["logits"], x["draft_token"], x["parent"], T, x["uniforms"])
    ref = PY.oracle_sample(orc, x["logits"], x["draft_token"], x["parent"], T, x["uniforms"])
    PY.compare_sample(got, ref)
    eg = PY.gpu_sample(h, x["logits"], x["draft_token"], x["parent"], T, x["uniforms"])
    keep = (ref["decision_margin"] >= PY.MARGIN) & (ref["cdf_margin"] >= PY.MARGIN)
    for k in PY.KEYS:
        assert np.array_equal(got[k][keep], eg[k][keep])


def test_lazy_sample_many_small_requests(h, orc):
    w = W.WORKLOADS["sampling_trie"].scaled(B=256, N=24, V=3001, dtype="f32", boost=6.0,
                                            sigma=1.5, temperature=1.0, seed=9)
    x = W.make(w, device=DEV)
    got = lazy_sample(h, x["logits"], x["draft_token"], x["parent"], 1.0, x["uniforms"])
    ref = PY.oracle_sample(orc, x["logits"], x["draft_token"], x["parent"], 1.0, x["uniforms"])
    PY.compare_sample(got, ref)
    assert got["accept_len"].max() >= 2


def test_lazy_sample_rejected_mass_resummed(h, orc):
    B, N, V = 8, 4, 151936
    logits = (3.0 * torch.randn((B, N, V), device=DEV)).to(torch.bfloat16)
    parent = np.tile(np.array([-1, 0, 0, 0], np.int32), (B, 1))
    tok = np.tile(np.array([0, 11, 22, 33], np.int32), (B, 1))
    logits[:, 0, 11] = 20.0
    logits[:, 0, 22] = 3.0
    u = torch.rand((B, N + 1), device=DEV)
    u[:, 1] = 0.99999
    got = lazy_sample(h, logits, _to(tok), _to(parent), 1.0, u)
    ref = PY.oracle_sample(orc, logits, _to(tok), _to(parent), 1.0, u)
    PY.compare_sample(got, ref)


def test_lazy_dense_chain_logits_and_probs(h, orc):
    w = W.WORKLOADS["dense_chain"]
    x = W.make(w, device=DEV)
    got = lazy_sample(h, x["logits"], x["draft_token"], x["parent"], 1.0, x["uniforms"],
                      x["draft"], G.SPEC_DRAFT_LOGITS)
    ref = PY.oracle_sample(orc, x["logits"], x["draft_token"], x["parent"], 1.0, x["uniforms"],
                           x["draft"], G.SPEC_DRAFT_LOGITS)
    PY.compare_sample(got, ref)
    w2 = W.WORKLOADS["dense_chain"].scaled(B=32, V=4103, dtype="f32", seed=5)
    x2 = W.make(w2, device=DEV)
    probs = torch.softmax(x2["draft"].float().cpu(), dim=-1).contiguous()
    probs[:, -1] = float("nan")
    got = lazy_sample(h, x2["logits"], x2["draft_token"], x2["parent"], 1.0, x2["uniforms"],
                      probs.to(DEV), G.SPEC_DRAFT_PROBS_F32)
    ref = PY.oracle_sample(orc, x2["logits"], x2["draft_token"], x2["parent"], 1.0,
                           x2["uniforms"], probs, G.SPEC_DRAFT_PROBS_F32)
    PY.compare_sample(got, ref)


def test_lazy_dense_tree(h, orc):
    rng = np.random.default_rng(9)
    B, N, V, T = 64, 12, 3000, 1.0
    parent = np.stack([W.random_trie(rng, N, 3, 4) for _ in range(B)])
    target = torch.randn((B, N, V), generator=torch.Generator().manual_seed(11))
    draft = target + 0.7 * torch.randn((B, N, V), generator=torch.Generator().manual_seed(12))
    probs = torch.softmax(draft / T, dim=-1)
    tok = np.zeros((B, N), np.int32)
    for b in range(B):
        for c in range(1, N):
            tok[b, c] = int(torch.multinomial(probs[b, parent[b, c]], 1,
                                              generator=torch.Generator().manual_seed(b * N + c)))
    u = torch.rand((B, N + 1), generator=torch.Generator().manual_seed(13))
    args = (_to(target), _to(tok), _to(parent), T, _to(u))
    got = lazy_sample(h, *args, _to(draft), G.SPEC_DRAFT_LOGITS)
    ref = PY.oracle_sample(orc, *args, draft, G.SPEC_DRAFT_LOGITS)
    PY.compare_sample(got, ref)


@pytest.mark.parametrize("boost", [8.0, 20.0])
def test_lazy_large_tree(h, orc, boost):
    """The large tree at the synthetic recipe's boost (walks stop at the root) and at boost 20
    (walks several levels deep): lazy sampling and lazy greedy against the oracle on all 256
    requests."""
    w = W.WORKLOADS["large_tree"].scaled(boost=boost)
    x = W.make(w, device=DEV)
    threads = os.cpu_count() or 8
    got = lazy_sample(h, x["logits"], x["draft_token"], x["parent"], w.temperature,
                      x["uniforms"])
    ref = PY.oracle_sample(orc, x["logits"], x["draft_token"], x["parent"], w.temperature,
                           x["uniforms"], nthreads=threads)
    PY.compare_sample(got, ref)
    lg = lazy_greedy(h, x["logits"], x["draft_token"], x["parent"])
    gref = orc.verify_greedy(PY.host(x["logits"]), x["tok_np"], x["parent_np"], nthreads=threads)
    PY.assert_exact(lg, gref)
    # the eager call differs only where float32 rounding of a sum decides
    eg = PY.gpu_sample(h, x["logits"], x["draft_token"], x["parent"], w.temperature,
                       x["uniforms"])
    agree = np.mean([np.array_equal(got["out_tokens"][b], eg["out_tokens"][b])
                     for b in range(w.B)])
    assert agree > 0.97, agree


def test_lazy_profiling_classes(h):
    w = W.WORKLOADS["sampling_trie"].scaled(B=4, N=8, V=20000, seed=3)
    x = W.make(w, device=DEV)
    G.spec_profile_begin(h)
    lazy_sample(h, x["logits"], x["draft_token"], x["parent"], 0.7, x["uniforms"])
    lazy_greedy(h, x["logits"], x["draft_token"], x["parent"])
    prof = G.spec_profile_end(h)
    assert prof["lazy_sample"][1] == 1 and prof["lazy_greedy"][1] == 1
    assert prof["row_stats"][1] == 0


def test_lazy_reads_pinned_host_logits(h, orc):
    w = W.WORKLOADS["sampling_trie"].scaled(B=16, V=20000, boost=12.0, seed=21)
    x = W.make(w, device=DEV)
    host = x["logits"].cpu().pin_memory()
    a = lazy_sample(h, host, x["draft_token"], x["parent"], 0.7, x["uniforms"])
    b = lazy_sample(h, x["logits"], x["draft_token"], x["parent"], 0.7, x["uniforms"])
    for k in PY.KEYS:
        assert np.array_equal(a[k], b[k]), k
    g1 = lazy_greedy(h, host, x["draft_token"], x["parent"])
    g2 = PY.gpu_greedy(h, x["logits"], x["draft_token"], x["parent"])
    for k in PY.KEYS:
        assert np.array_equal(g1[k], g2[k]), k


def test_lazy_refuses_pageable_host_logits(h):
    """A pageable host pointer is rejected by the library before any launch."""
    import ctypes
    w = W.WORKLOADS["sampling_trie"].scaled(B=2, N=4, V=64, seed=22)
    x = W.make(w, device=DEV)
    pageable = np.zeros((2, 4, 64), np.uint16)
    out = G.alloc_outputs(2, 4, DEV)
    lib = G.load()
    rc = lib.spec_verify_greedy_lazy(
        h.ptr, ctypes.c_void_p(pageable.ctypes.data), G.SPEC_BF16, 2, 4, 64,
        ctypes.c_void_p(x["draft_token"].data_ptr()), ctypes.c_void_p(x["parent"].data_ptr()),
        ctypes.c_void_p(out["accept_len"].data_ptr()),
        ctypes.c_void_p(out["out_tokens"].data_ptr()),
        ctypes.c_void_p(out["kv_commit"].data_ptr()), ctypes.c_void_p(out["bonus"].data_ptr()),
        ctypes.c_void_p(out["status"].data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == G.SPEC_ERR_ARG
