"""The greedy entry point that allocates no device memory (spec_verify_greedy_noalloc).

Some callers cannot call cudaMalloc: plugins inside an engine that owns all device memory and
hands a kernel only its tensors, or latency-critical loops that cannot take cudaMalloc's
implicit device synchronisation. For them the library offers a greedy verify whose per-row
scratch is a static device array. This file checks, through the C ABI, that it returns exactly
what the handle-based spec_verify_greedy returns, on two calls in a row (the second call
finds the first call's leftovers in the shared array), and that requests beyond its fixed
capacity are refused. It runs last so that a failure here leaves every other test run.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_tree_mask_gb300 import binding as G
from speculative_decoding_tree_mask_gb300 import build as Build
from speculative_decoding_tree_mask_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
KEYS = ("accept_len", "out_tokens", "kv_commit", "bonus", "status")


def _noalloc(x):
    B, N, _ = x["logits"].shape
    out = G.alloc_outputs(B, N, DEV)
    G.spec_verify_greedy_noalloc(x["logits"], x["draft_token"], x["parent"], out["accept_len"],
                                 out["out_tokens"], out["kv_commit"], out["bonus"],
                                 out["status"])
    return out


def test_noalloc_greedy_equals_handle_path_on_consecutive_calls():
    Build.build()
    torch.cuda.set_device(0)
    cases = [
        # full scratch capacity (256 x 64 rows), small vocabulary, deep accepted paths
        W.WORKLOADS["large_tree"].scaled(V=1000, boost=40.0, seed=71),
        # the greedy trie at its real vocabulary, fewer rows than the first call left behind
        W.WORKLOADS["greedy_trie"].scaled(B=16, boost=20.0, seed=72),
    ]
    with G.Handle(256, 64, 1 << 21, 0) as h:
        for w in cases:
            assert w.B * w.N <= G.SPEC_NOALLOC_MAX_ROWS
            x = W.make(w, device=DEV)
            x["logits"][1, 3] = float("nan")           # a request that must fail with status 3
            ref = G.verify_greedy(h, x["logits"], x["draft_token"], x["parent"])
            got = _noalloc(x)
            torch.cuda.synchronize()
            for k in KEYS:
                assert torch.equal(got[k], ref[k]), k
            assert int(got["accept_len"].max()) >= 1


def test_noalloc_refuses_more_rows_than_its_scratch():
    Build.build()
    w = W.WORKLOADS["large_tree"].scaled(B=257, V=16, boost=0.0, seed=73)
    x = W.make(w, device=DEV)
    with pytest.raises(G.SpecError) as e:
        _noalloc(x)
    assert e.value.code == G.SPEC_ERR_ARG
