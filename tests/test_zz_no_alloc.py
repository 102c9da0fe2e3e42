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

import parity as PY
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


def test_noalloc_greedy_equals_handle_path_on_consecutive_calls(orc):
    Build.build()
    torch.cuda.set_device(0)
    cases = [
        # full scratch capacity (256 x 64 rows), small vocabulary, deep accepted paths
        W.WORKLOADS["large_tree"].scaled(V=1000, boost=40.0, seed=71),
        # the greedy trie at its real vocabulary, fewer rows than the first call left behind
        W.WORKLOADS["greedy_trie"].scaled(B=16, boost=20.0, seed=72),
    ]
    with G.Handle(256, 64, 1 << 21, 0) as h:
        for i, w in enumerate(cases):
            assert w.B * w.N <= G.SPEC_NOALLOC_MAX_ROWS
            x = W.make(w, device=DEV)
            # request 1 must fail with status 3: NaN in its root row, which every walk reads
            x["logits"][1, 0, 5] = float("nan")
            ref = G.verify_greedy(h, x["logits"], x["draft_token"], x["parent"])
            got = _noalloc(x)
            torch.cuda.synchronize()
            for k in KEYS:
                assert torch.equal(got[k], ref[k]), k
            assert int(got["status"][1]) == G.SPEC_REQ_BAD_ROW
            assert int(got["accept_len"][1]) == 0 and int(got["bonus"][1]) == -1
            assert int(got["accept_len"].max()) >= 1
            if i == 1:   # the second call against the oracle itself, request by request
                oref = orc.verify_greedy(PY.host(x["logits"]), x["tok_np"], x["parent_np"],
                                         nthreads=8)
                PY.assert_exact(PY.to_np(got), oref)


def test_noalloc_refuses_more_rows_than_its_scratch():
    Build.build()
    w = W.WORKLOADS["large_tree"].scaled(B=257, V=16, boost=0.0, seed=73)
    x = W.make(w, device=DEV)
    with pytest.raises(G.SpecError) as e:
        _noalloc(x)
    assert e.value.code == G.SPEC_ERR_ARG


def test_noalloc_refuses_logits_not_on_the_current_device():
    """Logits the current GPU cannot stream (here: pageable host memory) are refused before
    any launch, so a caller's mistake cannot turn into a kernel reading a foreign address."""
    import ctypes
    Build.build()
    w = W.WORKLOADS["greedy_trie"].scaled(B=2, N=4, V=64, seed=74)
    x = W.make(w, device=DEV)
    pageable = np.zeros((2, 4, 64), np.uint16)
    out = G.alloc_outputs(2, 4, DEV)
    fn = G.load().spec_verify_greedy_noalloc
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    fn.argtypes = [P, i32, i32, i32, i64, P, P, P, P, P, P, P, P]
    rc = fn(ctypes.c_void_p(pageable.ctypes.data), G.SPEC_BF16, 2, 4, 64,
            ctypes.c_void_p(x["draft_token"].data_ptr()), ctypes.c_void_p(x["parent"].data_ptr()),
            *[ctypes.c_void_p(out[k].data_ptr()) for k in KEYS],
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == G.SPEC_ERR_ARG
