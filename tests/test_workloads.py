"""The seeded input generators (host logic only, no verification arithmetic)."""
import numpy as np
import pytest

from speculative_decoding_tree_mask_gb300 import workloads as W


@pytest.mark.parametrize("V", [1, 2, 3, 8, 9, 255, 1000])
@pytest.mark.parametrize("N", [1, 2, 9, 33, 64])
def test_trees_and_tokens_any_vocab(V, N):
    rng = np.random.default_rng(V * 100 + N)
    for _ in range(4):
        par = W.random_trie(rng, N, 10, 6)
        assert par[0] == -1 and all(0 <= par[i] < i for i in range(1, N))
        tok = W.child_tokens(rng, par, V)
        assert ((tok >= 0) & (tok < V)).all()
        for node in range(N):
            kids = [c for c in range(N) if c and par[c] == node]
            toks = [int(tok[c]) for c in kids]
            assert len(set(toks)) == min(len(toks), V)


@pytest.mark.parametrize("name", sorted(W.WORKLOADS))
def test_workloads_small_scale(name):
    w = W.WORKLOADS[name].scaled(B=3, V=64 if W.WORKLOADS[name].V > 64 else W.WORKLOADS[name].V)
    x = W.make(w)
    assert x["logits"].shape == (w.B, w.N, w.V)
    assert x["uniforms"].shape == (w.B, w.N + 1)
    assert float(x["uniforms"].min()) >= 0 and float(x["uniforms"].max()) < 1
    if w.mode == "dense":
        assert x["draft"].shape == x["logits"].shape
    for b in range(w.B):
        assert x["parent_np"][b, 0] == -1


def test_depth_limit_respected():
    rng = np.random.default_rng(0)
    for _ in range(20):
        par = W.random_trie(rng, 64, 10, 6)
        depth = [0] * 64
        for i in range(1, 64):
            depth[i] = depth[par[i]] + 1
        assert max(depth) <= 10


@pytest.mark.parametrize("V,dtype,offset", [(v, d, o) for v in [1, 3, 8, 9, 255, 256, 257, 1000,
                                                                  4097]
                                            for d in ["bf16", "f32"] for o in [0, 1]])
def test_gpu_test_inputs_build_on_cpu(V, dtype, offset):
    """The inputs of the ragged-vocabulary GPU test build on the host."""
    w = W.WORKLOADS["greedy_trie"].scaled(B=5, N=9, V=V, dtype=dtype, boost=15.0, seed=V + offset)
    x = W.make(w)
    assert x["logits"].shape == (5, 9, V)
