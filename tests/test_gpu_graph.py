"""A whole verify step (tree mask, eager and lazy sampling verify) captured in one CUDA graph
and replayed on new inputs gives the results of direct calls: no call synchronises with the
host or allocates, so the step can be captured (the vLLM SCV page runs its mask computation
from captured graphs)."""
import numpy as np
import pytest
import torch

from speculative_decoding_tree_mask_gb300 import binding as G
from speculative_decoding_tree_mask_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
KEYS = ("accept_len", "out_tokens", "kv_commit", "bonus", "status")


def test_verify_step_replays_from_a_cuda_graph():
    G.load()
    w = W.WORKLOADS["sampling_trie"].scaled(B=8, V=20000, boost=12.0)
    h = G.Handle(w.B, w.N, w.V, 0)
    x = W.make(w, device=DEV, seed=1)
    static = {k: x[k].clone() for k in ("logits", "draft_token", "parent", "uniforms")}
    mask = G.build_tree_mask(h, static["parent"])
    eager = G.alloc_outputs(w.B, w.N, DEV)
    lazy = G.alloc_outputs(w.B, w.N, DEV)

    def step():
        G.spec_build_tree_mask(h, static["parent"], mask["anc_mask"], mask["depth"],
                               mask["status"])
        G.verify_sample(h, static["logits"], static["draft_token"], static["parent"], 0.7,
                        static["uniforms"], out=eager)
        G.verify_sample_lazy(h, static["logits"], static["draft_token"], static["parent"], 0.7,
                             static["uniforms"], out=lazy)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (2, 3, 4):
        y = W.make(w, device=DEV, seed=seed)
        for k in static:
            static[k].copy_(y[k])
        graph.replay()
        torch.cuda.synchronize()
        got_e = {k: v.clone() for k, v in eager.items()}
        got_l = {k: v.clone() for k, v in lazy.items()}
        got_m = {k: v.clone() for k, v in mask.items()}
        ref_e = G.verify_sample(h, y["logits"], y["draft_token"], y["parent"], 0.7, y["uniforms"])
        ref_l = G.verify_sample_lazy(h, y["logits"], y["draft_token"], y["parent"], 0.7,
                                     y["uniforms"])
        ref_m = G.build_tree_mask(h, y["parent"])
        torch.cuda.synchronize()
        for k in KEYS:
            assert torch.equal(got_e[k], ref_e[k]), k
            assert torch.equal(got_l[k], ref_l[k]), k
        for k in ref_m:
            assert torch.equal(got_m[k], ref_m[k]), k
    h.close()
