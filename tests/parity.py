"""Helpers that run one workload through the CUDA path and through the oracle and compare.

Bar (from the method's exactness claim): masks, argmax, accepted paths and greedy tokens are
bit-exact; in sampling mode decisions and sampled tokens are identical except for requests
whose decision margin or inverse-CDF margin is below 1e-6 in the oracle's float64 arithmetic
(those are excluded and counted). The decision margin is |u - r(x)/q(x)|, which is never below
|u*q - r| (q <= 1), so the excluded set is a subset of the |u*q - r| < 1e-6 set.
"""
import numpy as np
import torch

from oracle import oracle as O
from speculative_decoding_tree_mask_gb300 import binding as G
from speculative_decoding_tree_mask_gb300 import workloads as W

MARGIN = 1e-6
KEYS = ("accept_len", "out_tokens", "kv_commit", "bonus", "status")
ORACLE_KIND = {G.SPEC_DRAFT_POINT: O.DRAFT_POINT, G.SPEC_DRAFT_PROBS_F32: O.DRAFT_PROBS_F32,
               G.SPEC_DRAFT_LOGITS: O.DRAFT_LOGITS}


def to_np(d):
    return {k: v.cpu().numpy() for k, v in d.items()}


def host(t):
    return W.host_logits(t)


def gpu_greedy(h, logits, tok, parent):
    out = G.verify_greedy(h, logits, tok, parent)
    torch.cuda.synchronize()
    return to_np(out)


def gpu_sample(h, logits, tok, parent, T, u, draft=None, kind=G.SPEC_DRAFT_POINT):
    out = G.verify_sample(h, logits, tok, parent, T, u, draft=draft, draft_kind=kind)
    torch.cuda.synchronize()
    return to_np(out)


def oracle_sample(orc, logits, tok, parent, T, u, draft=None, kind=G.SPEC_DRAFT_POINT,
                  nthreads=8):
    d = None if draft is None else host(draft)
    return orc.verify_sample(host(logits), tok.cpu().numpy(), parent.cpu().numpy(), T,
                             u.cpu().numpy(), draft=d, draft_kind=ORACLE_KIND[kind],
                             nthreads=nthreads)


def assert_exact(gpu, ref, rows=None):
    for k in KEYS:
        a, b = gpu[k], ref[k]
        if rows is not None:
            a = a[rows]
        if not np.array_equal(a, b):
            bad = np.argwhere(np.asarray(a != b).reshape(len(a), -1).any(1)).ravel()[:5]
            raise AssertionError(f"{k} differs at requests {bad.tolist()}: gpu "
                                 f"{a[bad].tolist()} oracle {b[bad].tolist()}")


def compare_sample(gpu, ref, rows=None, max_excluded_frac=0.10):
    """Identity outside the margins. A request whose decision margin is below 1e-6 is
    excluded; one whose bonus draw lies within 1e-6 of a CDF boundary must still match in
    every output except the bonus, and its bonus must lie in the oracle's draw window (the
    tokens with mass whose CDF interval comes within 1e-6 * S of tau: the oracle's token, the
    one across the boundary, and any tokens of tiny mass in between). Returns (excluded,
    near-boundary) counts."""
    g = {k: (gpu[k][rows] if rows is not None else gpu[k]) for k in KEYS}
    excl = ref["decision_margin"] < MARGIN
    near = (ref["cdf_margin"] < MARGIN) & ~excl
    keep = ~excl
    L = g["accept_len"]
    for k in KEYS:
        a, b = g[k].copy(), ref[k].copy()
        if k == "bonus":
            a, b = a[keep & ~near], b[keep & ~near]
        elif k == "out_tokens":
            idx = np.nonzero(near)[0]
            a[idx, L[idx]] = b[idx, L[idx]]        # the bonus slot, checked below
            a, b = a[keep], b[keep]
        else:
            a, b = a[keep], b[keep]
        if not np.array_equal(a, b):
            bad = np.argwhere(np.asarray(a != b).reshape(len(a), -1).any(1)).ravel()[:5]
            raise AssertionError(f"{k} differs at kept requests {bad.tolist()}: gpu "
                                 f"{a[bad].tolist()} oracle {b[bad].tolist()}")
    for i in np.nonzero(near)[0]:
        gb = int(g["bonus"][i])
        assert int(ref["cdf_lo"][i]) <= gb <= int(ref["cdf_hi"][i]), \
            (i, gb, int(ref["bonus"][i]), int(ref["cdf_lo"][i]), int(ref["cdf_hi"][i]))
        assert g["out_tokens"][i, L[i]] == gb
    n = int(excl.sum())
    assert n <= max(1, max_excluded_frac * len(excl)), f"{n} decision-margin cases of {len(excl)}"
    return n, int(near.sum())
