"""Helpers that run one workload through the CUDA path and through the oracle and compare.

Bar (from the method's exactness claim): masks, argmax, accepted paths and greedy tokens are
bit-exact; in sampling mode decisions and sampled tokens are identical except for requests
whose decision margin or inverse-CDF margin is below 1e-6 in the oracle's float64 arithmetic
(those are counted and reported). The decision margin is |u - r(x)/q(x)|, which is never
below |u*q - r| (q <= 1), so the excluded set is a subset of the |u*q - r| < 1e-6 set.

How many decision-margin exclusions the inputs justify: every accept decision compares a
seeded uniform u, independent of the threshold r(x)/q(x), so it lands within 1e-6 of the
threshold with probability at most 2e-6. A request takes at most N - 1 decisions, so the count
over B requests is at most Poisson with mean lam = 2e-6 * B * (N - 1); the bound asserted is
the smallest k with P(count > k) < 1e-9 under that law (k = 4 for the large tree). Draws
within 1e-6 of a CDF boundary ("near-boundary") are not excluded and not bounded: with V in
the hundred thousands a token's CDF interval is often only a few 1e-6 wide, so such draws are
common; they must match in every output but the bonus, which must lie in the oracle's draw
window. Every comparison appends its counts to RECORDS, which the test session prints.
"""
import math
import os

import numpy as np
import torch

from oracle import oracle as O
from speculative_decoding_tree_mask_gb300 import binding as G
from speculative_decoding_tree_mask_gb300 import workloads as W

MARGIN = 1e-6
RECORDS = []   # one dict per sampling comparison: test, requests, excluded, near, bound


def margin_bound(requests: int, nodes: int, tail: float = 1e-9) -> int:
    """Smallest k with P(X > k) < tail for X ~ Poisson(2 * MARGIN * requests * (nodes - 1)),
    the law that bounds the number of requests with a decision within MARGIN of its
    threshold."""
    lam = 2.0 * MARGIN * requests * max(nodes - 1, 1)
    k, term = 0, math.exp(-lam)
    cdf = term
    while 1.0 - cdf >= tail:
        k += 1
        term *= lam / k
        cdf += term
    return k
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


def compare_sample(gpu, ref, rows=None, label=None, max_excluded=None):
    """Identity outside the margins. A request whose decision margin is below 1e-6 is
    excluded; one whose bonus draw lies within 1e-6 of a CDF boundary must still match in
    every output except the bonus, and its bonus must lie in the oracle's draw window (the
    tokens with mass whose CDF interval comes within 1e-6 * S of tau: the oracle's token, the
    one across the boundary, and any tokens of tiny mass in between). The number of
    exclusions must stay within margin_bound (or within max_excluded, where a test needs
    fewer). Records and returns (excluded, near-boundary) counts."""
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
    nodes = np.asarray(g["out_tokens"]).reshape(len(excl), -1).shape[1]
    bound = margin_bound(len(excl), nodes) if max_excluded is None else max_excluded
    test = label or os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    RECORDS.append(dict(test=test, requests=int(len(excl)), excluded=n, near=int(near.sum()),
                        bound=bound))
    assert n <= bound, f"{n} decision-margin cases of {len(excl)} (bound {bound})"
    return n, int(near.sum())
