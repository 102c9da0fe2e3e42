"""Loading and checking the hand-worked fixtures under tests/golden/."""
import glob
import json
import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _num(x):
    if isinstance(x, str):
        return {"nan": np.nan, "inf": np.inf, "-inf": -np.inf}[x]
    return x


def _arr(nested, dtype):
    def conv(v):
        return [conv(w) for w in v] if isinstance(v, list) else _num(v)
    return np.array(conv(nested), dtype=dtype)


def names():
    return sorted(os.path.splitext(os.path.basename(p))[0]
                  for p in glob.glob(os.path.join(GOLDEN_DIR, "*.json")))


def load(name):
    with open(os.path.join(GOLDEN_DIR, name + ".json")) as f:
        g = json.load(f)
    out = dict(g)
    out["parent"] = _arr(g["parent"], np.int32)
    if g["op"] != "mask":
        out["draft_token"] = _arr(g["draft_token"], np.int32)
        out["logits"] = _arr(g["logits"], np.float32)
        if "uniforms" in g:
            out["uniforms"] = _arr(g["uniforms"], np.float32)
        if "draft" in g:
            out["draft"] = _arr(g["draft"], np.float32)
    return out


def mismatches(g, got):
    """Compare a result dict against the golden's expected values; returns a list of text."""
    bad = []
    for key, want in g["expected"].items():
        want = np.array(want)
        have = np.asarray(got[key]).astype(np.int64)
        if key == "anc":
            have = np.asarray(got[key]).astype(np.uint64).astype(object)
            want = np.array(g["expected"][key], dtype=object)
        if have.shape != want.shape or not np.array_equal(have, want):
            bad.append(f"{g['name']}: {key} = {have.tolist()} expected {want.tolist()}")
    return bad
