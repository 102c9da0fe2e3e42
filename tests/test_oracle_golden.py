"""The oracle against hand-worked examples (tests/golden/*.json, each citing its passage)."""
import pytest

import golden_io
from oracle import oracle as O


def run_oracle(orc, g):
    if g["op"] == "mask":
        anc, depth, status = orc.build_mask(g["parent"])
        return dict(anc=anc, depth=depth, status=status)
    if g["op"] == "greedy":
        return orc.verify_greedy(g["logits"], g["draft_token"], g["parent"])
    kind = {"probs_f32": O.DRAFT_PROBS_F32, "logits": O.DRAFT_LOGITS}.get(
        g.get("draft_kind"), O.DRAFT_POINT)
    return orc.verify_sample(g["logits"], g["draft_token"], g["parent"], g["temperature"],
                             g["uniforms"], draft=g.get("draft"), draft_kind=kind)


@pytest.mark.parametrize("name", golden_io.names())
def test_golden(orc, name):
    g = golden_io.load(name)
    assert golden_io.mismatches(g, run_oracle(orc, g)) == []


def test_goldens_present():
    assert len(golden_io.names()) >= 8
