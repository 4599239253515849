"""The oracle reproduces its committed regression fixture bit for bit (a change to
its arithmetic must come with a regenerated fixture and a reason)."""
import json
import os

from tests.golden import make_golden


def test_oracle_matches_committed_fixture():
    with open(os.path.join(os.path.dirname(__file__), "golden", "oracle_small_bf16.json")) as f:
        want = json.load(f)
    got = make_golden.compute()
    for key in ("S", "R", "k", "y", "M_bits"):
        assert got[key] == want[key], key
