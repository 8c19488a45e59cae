"""The oracle against its recorded results on the seeded tiny workload
(tests/golden/oracle_tiny16.json, written by tests/golden/make_golden.py from
the oracle alone).  The pages print no worked example of the layer, so this is
a regression pin: it fails when the oracle's arithmetic changes, and such a
change must name, in its commit message, the passage or reading that
justifies it before the fixture is rewritten."""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def test_oracle_matches_recorded_tiny16(oracle_mod, synth_mod):
    with open(os.path.join(HERE, "golden", "oracle_tiny16.json")) as f:
        want = json.load(f)
    got = make_golden.fixture()
    for key, value in want.items():
        assert got[key] == value, key
