"""The stored golden fixtures match the oracle (regression pin of the oracle;
the fixtures are written by tests/golden/make_golden.py from oracle/ only)."""
import json
import os

import numpy as np
import pytest

from tests.golden import make_golden

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("name,fn", [("quest_tiny", make_golden.quest_case),
                                     ("snapkv_tiny", make_golden.snapkv_case),
                                     ("h2o_tiny", make_golden.h2o_case)])
def test_fixture_matches_oracle(name, fn):
    with open(os.path.join(GOLDEN, name + ".json")) as f:
        stored = json.load(f)
    fresh = fn()
    for key, want in stored["expected"].items():
        got = fresh["expected"][key]
        if isinstance(want, list) and want and isinstance(np.asarray(want).flat[0], float):
            assert np.allclose(got, want, rtol=1e-12, atol=1e-12), key
        else:
            assert got == want, key
