"""The oracle reproduces the stored outputs under tests/golden/ (written by
tests/golden/make_golden.py from the oracle alone).  The pages print no
worked example, so these files pin the oracle across machines and changes,
not against the pages."""
import json
import os
import sys

import numpy as np

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
sys.path.insert(0, HERE)
import make_golden  # noqa: E402


def test_tiny_matches_stored():
    rows = [ln.split() for ln in open(os.path.join(HERE, "tiny_rmsnorm_linear_bf16.txt"))
            if not ln.startswith("#")]
    stored = np.array([[int(v, 16) for v in r] for r in rows], np.uint16)
    assert np.array_equal(make_golden.tiny_case(), stored)


def test_small_w8a8_matches_stored():
    meta = json.load(open(os.path.join(HERE, "w8a8_T8_K256_N64.json")))
    r = make_golden.small_w8a8_case()
    assert make_golden.digest(r["q"]) == meta["q_sha256"]
    assert make_golden.digest(r["acc"]) == meta["acc_sha256"]
    assert make_golden.digest(r["out"]) == meta["out_sha256"]
    assert [float(v) for v in r["x_scale"]] == meta["x_scale"]
