"""The oracle still reproduces the fixture written by tests/golden/make_golden.py."""
import json
import os

import numpy as np

import oracle
from tests.golden.make_golden import cases

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_matches_its_regression_fixture():
    with open(os.path.join(HERE, "oracle_regression.json")) as f:
        fx = json.load(f)
    got = {name: U for name, U in cases()}
    for case in fx["cases"]:
        U = got[case["name"]]
        assert list(U.shape) == case["shape"]
        want = np.array([int(h, 16) for h in case["O_bf16_hex"].split()], dtype=np.uint16)
        assert np.array_equal(oracle.bf16_rne(oracle.ns(U, steps=5)).ravel(), want)
