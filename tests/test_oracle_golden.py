"""The oracle still reproduces its stored tiny-workload record
(tests/golden/oracle_tiny.json, written by tests/golden/make_golden.py)."""
import json
import os

from tests.golden.make_golden import make

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_reproduces_golden_record():
    with open(os.path.join(HERE, "golden", "oracle_tiny.json")) as f:
        stored = json.load(f)
    assert make() == stored
