"""The stored schedule fixtures still equal what the oracle produces (regression guard)."""

import os

import pytest

from oracle import schedule

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_fixture(name):
    meta = {}
    rows = []
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            if line.startswith("#"):
                for tok in line[1:].split():
                    if "=" in tok:
                        k, v = tok.split("=")
                        meta[k] = int(v)
                continue
            rows.append(tuple(int(x) for x in line.split()))
    return meta, rows


@pytest.mark.parametrize("name", sorted(n for n in os.listdir(HERE) if n.startswith("schedule_")))
def test_fixture_matches_oracle(name):
    meta, rows = load_fixture(name)
    want = schedule.enumerate_schedule(meta["m_blocks"], meta["n_blocks"], meta["workers"], meta["group"])
    assert rows == want
