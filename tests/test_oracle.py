"""The CPU oracle against its pins, and mutants of it against the same pins."""

import json
import os

import numpy as np
import pytest

import oracle
from tests import oracle_pins as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)


# Each mutant plants one plausible mistake in the oracle source (see the
# ORACLE_MUTANT switch in topk_oracle.cpp); at least one pin must catch it.
MUTANTS = {
    1: "signed zeros compared as equal",
    2: "ties go to the larger index",
    3: "ascending value order",
    4: "per-row lengths ignored",
    5: "padding index 0 instead of -1",
    6: "off-by-one on rows shorter than k",
    7: "row stride ignored",
    8: "-inf dropped from the selection",
    9: "+inf clamped to the largest finite value",
    10: "block pool: a block scored by its first value",
    11: "block pool: the oldest blocks pinned",
    12: "block pool: ties between blocks to the larger index",
    13: "block pool: the short last block dropped",
    14: "block pool: pinned blocks also compete for the free places",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m])
def test_pins_catch_mutant(mutant):
    orc = oracle.load(mutant)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {mutant}: {MUTANTS[mutant]}"


def test_multithreaded_matches_single(oracle_lib):
    rng = np.random.default_rng(21)
    x = rng.standard_normal((9, 5000)).astype(np.float32)
    lengths = rng.integers(0, 5001, size=9).astype(np.int32)
    a = oracle_lib.topk(x, 300, lengths=lengths, nthreads=1)
    b = oracle_lib.topk(x, 300, lengths=lengths, nthreads=4)
    assert a[2] == b[2] == 0
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[0].view(np.uint32), b[0].view(np.uint32))


def _harmonic(m):
    return sum(1.0 / j for j in range(1, m + 1))


def test_survivor_bound_reading():
    """The printed ~29,000 ceiling fixes the tray reading T = k + 2 blocks."""
    g = json.load(open(os.path.join(GOLDEN, "survivor_bound.json")))
    m = g["n"] // g["block"]
    T = g["k"] + 2 * g["block"]
    bound = 1.5 * T * _harmonic(m)
    # "29,000" is given to two significant digits
    assert abs(bound - g["printed_bound"]) < 500, bound
    assert bound / g["n"] < g["printed_fraction_under"]
    # the neighbouring readings miss the printed figure
    for T_alt in (g["k"], g["k"] + g["block"], 2 * g["k"] + 2 * g["block"]):
        assert abs(1.5 * T_alt * _harmonic(m) - g["printed_bound"]) > 2500
