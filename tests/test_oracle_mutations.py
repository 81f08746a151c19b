"""Every planted mistake in the oracle fails at least one pin.

Each mutation is a build of the oracle with one plausible error compiled in
(ORACLE_MUTATION in dattn_oracle.cpp): an off-by-one ring slot, a dropped new
token, a wrong KV-head map, a skipped gate, a RoPE sign flip, adjacent RoPE
pairs, frequencies over the wrong width, a wrong score scale, a tree depth off
by one, a missing tree mask, a page offset off by one, sigmoid(-g), values
taken from keys, truncation instead of rounding, quarter turns of the RoPE
phase taken the wrong way, an uncentred phase remainder, the K entry rounded
from the fp64-rounded sum instead of the exact one, a ring append slot off by
one, the QK-norm eps outside the root, the QK-norm sum of squares not divided
by D, a ring verify row that keeps the entries its path pushed out, a commit
that takes the first nodes instead of the accepted path's, prefill positions
shifted by one, E4M3 rounding by truncation, the fp8 K scale dropped. If one
of them passed every
pin, the pins would not be sharp enough to trust the oracle.
"""
import pytest

import oracle as oracle_pkg
from oracle_pins import ALL_PINS

MUTATIONS = list(range(1, 26))


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_mutation_is_caught(mutation):
    o = oracle_pkg.Oracle(mutation)
    assert o.lib.oracle_mutation() == mutation
    caught = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"mutation {mutation} passed every pin"
