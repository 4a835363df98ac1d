"""The CPU oracle against its pins (values printed on the pages, closed forms,
invariants, a library attention routine, brute force)."""
import pytest

import oracle
from tests import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("name", sorted(oracle_pins.PINS))
def test_pin(orc, name):
    oracle_pins.PINS[name](orc)


def test_empty_sequence_reads_nothing(orc):
    """Reading (pages silent): attention over zero keys yields zeros."""
    import numpy as np
    q = np.zeros((1, 2, 8), np.uint16)
    pool = np.zeros((2, 2, 1, 4, 8), np.uint16)
    out = orc.paged_decode(q, pool, oracle.dense_geom(2, 1, 4, 8), [[-1]], [0], 2, 0.5)
    assert out.shape == (1, 2, 8) and not out.any()
