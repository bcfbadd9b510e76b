"""The CPU oracle against its pins (closed forms, invariants, brute force,
library routines for the special cases, hand-enumerated BeamPath chains)."""

import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_oracle_rejects_bad_parent(orc):
    inp = pins.tiny_inputs()
    inp["beam_path"][0, 2, 1] = 4          # widths[1] == 4: out of range
    with pytest.raises(ValueError):
        orc.decode_attn(inp, 2)
    with pytest.raises(ValueError):
        orc.ancestors(inp, 2)


def test_oracle_threads_do_not_change_results(orc):
    inp = pins.tiny_inputs()
    a = orc.decode_attn(inp, 2, num_threads=1)
    b = orc.decode_attn(inp, 2, num_threads=4)
    for x, y in zip(a, b):
        assert (x == y).all()
