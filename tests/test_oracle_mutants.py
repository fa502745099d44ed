"""Plant plausible mistakes in copies of the oracle (compiled with
-DORC_MUTANT=k, CPU only) and require the pins to catch every one:
  1 wrong e4m3 maximum in the scale (amax/447)
  2 reciprocal multiply x*(448/amax) instead of x/s
  3 ties rounded away from zero in the encoder
  4 weight-scale grid read transposed
  5 last K chunk dropped from the GEMM
  6 bias subtracted instead of added
  7 silu with the exponent's sign flipped
  8 MoE combine dropping the last routed expert
  9 MoE dispatch taking the scales of the wrong row
 10 router ignoring the bias in the selection
 11 router gate values not normalised
 12 routing tables with tokens in reverse order within an expert
 13 column quantisation leaving a block's last row out of the amax
 14 dgrad reading the weight's block grid as if stored transposed
 15 wgrad dropping a ragged last block of tokens
 16 power-of-two scales rounded down (the top codes saturate)
"""
import pytest

from oracle import Oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 16])
def test_mutant_is_caught(mutant):
    o = Oracle(mutant)
    assert o.lib.orc_mutant_id() == mutant
    caught = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"
