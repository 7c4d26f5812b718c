"""Each planted mistake in the oracle (ORACLE_MUTANT=n, CPU only) must be
caught by at least one pin, which shows the pins are not vacuous."""
import os

import pytest

import oracle
import oracle_pins

# mutant id -> the pins expected to catch it
MUTANTS = {
    1: ["combine_closed_forms", "combine_error_bound", "combine_exact"],  # last k term dropped
    2: ["combine_closed_forms", "combine_error_bound", "combine_exact"],  # weight index reversed
    3: ["layout_hand", "layout_bruteforce", "layout_random"],  # unstable order
    4: ["layout_hand", "layout_random"],  # off-by-one offsets
    5: ["dispatch"],  # wrong source row
    6: ["bf16"],  # truncating conversion
    7: ["combine_closed_forms", "combine_error_bound"],  # sign error in the chain
    8: ["pipeline"],  # min instead of max
    9: ["combine_exact"],  # multiply and add rounded separately
    10: ["combine_exact"],  # k descending
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, mutant):
    path = oracle.build(os.path.join(tmp_path, f"libmut{mutant}.so"), mutant=mutant)
    o = oracle.Oracle(oracle.load(path))
    caught = []
    for name in MUTANTS[mutant]:
        try:
            oracle_pins.ALL_CHECKS[name](o)
        except AssertionError:
            caught.append(name)
    assert caught, f"mutant {mutant} passed every pin in {MUTANTS[mutant]}"
