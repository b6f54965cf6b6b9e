"""The oracle against what mathematics and the pages fix (CPU only).

Every pin in ``oracle_pins`` must pass on the oracle as built, and each
planted mistake (compiled from the same C source with ORACLE_MUTANT=n) must
fail at least one pin -- evidence that the pins would notice such an error.
"""
import functools

import pytest

import oracle
from oracle_pins import ALL_PINS, GENERATOR_PINS


def _attn(lib):
    return functools.partial(oracle.attention, lib=lib, n_threads=2)


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin, oracle_lib):
    assert oracle_lib.oracle_mutant_id() == 0
    pin(_attn(oracle_lib))


MUTANTS = {
    1: "scale dropped",
    2: "wrong GQA head map",
    3: "causal off by one",
    4: "L without the max",
    5: "q and k roles swapped",
    6: "mask scaled with the scores",
    7: "bool polarity flipped",
    8: "no division by l",
    9: "softcap not multiplied back",
    10: "query offset sign",
    11: "window one key too wide",
    12: "dropout keep test inverted",
    13: "dropout weights not rescaled",
    14: "Philox key not raised between rounds",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m].replace(" ", "_"))
def test_pins_catch_planted_mistake(mutant, tmp_path):
    lib = oracle.load(oracle.build(mutant, str(tmp_path / f"liboracle_m{mutant}.so")))
    assert lib.oracle_mutant_id() == mutant
    attn = _attn(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(attn)
        except AssertionError:
            caught.append(pin.__name__)
    for pin in GENERATOR_PINS if not caught else ():
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {mutant} ({MUTANTS[mutant]})"


@pytest.mark.parametrize("pin", GENERATOR_PINS, ids=lambda p: p.__name__)
def test_generator_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_oracle_rejects_bad_arguments(oracle_lib):
    import numpy as np
    q = np.zeros((1, 3, 2, 4)); k = np.zeros((1, 2, 2, 4))
    with pytest.raises(ValueError):
        oracle.attention(q, k, k, 1.0, lib=oracle_lib)   # 3 % 2 != 0
