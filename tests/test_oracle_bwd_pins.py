"""The gradient oracle against what mathematics fixes (CPU only).

Every pin in ``oracle_pins_bwd`` must pass on the gradient oracle as built,
and each planted mistake (compiled from the same C source with
ORACLE_MUTANT=n) must fail at least one pin.
"""
import functools

import pytest

import oracle
from oracle_pins_bwd import ALL_PINS


@pytest.fixture(scope="module")
def bwd_lib():
    oracle.build_bwd()
    return oracle.load_bwd()


def _fns(lib, fwd_lib):
    return (functools.partial(oracle.attention_bwd, lib=lib, n_threads=2),
            functools.partial(oracle.attention, lib=fwd_lib, n_threads=2))


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin, bwd_lib, oracle_lib):
    assert bwd_lib.oracle_bwd_mutant_id() == 0
    pin(*_fns(bwd_lib, oracle_lib))


MUTANTS = {
    1: "scale dropped from dK",
    2: "sign of the D term",
    3: "q in place of dO in dV",
    4: "wrong heads summed into dK dV",
    5: "causal off by one",
    6: "dQ sign",
    7: "query offset sign",
    8: "window one key too wide",
    9: "softcap derivative dropped",
    10: "dropout left out of dV",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m].replace(" ", "_"))
def test_pins_catch_planted_mistake(mutant, tmp_path, oracle_lib):
    lib = oracle.load_bwd(oracle.build_bwd(mutant, str(tmp_path / f"liboracle_bwd_m{mutant}.so")))
    assert lib.oracle_bwd_mutant_id() == mutant
    grad, fwd = _fns(lib, oracle_lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(grad, fwd)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {mutant} ({MUTANTS[mutant]})"


def test_gradient_oracle_rejects_bad_arguments(bwd_lib):
    import numpy as np
    q = np.zeros((1, 3, 2, 4)); k = np.zeros((1, 2, 2, 4))
    with pytest.raises(ValueError):
        oracle.attention_bwd(q, k, k, q, 1.0, lib=bwd_lib)   # 3 % 2 != 0
