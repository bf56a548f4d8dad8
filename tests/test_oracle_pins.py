"""The FP64 oracle against facts that do not come from the oracle (CPU only)."""
import pytest

import oracle_pins
from oracle import oracle


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.load())


# Planted mistakes: each mutant changes one step of the oracle (see the
# ORACLE_MUTANT cases in oracle/attn_oracle.c).  At least one pin must fail.
MUTANTS = {
    1: "sink dropped from the denominator",
    2: "GQA head mapping h % Hkv",
    3: "window keeps W+1 keys",
    4: "causal block aligned top-left",
    5: "in-page offset reversed",
    6: "k_scale ignored",
    7: "v_scale ignored",
    8: "E4M3 exponent bias 8",
    9: "last QK dimension dropped",
    10: "V read from the wrong KV head",
    11: "lse without ln Z",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m])
def test_pins_reject_mutant(mutant):
    o = oracle.load(mutant)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError) as e:  # noqa: PERF203
            failed.append(pin.__name__)
            del e
    assert failed, f"no pin caught mutant {mutant} ({MUTANTS[mutant]})"
