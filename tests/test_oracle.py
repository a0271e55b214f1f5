"""The CPU oracle against its pins, and each planted mistake against the same pins."""
import pytest

import oracle
from oracle_pins import PINS

MUTANTS = {
    1: "query head mapped to kv head hq % Hkv",
    2: "scale dropped",
    3: "newest key dropped",
    4: "verify row sees one future token",
    5: "lse without its max term",
    6: "value rows from the neighbouring kv head",
    7: "merge without rescaling partials",
    8: "partials normalised before the merge",
    9: "cache read as [D][Smax] per head",
    10: "append writes one row late",
    11: "append does not advance seq_lens",
    12: "decode reads one row past seq_len",
    13: "bf16 bits read as IEEE half",
    14: "rotary pairs turned the wrong way",
    15: "rotary pairs taken as neighbours (2i, 2i+1)",
    16: "acceptance ratio inverted (q/p)",
    17: "residual taken as max(0, q - p)",
    18: "greedy compares with the draft's argmax",
    19: "int8 scale from a full-scale code of 128",
    20: "int8 codes truncated instead of rounded",
}


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(orc, pin):
    pin(orc)


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=[f"m{k}" for k in sorted(MUTANTS)])
def test_planted_mistake_is_caught(mutant):
    mut = oracle.load(mutant)
    assert mut.mutant == mutant
    failed = []
    for pin in PINS:
        try:
            pin(mut)
        except Exception:  # noqa: BLE001 - any failure counts as caught
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {mutant} ({MUTANTS[mutant]})"
