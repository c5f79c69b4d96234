"""Planted mistakes in the oracle must fail at least one pin (CPU only).

Each mutant is sv_oracle.c rebuilt with -DSVO_MUTANT=n, which plants one
plausible mistake: the residual over raw logits (as the C++ scheduler snippet
of the deferred-speculation page has it), a strict accept test, no bonus
token, no temperature on the draft row, '>=' in the inverse CDF, resampling
from the wrong row, swapped residual operands, no max shift in the softmax, a
dropped softmax term, a greedy tie broken to the last index, a draft sample
without the temperature, a ring slot without the sink offset, a KV commit
that drops the last emitted token's entry, a draft window start not aligned
to a block, a block-table clone not zeroed past `needed`, a token-tree
sibling tested against the target row instead of the current residual, and a
token-tree residual that restarts from the target row at every rejection.
"""
import pytest

import oracle
import oracle_pins

MUTANTS = {
    1: "residual over raw logits",
    2: "strict accept test u < r",
    3: "no bonus token",
    4: "temperature not applied to the draft row",
    5: "inverse CDF with >=",
    6: "resample from the row after the rejection",
    7: "residual operands swapped",
    8: "softmax without the max shift",
    9: "softmax sum drops the last term",
    10: "greedy tie goes to the last index",
    11: "draft sample ignores the temperature",
    12: "ring slot without the sink offset",
    13: "KV commit drops the last emitted token's entry",
    14: "draft window start not block-aligned",
    15: "block-table clone not zeroed past needed",
    16: "tree sibling tested against P_t instead of the residual",
    17: "tree residual restarts from P_t at every rejection",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: f"m{m}")
def test_mutant_is_caught(mutant, tmp_path):
    path = oracle.compile_oracle(str(tmp_path / f"libsvoracle_m{mutant}.so"), mutant=mutant)
    lib = oracle.load(path)
    assert lib.svo_mutant_id() == mutant
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except Exception as e:  # noqa: BLE001 - any failure counts as caught
            caught.append((pin.__name__, repr(e)[:120]))
            break
    assert caught, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"
