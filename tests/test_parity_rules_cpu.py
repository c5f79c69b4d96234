"""The parity rule for flagged near-ties (tests/gpu_util.check_valid_draw),
checked on the CPU against the oracle's own results: every request the
oracle returns is a valid draw under the rule, and planted wrong results
are not (a token outside u's CDF interval, an accepted count that moved at
a position far from its ratio, outputs out of the rule's shape)."""
import numpy as np
import pytest

import oracle
from gpu_util import check_valid_draw
from speculative_decoding_verification_09_gb300 import synth


@pytest.fixture(scope="module")
def case():
    cfg = synth.custom_config(24, 3, 600, "f32", "normal", temp=0.9, sigma_noise=1.0)
    inp = synth.make_inputs(cfg, seed=123)
    ref = oracle.verify(inp.Lt, inp.Ld, inp.x, inp.u_acc, inp.u_res, inp.temp, inp.dtype)
    assert np.all((ref["flags"] & oracle.INVALID_ANY) == 0)
    return inp, ref


def test_oracle_results_are_valid_draws(case):
    inp, ref = case
    for b in range(inp.B):
        check_valid_draw(inp, ref, ref, b)


def test_wrong_token_is_rejected(case):
    inp, ref = case
    b = 0
    k = int(ref["n"][b])
    got = {k_: v.copy() for k_, v in ref.items()}
    # the neighbour with mass whose interval is furthest from u
    got["tokens"][b, k] = (int(ref["tokens"][b, k]) + inp.V // 2) % inp.V
    with pytest.raises(AssertionError):
        check_valid_draw(inp, got, ref, b)


def test_moved_count_far_from_its_ratio_is_rejected(case):
    inp, ref = case
    g = inp.gamma
    for b in range(inp.B):
        k = int(ref["n"][b])
        if k < g:
            pt, pd = float(ref["pt"][b, k]), float(ref["pd"][b, k])
            r = 1.0 if pd == 0.0 else min(1.0, pt / pd)
            if abs(float(inp.u_acc[b, k]) - r) > 1e-3:
                got = {k_: v.copy() for k_, v in ref.items()}
                got["n"][b] = k + 1  # accept the rejected draft
                got["tokens"][b, :] = -1
                got["tokens"][b, :k + 1] = inp.x[b, :k + 1]
                got["tokens"][b, k + 1] = ref["tokens"][b, k]
                with pytest.raises(AssertionError):
                    check_valid_draw(inp, got, ref, b)
                return
    pytest.skip("no rejection far from its ratio in this case")


def test_shape_violation_is_rejected(case):
    inp, ref = case
    b = int(np.argmax(ref["n"] < inp.gamma))
    got = {k_: v.copy() for k_, v in ref.items()}
    got["tokens"][b, -1] = 0  # past the drawn token: must stay -1
    with pytest.raises(AssertionError):
        check_valid_draw(inp, got, ref, b)
