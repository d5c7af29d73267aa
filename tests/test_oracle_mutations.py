"""Planted mistakes in the CPU oracle must be caught by some pin.

Each case swaps one oracle function for a plausibly wrong version (a dropped
term, a flipped comparison, a transposed operand) on the CPU only, runs the
pins that should notice, and asserts that at least one fails.  This is what
shows that the pins in tests/pins.py constrain the oracle rather than echo it.
"""

import math

import numpy as np
import pytest

from oracle import verify as V

from . import pins


def _caught(checks):
    for check in checks:
        try:
            check()
        except Exception:  # a failed assertion, or the mutant crashing
            return True
    return False


MUTANTS = {
    # residual computed the wrong way round (transposed operands)
    "residual_q_minus_p": ("residual", lambda p, q: np.maximum(q - p, 0.0),
                           [lambda: pins.pin_hand_examples(V), lambda: pins.pin_chain_grid_law(V)]),
    # non-strict accept test
    "accept_le": ("keeps", lambda u, r: u <= min(1.0, r),
                  [lambda: pins.pin_hand_examples(V)]),
    # ratio inverted
    "ratio_q_over_p": ("accept_ratio", lambda p, q: (q / p) if p > 0 else math.inf,
                       [lambda: pins.pin_acceptance_probability(V, n=6000)]),
    # temperature multiplies instead of dividing
    "temperature_times": ("temperature_softmax",
                          lambda l, T: (lambda z: np.exp(z - z.max()) / np.exp(z - z.max()).sum())(l * T),
                          [lambda: pins.pin_log_partition(V), lambda: pins.pin_acceptance_probability(V, n=6000)]),
    # searchsorted-left instead of right (>= instead of >)
    "invcdf_left": ("inverse_cdf",
                    lambda w, v: (lambda c: (int(np.flatnonzero(c >= v * c[-1])[0]), float(c[-1]), 0.0))(np.cumsum(w)),
                    [lambda: pins.pin_inverse_cdf(V)]),
    # greedy ties go to the highest index
    "argmax_last": ("first_argmax", lambda l: int(np.flatnonzero(l == np.max(l))[-1]),
                    [lambda: pins.pin_greedy_argmax(V), lambda: pins.pin_hand_examples(V)]),
    # the tree keeps testing siblings against the unchanged p
    "tree_no_residual_update": ("residual", lambda p, q: p.copy(),
                                [lambda: pins.pin_hand_examples(V), lambda: pins.pin_tree_lossless(V, n=4000)]),
    # reading R3's fallback loses its error bit (the draw still comes from p)
    "zero_mass_bit_dropped": ("ERR_ZERO_MASS", 0, [lambda: pins.pin_hand_examples(V)]),
    # +inf logits silently accepted
    "inf_not_flagged": ("row_is_nonfinite", lambda l: bool(np.isnan(l).any()),
                        [lambda: pins.pin_nonfinite_rows(V)]),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, bad, checks = MUTANTS[name]
    # the pins pass on the real oracle ...
    assert not _caught(checks[:1]), f"pin fails on the unmodified oracle ({name})"
    # ... and at least one fails once the mistake is planted
    monkeypatch.setattr(V, attr, bad)
    assert _caught(checks), f"planted mistake {name} was not caught"
