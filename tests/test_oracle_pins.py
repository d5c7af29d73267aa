"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""

import pytest

from oracle import verify as V

from . import pins


def test_hand_examples():
    pins.pin_hand_examples(V)


def test_inverse_cdf_is_searchsorted_right():
    pins.pin_inverse_cdf(V)


def test_greedy_is_first_argmax():
    pins.pin_greedy_argmax(V)


def test_log_partition_matches_logsumexp():
    pins.pin_log_partition(V)


def test_onehot_equal_distributions_keep_every_draft():
    pins.pin_onehot_accepts_all(V)


def test_data_errors():
    pins.pin_nonfinite_rows(V)


def test_acceptance_probability_closed_form():
    pins.pin_acceptance_probability(V)


@pytest.mark.parametrize("alpha", [0.05, 0.3, 0.6, 0.9])
@pytest.mark.parametrize("gamma", [1, 4, 5, 8])
def test_accept_length_law(alpha, gamma):
    pins.pin_accept_length_law(V, alpha, gamma, n=1500, seed=int(alpha * 100) + gamma)


@pytest.mark.parametrize("alpha,gamma", [(0.6, 4), (0.3, 2), (0.9, 8)])
def test_pipespec_rho_recurrence(alpha, gamma):
    pins.pin_rho_recurrence(V, alpha, gamma, steps=12000, seed=gamma)


def test_gamma_zero_and_theorem1():
    pins.pin_gamma_zero(V)


def test_chain_grid_law_exact():
    pins.pin_chain_grid_law(V)


def test_chain_lossless():
    pins.pin_chain_lossless(V)


def test_tree_lossless():
    pins.pin_tree_lossless(V)


def test_tree_exact_law():
    pins.pin_tree_exact_law(V)


def test_cascade_lossless():
    pins.pin_cascade_lossless(V)


def test_cascade_invariants():
    pins.pin_cascade_invariants(V)


def test_tree_chain_shaped_equals_chain():
    pins.pin_tree_chain_shaped(V)


# --------------------------------------------------------------------------
# the statistical pins at full power: the trial counts the contract names
# (1e5 for the accept-length law and the acceptance probability, 2e5 for the
# losslessness tests, 1e6 steps for the PipeSpec recurrence).  Several
# minutes in all, so they run only when asked for: pytest -m slow
# --------------------------------------------------------------------------

@pytest.mark.slow
@pytest.mark.parametrize("alpha", [0.05, 0.3, 0.6, 0.9])
@pytest.mark.parametrize("gamma", [1, 4, 5, 8])
def test_accept_length_law_full(alpha, gamma):
    pins.pin_accept_length_law(V, alpha, gamma, n=100_000, seed=1000 + int(alpha * 100) + gamma)


@pytest.mark.slow
def test_acceptance_probability_full():
    pins.pin_acceptance_probability(V, seed=11, n=100_000)


@pytest.mark.slow
@pytest.mark.parametrize("alpha,gamma", [(0.6, 4), (0.3, 2), (0.9, 8)])
def test_pipespec_rho_recurrence_full(alpha, gamma):
    pins.pin_rho_recurrence(V, alpha, gamma, steps=1_000_000, seed=100 + gamma)


@pytest.mark.slow
def test_chain_lossless_full():
    pins.pin_chain_lossless(V, seed=21, n=200_000)


@pytest.mark.slow
def test_tree_lossless_full():
    pins.pin_tree_lossless(V, seed=22, n=200_000)


@pytest.mark.slow
def test_cascade_lossless_full():
    pins.pin_cascade_lossless(V, seed=24, n=200_000)
