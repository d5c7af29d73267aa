"""PipeSpec analytical model, restated in float64 (test infrastructure only).

Source: Pith review of "PipeSpec: Breaking Stage Dependencies in Hierarchical
LLM Decoding" (arXiv 2505.01572), sections "What carries the argument" and
"Core claim" (Eq. (1), Eq. (4) and Theorem 1), and the "Assumptions" list,
which attributes the per-round expected-token formula to Leviathan et al.

Pins: these functions are checked against Monte-Carlo runs of the oracle's
verification rule (tests/test_oracle_pins.py), not against re-typed copies
of themselves.
"""

from __future__ import annotations


def expected_tokens_per_round(alpha: float, gamma: int) -> float:
    """Expected tokens one verification round emits under i.i.d. acceptance.

    A round that tests gamma drafted tokens, each accepted independently with
    probability alpha, stops at the first rejection and always emits one
    extra token (the correction or the bonus).  The count is a truncated
    geometric series: 1 + alpha + ... + alpha**gamma.  The PipeSpec review
    quotes its closed form (1 - alpha**(gamma+1)) / (1 - alpha) ("Assumptions",
    Eq. (1)).  At alpha == 1 the series is gamma + 1.
    """
    if not 0.0 <= alpha <= 1.0:
        raise ValueError("alpha must lie in [0, 1]")
    if gamma < 0:
        raise ValueError("gamma must be >= 0")
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def accept_length_pmf(alpha: float, gamma: int) -> list[float]:
    """Law of the accepted-prefix length a in {0..gamma} under i.i.d. acceptance.

    P(a = k) = alpha**k (1 - alpha) for k < gamma and alpha**gamma for
    k == gamma: the first rejection happens at position k, or never.
    """
    pmf = [alpha ** k * (1.0 - alpha) for k in range(gamma)]
    pmf.append(alpha ** gamma)
    return pmf


def rho_step(rho_prev: float, alpha: float, gamma: int) -> float:
    """One step of the PipeSpec verification-probability recurrence.

    rho(t_j) = rho(t_{j-1}) * alpha**(gamma+1) + (1 - rho(t_{j-1})) * alpha
    ("What carries the argument").  Read as a two-state chain: from the
    verifying state the stage stays there when a full window of gamma+1
    tokens is accepted; from the other state it enters when one token is.
    """
    return rho_prev * alpha ** (gamma + 1) + (1.0 - rho_prev) * alpha


def rho_steady(alpha: float, gamma: int) -> float:
    """Steady state of the recurrence: alpha / (1 - alpha**(gamma+1) + alpha).

    "What carries the argument" and "Core claim" give this limit.
    """
    return alpha / (1.0 - alpha ** (gamma + 1) + alpha)


def pipespec_expected_tokens(alpha: float, gamma: int) -> float:
    """E[N] of Theorem 1 / Eq. (4): (1 - rho) * 1 + rho * E[tokens per round]."""
    rho = rho_steady(alpha, gamma)
    return (1.0 - rho) * 1.0 + rho * expected_tokens_per_round(alpha, gamma)
