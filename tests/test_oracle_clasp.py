"""The CLaSp DP oracle against what fixes it independently (no GPU).

Pins:
  * consistency: the reported D(L, M) is the cosine between h_L and the state
    rebuilt by running the stack with the returned mask (no DP involved);
  * brute force on small stacks: no skip set of size M beats the DP's score
    (the review, "What would settle it": compare the DP's skip set with a
    brute-force search), and the DP's mask has exactly M skips;
  * a two-layer hand example worked out on paper;
  * M = 0 keeps every layer (score 1 on a full-model trajectory); M = L skips
    all (score cos(h_L, h_0)).
Planted mistakes (minimum instead of maximum, a backtracking step onto the
wrong layer) must fail a pin.
"""

import itertools

import numpy as np
import pytest

from oracle import clasp as K


def _stack(rng, L, d, scale=0.6):
    Ws = [K.bf16_round(rng.normal(0, scale / np.sqrt(d), (d, d))) for _ in range(L)]
    h = [rng.normal(0, 1, d)]
    for W in Ws:
        h.append(K.layer(W, h[-1]))
    return np.stack(h), Ws


def pin_consistency(fn, seeds=range(6)):
    for seed in seeds:
        rng = np.random.default_rng(seed)
        L, d, M = 7, 16, 3
        h, Ws = _stack(rng, L, d)
        mask, score, _ = fn(h, Ws, M)
        assert mask.sum() == M
        assert abs(score - K.cosine(h[L], K.apply_skips(h[0], Ws, mask))) < 1e-12


def pin_brute_force(fn, seeds=range(6)):
    for seed in seeds:
        rng = np.random.default_rng(100 + seed)
        L, d, M = 6, 12, 2
        h, Ws = _stack(rng, L, d, scale=1.2)
        _, score, _ = fn(h, Ws, M)
        best = max(K.cosine(h[L], K.apply_skips(h[0], Ws, np.isin(np.arange(L), S).astype(int)))
                   for S in itertools.combinations(range(L), M))
        assert score <= best + 1e-12


def pin_hand_example(fn):
    h0 = np.array([1.0, 0.0])
    W0 = np.array([[0.0, 0.0], [1.0, 0.0]])   # f0(x) = x + (0, x0)
    W1 = np.array([[0.0, -1.0], [0.0, 0.0]])  # f1(x) = x + (-x1, 0)
    h = np.stack([h0, K.layer(W0, h0), K.layer(W1, K.layer(W0, h0))])
    # h1 = (1, 1), h2 = (0, 1).  Skip one layer: skipping layer 0 gives
    # f1(h0) = (1, 0), cosine 0 with h2; skipping layer 1 gives f0(h0) =
    # (1, 1), cosine 1/sqrt(2): the DP skips layer 1
    mask, score, _ = fn(h, [W0, W1], 1)
    assert list(mask) == [0, 1]
    assert abs(score - 1 / np.sqrt(2)) < 1e-15


def pin_extremes(fn):
    rng = np.random.default_rng(7)
    h, Ws = _stack(rng, 5, 10)
    mask, score, _ = fn(h, Ws, 0)
    assert mask.sum() == 0 and abs(score - 1.0) < 1e-12
    mask, score, _ = fn(h, Ws, 5)
    assert mask.sum() == 5 and abs(score - K.cosine(h[5], h[0])) < 1e-12


PINS = [pin_consistency, pin_brute_force, pin_hand_example, pin_extremes]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(K.clasp_dp)


def _minimum(h, Ws, M):
    """Planted: the smaller cosine wins."""
    L = len(Ws)
    g = {(0, 0): h[0]}
    ch = {}
    for i in range(1, L + 1):
        for j in range(0, min(i, M) + 1):
            c = []
            if j <= i - 1:
                k = K.layer(Ws[i - 1], g[(i - 1, j)])
                c.append((K.cosine(h[i], k), 0, k))
            if j >= 1:
                c.append((K.cosine(h[i], g[(i - 1, j - 1)]), 1, g[(i - 1, j - 1)]))
            pick = min(c, key=lambda t: t[0])
            g[(i, j)], ch[(i, j)] = pick[2], pick[1]
    mask = np.zeros(L, np.int64)
    j = M
    for i in range(L, 0, -1):
        if ch[(i, j)]:
            mask[i - 1] = 1
            j -= 1
    return mask, K.cosine(h[L], g[(L, M)]), np.inf


def _shifted_mask(h, Ws, M):
    """Planted: backtracking marks layer i instead of i - 1."""
    mask, score, m = K.clasp_dp(h, Ws, M)
    return np.roll(mask, 1), score, m


@pytest.mark.parametrize("mutant", [_minimum, _shifted_mask], ids=lambda m: m.__name__)
def test_planted_mistake_is_caught(mutant):
    caught = False
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught = True
            break
    assert caught
