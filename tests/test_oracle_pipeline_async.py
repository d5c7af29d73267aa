"""The asynchronous PipeSpec snapshot oracle against what fixes it (no GPU).

Pins:
  * k = 2 with the window reaching the end of O_0 is one chain verification:
    accept length, emitted token and committed = the chain's rollback index
    + 1 (``oracle.verify.verify_chain``, pinned in tests/pins.py);
  * a token-level simulation of the buffers as lists (append the kept window
    tokens and the emitted token, cut every earlier buffer at each rejection,
    in any stage order) ends at the lengths the oracle reports, and every
    buffer stays consistent with the one below it on their overlap;
  * a hand example worked on paper;
  * a window that does not fit in the buffer below is malformed (ERR_WINDOW,
    nothing changes).
Planted mistakes (a rejection cutting only the buffer directly below, the
rejection position taken one past the rejected token, a bonus over an
unchecked draft token) must fail a pin.
"""

import numpy as np
import pytest

from oracle import pipeline_async as A
from oracle import verify as V

T = 1.0


def _layout(rng, k, windows, extra):
    """Buffer lengths l_0 .. l_{k-1} with l_{s-1} = l_s + w_s + extra_s, and
    the buffers' contents (each a prefix-consistent extension of the next)."""
    lengths = [0] * k
    lengths[k - 1] = int(rng.integers(0, 5))
    for s in range(k - 1, 0, -1):
        lengths[s - 1] = lengths[s] + windows[s - 1] + extra[s - 1]
    O0 = [int(x) for x in rng.integers(0, 7, lengths[0])]
    bufs = [O0[:l] for l in lengths]
    return lengths, bufs


def _stage_rows(rng, k, windows, V_, alpha=0.8):
    targets, drafts = [], []
    for s in range(1, k):
        q = rng.normal(0, 1.5, (windows[s - 1] + 1, V_))
        p = alpha * q + rng.normal(0, 0.6, q.shape)
        targets.append(p)
        drafts.append(q[:windows[s - 1]])
    return targets, drafts


def _run(fn, rng, k, windows, extra, greedy, final_bonus, V_=7):
    lengths, bufs = _layout(rng, k, windows, extra)
    targets, drafts = _stage_rows(rng, k, windows, V_)
    wins = [bufs[s - 1][lengths[s]:lengths[s] + windows[s - 1]] for s in range(1, k)]
    us = [rng.random(w) for w in windows]
    vs = [float(rng.random()) for _ in windows]
    return fn(targets, drafts, wins, us, vs, lengths, T, greedy, final_bonus), lengths, bufs, wins


def pin_two_models_is_the_chain(fn):
    rng = np.random.default_rng(1)
    for trial in range(60):
        g = int(rng.integers(1, 6))
        greedy = trial % 3 == 0
        l1 = int(rng.integers(0, 5))
        lengths = [l1 + g, l1]
        win = [int(x) for x in rng.integers(0, 7, g)]
        tgt = rng.normal(0, 1.5, (g + 1, 7)).astype(np.float32)
        drf = (0.8 * tgt[:g] + rng.normal(0, 0.6, (g, 7))).astype(np.float32)
        u = rng.random(g, dtype=np.float32)
        v = rng.random(1, dtype=np.float32)
        r = fn([tgt.astype(np.float64)], [drf.astype(np.float64)], [win], [u.astype(np.float64)], [float(v[0])],
               lengths, T, greedy, False)
        c = V.verify_chain(tgt[None], drf[None], np.array([win], np.int32), u[None], v, np.array([l1]), T, greedy,
                           "f32")
        assert r["a"][0] == c["accept_len"][0] and r["t"][0] == c["out_token"][0] and r["t_valid"][0] == 1
        assert r["committed"] == c["rollback_idx"][0] + 1


def _simulate(r, lengths, bufs, wins, k):
    """The buffers as token lists, the stages applied one after another."""
    O = [list(b) for b in bufs]
    for s in range(1, k):
        a = r["a"][s - 1]
        O[s] = O[s] + wins[s - 1][:a] + ([r["t"][s - 1]] if r["t_valid"][s - 1] else [])
    for s in range(1, k):
        if r["a"][s - 1] < len(wins[s - 1]):
            P = lengths[s] + r["a"][s - 1]
            for j in range(s):
                O[j] = O[j][:P]
    return O


def pin_list_simulation(fn):
    rng = np.random.default_rng(2)
    for trial in range(300):
        k = int(rng.integers(2, 6))
        windows = [int(rng.integers(1, 5)) for _ in range(k - 1)]
        extra = [int(rng.integers(0, 3)) * (trial % 2) for _ in range(k - 1)]
        r, lengths, bufs, wins = _run(fn, rng, k, windows, extra, trial % 4 == 0, trial % 3 == 0)
        assert r["error"] == 0
        O = _simulate(r, lengths, bufs, wins, k)
        assert [len(o) for o in O] == r["r"], (trial, [len(o) for o in O], r["r"])
        assert r["committed"] == len(O[k - 1])
        for j in range(1, k):
            n = min(len(O[j]), len(O[j - 1]))
            assert O[j][:n] == O[j - 1][:n], (trial, j)


def pin_hand_example(fn):
    # k = 3, greedy.  O_0 = [1, 2, 3, 4, 5], O_1 = [1, 2], O_2 = [] (l = 5, 2, 0).
    # stage 1 verifies O_0[2:5] = [3, 4, 5] (w = 3) and stage 2 verifies
    # O_1[0:2] = [1, 2] (w = 2).  Stage 1's argmaxes are 3, 4, 5, then 6:
    # all kept and the window ends O_0, so the bonus 6 is emitted: O_1 =
    # [1, 2, 3, 4, 5, 6].  Stage 2's argmaxes are 1, 0: token 2 is rejected
    # at position 1, the correction 0 is emitted (O_2 = [1, 0]), and both
    # earlier buffers are cut to length 1.
    def rows(best, n=7):
        x = np.zeros((len(best), n))
        for i, c in enumerate(best):
            x[i, c] = 1.0
        return x
    r = fn([rows([3, 4, 5, 6]), rows([1, 0, 2])], None, [[3, 4, 5], [1, 2]], None, None, [5, 2, 0], T, True,
           False)
    assert r["a"] == [3, 1] and r["t"] == [6, 0] and r["t_valid"] == [1, 1]
    assert r["r"] == [1, 1, 2] and r["committed"] == 2


def pin_malformed_window(fn):
    rng = np.random.default_rng(3)
    targets, drafts = _stage_rows(rng, 3, [3, 2], 7)
    for lengths in ([4, 2, 0], [5, 2, 1], [5, -1, 0]):
        r = fn(targets, drafts, [[0, 1, 2], [0, 1]], [rng.random(3), rng.random(2)], [0.5, 0.5], lengths, T,
               False, False)
        assert r["error"] == A.ERR_WINDOW and r["r"] == lengths and r["a"] == [0, 0] and r["t"] == [-1, -1]


PINS = [pin_two_models_is_the_chain, pin_list_simulation, pin_hand_example, pin_malformed_window]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(A.verify_pipeline_async_sequence)


def _cut_one_below(*args):
    r = A.verify_pipeline_async_sequence(*args)
    lengths, final_bonus = args[5], args[8]
    if r["error"]:
        return r
    k = len(lengths)
    new = [lengths[0]] + [lengths[s] + r["a"][s - 1] + r["t_valid"][s - 1] for s in range(1, k)]
    for s in range(1, k):
        if r["a"][s - 1] < len(args[2][s - 1]):
            new[s - 1] = min(new[s - 1], lengths[s] + r["a"][s - 1])
    r["r"], r["committed"] = new, new[k - 1]
    return r


def _cut_one_late(*args):
    r = A.verify_pipeline_async_sequence(*args)
    lengths = args[5]
    k = len(lengths)
    for s in range(1, k):
        if not r["error"] and r["a"][s - 1] < len(args[2][s - 1]):
            for j in range(s):
                r["r"][j] = max(r["r"][j], min(lengths[j], lengths[s] + r["a"][s - 1] + 1))
    return r


def _bonus_always(*args):
    targets, drafts, windows, us, vs, lengths, temperature, greedy, final_bonus = args
    r = A.verify_pipeline_async_sequence(*args)
    if r["error"] or r["a"][0] < len(windows[0]) or r["t_valid"][0]:
        return r
    # stage 1 emits its bonus even though O_0 holds an unchecked token there
    c = V.verify_chain_sequence(targets[0], None if greedy else drafts[0], windows[0],
                                None if greedy else us[0], None if greedy else vs[0], temperature, greedy)
    r["t"][0], r["t_valid"][0] = c["out_token"], 1
    r["r"][1] += 1
    if len(lengths) == 2:
        r["committed"] += 1
    return r


@pytest.mark.parametrize("mutant", [_cut_one_below, _cut_one_late, _bonus_always], ids=lambda m: m.__name__)
def test_planted_mistake_is_caught(mutant):
    caught = False
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught = True
            break
    assert caught
