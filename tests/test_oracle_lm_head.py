"""The LM-head chain oracle against what fixes it (no GPU).

Pins:
  * identity and permutation heads (exact in bfloat16; d = V): the target
    head the identity and the draft head a permutation matrix give the chain
    oracle's results on the hidden states as stored logits, the draft's
    columns permuted (tests/pins.py pins that oracle);
  * relabelling the vocabulary (both heads' rows and the tokens permuted)
    leaves every accept length unchanged, and moves the greedy token with it;
  * scaling both heads by 2 and the temperature by 2 changes nothing (every
    quotient logit / T is the same double).
Planted mistakes (a head applied transposed, the target head used for the
draft, the temperature dropped) must fail a pin.
"""

import numpy as np
import pytest

from oracle import lm_head as H
from oracle import verify as V
from workloads import synth

T = 0.8


def _bf16(x):
    return H.bf16_values(synth.bf16_from_float32(np.asarray(x, np.float32)))


def _case(seed, B=6, gamma=4, d=24, Vv=24, greedy=False):
    rng = np.random.default_rng(seed)
    w_d = _bf16(rng.normal(0, 1 / np.sqrt(d), (Vv, d)) * 4)
    w_t = _bf16(w_d + rng.normal(0, 0.3 / np.sqrt(d), (Vv, d)) * 4)
    h_d = _bf16(rng.normal(0, 1, (B, gamma, d)))
    h_t = np.concatenate([_bf16(0.9 * h_d + rng.normal(0, 0.3, h_d.shape)), _bf16(rng.normal(0, 1, (B, 1, d)))], 1)
    tokens = np.empty((B, gamma), np.int64)
    for b in range(B):
        logits = h_d[b] @ w_d.T / T
        g = logits + (0 if greedy else rng.gumbel(size=logits.shape))
        tokens[b] = np.argmax(g, axis=-1)
    u = rng.random((B, gamma))
    v = rng.random(B)
    prefix = rng.integers(0, 50, B)
    return h_t, h_d, w_t, w_d, tokens, u, v, prefix


def pin_identity_and_permutation_heads(fn):
    for greedy in (False, True):
        for seed in range(4):
            h_t, h_d, _, _, tokens, u, v, prefix = _case(seed, greedy=greedy)
            d = h_t.shape[2]
            perm = np.random.default_rng(100 + seed).permutation(d)
            eye = np.eye(d)
            P = eye[perm]                      # (P x)[i] = x[perm[i]]: draft logit i = h[perm[i]]
            r = fn(h_t, h_d, eye, P, tokens, u, v, prefix, T, greedy)
            tgt_bits = synth.bf16_from_float32(h_t.astype(np.float32))
            drf_bits = synth.bf16_from_float32(h_d[:, :, perm].astype(np.float32))
            o = V.verify_chain(tgt_bits, drf_bits, tokens.astype(np.int32), u.astype(np.float32),
                               v.astype(np.float32), prefix, T, greedy, "bf16")
            for k in ("accept_len", "out_token", "rollback_idx", "error"):
                assert np.array_equal(r[k], o[k]), (k, greedy, seed)


def pin_relabelled_vocabulary(fn):
    for greedy in (False, True):
        for seed in range(4):
            h_t, h_d, w_t, w_d, tokens, u, v, prefix = _case(10 + seed, greedy=greedy)
            Vv = w_t.shape[0]
            pi = np.random.default_rng(200 + seed).permutation(Vv)   # token x becomes pi[x]
            inv = np.argsort(pi)
            a = fn(h_t, h_d, w_t, w_d, tokens, u, v, prefix, T, greedy)
            b = fn(h_t, h_d, w_t[inv], w_d[inv], pi[tokens], u, v, prefix, T, greedy)
            assert np.array_equal(a["accept_len"], b["accept_len"]), (greedy, seed)
            if greedy:
                assert np.array_equal(pi[a["out_token"]], b["out_token"]), seed


def pin_scale_invariance(fn):
    for greedy in (False, True):
        h_t, h_d, w_t, w_d, tokens, u, v, prefix = _case(30, greedy=greedy)
        a = fn(h_t, h_d, w_t, w_d, tokens, u, v, prefix, T, greedy)
        b = fn(h_t, h_d, 2 * w_t, 2 * w_d, tokens, u, v, prefix, 2 * T, greedy)
        for k in a:
            assert np.array_equal(a[k], b[k]), (k, greedy)


PINS = [pin_identity_and_permutation_heads, pin_relabelled_vocabulary, pin_scale_invariance]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(H.verify_chain_from_hidden)


def _transposed(h_t, h_d, w_t, w_d, *rest):
    return H.verify_chain_from_hidden(h_t, h_d, w_t.T, w_d.T, *rest)


def _target_head_for_draft(h_t, h_d, w_t, w_d, *rest):
    return H.verify_chain_from_hidden(h_t, h_d, w_t, w_t, *rest)


def _no_temperature(h_t, h_d, w_t, w_d, tokens, u, v, prefix, temperature, greedy):
    return H.verify_chain_from_hidden(h_t, h_d, w_t, w_d, tokens, u, v, prefix, 1.0, greedy)


@pytest.mark.parametrize("mutant", [_transposed, _target_head_for_draft, _no_temperature],
                         ids=lambda m: m.__name__)
def test_planted_mistake_is_caught(mutant):
    caught = False
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught = True
            break
    assert caught
