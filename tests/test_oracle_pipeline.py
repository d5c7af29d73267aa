"""The k-model pipeline oracle against what fixes it independently (no GPU).

Pins:
  * k = 3 without the final bonus reproduces the three-model cascade oracle
    (itself pinned by losslessness and hand examples in tests/pins.py), for
    sampling and greedy, on seeded workloads;
  * k = 2 reproduces the chain oracle (accept length, token, rollback);
  * losslessness: with drafts drawn from M_0, the first token of the final
    buffer follows M_{k-1}'s distribution at position 0 (chi-square over many
    seeded trials), for k = 4 and 5, with and without the final bonus;
  * the final bonus: when the last stage keeps all w tokens, its bonus token
    follows M_{k-1}'s distribution at position w (chi-square);
  * rollback and length invariants on random snapshots.
Planted mistakes (a later stage testing against M_0 instead of the stage
below it, a rollback that ignores later rejections, a bonus drawn from the
wrong row) must each fail one pin.
"""

import numpy as np
import pytest
from scipy import stats as st

from oracle import pipeline as Pp
from oracle import verify as V
from workloads import synth


@pytest.mark.parametrize("greedy", [False, True])
@pytest.mark.parametrize("seed", [1, 2])
def test_k3_is_the_cascade(seed, greedy):
    spec = synth.with_sizes(synth.SPECS["cascade_b128_g8_g4_v128256_bf16"], B=12, V=700, greedy=greedy)
    w = synth.make(spec, seed=seed)
    o = V.verify_cascade(w["l0"], w["l1"], w["l2"], w["tokens"], w["u1"], w["v1"], w["u2"], w["v2"], w["base0"],
                         w["base1"], spec.temperature, greedy, spec.dtype, V=spec.V)
    p = Pp.verify_pipeline([w["l0"], w["l1"], w["l2"]], w["tokens"], [w["u1"], w["u2"]], [w["v1"], w["v2"]],
                           spec.temperature, greedy, False, spec.dtype, V=spec.V, base=[w["base0"], w["base1"]])
    for b in range(spec.B):
        assert p["error"][b] == o["error"][b]
        assert list(p["a"][b]) == [o["a1"][b], o["a2"][b]]
        assert p["w"][b][1] == o["w2"][b]
        assert p["t"][b][0] == o["t1"][b]
        assert (p["t"][b][1], p["t_valid"][b][1]) == (o["t2"][b], o["t2_valid"][b])
        assert list(p["r"][b]) == [o["r0"][b], o["r1"][b]]
        assert p["committed"][b] == o["committed"][b]


@pytest.mark.parametrize("greedy", [False, True])
def test_k2_is_the_chain(greedy):
    spec = synth.with_sizes(synth.SPECS["sampling_chain_b32_g8_v32000_bf16"], B=10, V=600, gamma=5, greedy=greedy)
    w = synth.make(spec, seed=4)
    o = V.verify_chain(w["target"], w["draft"], w["tokens"], w["u"], w["v"], w["prefix_len"], spec.temperature,
                       greedy, spec.dtype, V=spec.V)
    p = Pp.verify_pipeline([w["draft"], w["target"]], w["tokens"], [w["u"]], [w["v"]], spec.temperature, greedy,
                           False, spec.dtype, V=spec.V)
    assert np.array_equal(p["a"][:, 0], o["accept_len"])
    assert np.array_equal(p["t"][:, 0], o["out_token"])
    assert np.array_equal(p["r"][:, 0] + w["prefix_len"], o["rollback_idx"])
    assert np.array_equal(p["committed"], o["accept_len"] + 1)


def _softmax(x):
    e = np.exp(x - x.max())
    return e / e.sum()


def _models(rng, k, gs, final_bonus, Vv):
    """Logits per model and position; each model a perturbation of one base."""
    base = rng.normal(0, 1.0, (max(gs) + 2, Vv))
    models = [base[:gs[0]] + rng.normal(0, 0.8, (gs[0], Vv)),
              base[:gs[0] + 1] + rng.normal(0, 0.8, (gs[0] + 1, Vv))]
    for s in range(2, k):
        rows = gs[s - 1] + (1 if (final_bonus and s == k - 1) else 0)
        models.append(base[:rows] + rng.normal(0, 0.8, (rows, Vv)))
    return models


def _trial(rng, models, gs, k):
    q0 = [_softmax(models[0][j]) for j in range(gs[0])]
    tokens = [int(rng.choice(len(q0[0]), p=q0[j])) for j in range(gs[0])]
    us = [rng.random(gs[0])] + [rng.random(gs[s - 1]) for s in range(2, k)]
    vs = [rng.random() for _ in range(k - 1)]
    return tokens, us, vs


def pin_lossless(fn, k, final_bonus, trials=5000, seed=0):
    """First token of the final buffer ~ softmax(M_{k-1}[0])."""
    rng = np.random.default_rng(seed)
    Vv, gs = 5, [3] * (k - 1)
    models = _models(rng, k, gs, final_bonus, Vv)
    counts = np.zeros(Vv)
    for _ in range(trials):
        tokens, us, vs = _trial(rng, models, gs, k)
        r = fn(models, tokens, us, vs, 1.0, False, final_bonus)
        first = tokens[0] if r["a"][0] > 0 else r["t"][0]
        for s in range(2, k):
            if r["a"][s - 1] == 0:  # rejected at position 0 (w >= 1 always)
                first = r["t"][s - 1]
        counts[first] += 1
    want = _softmax(models[k - 1][0]) * trials
    assert st.chisquare(counts, want).pvalue > 1e-4, (counts, want)


def pin_bonus_law(fn, k, trials=6000, seed=0):
    """With the final bonus: when the last stage keeps all w tokens, the bonus
    follows softmax(M_{k-1}[w])."""
    rng = np.random.default_rng(seed)
    Vv, gs = 4, [2] * (k - 1)
    models = _models(rng, k, gs, True, Vv)
    seen = {}
    for _ in range(trials):
        tokens, us, vs = _trial(rng, models, gs, k)
        r = fn(models, tokens, us, vs, 1.0, False, True)
        a, w = r["a"][-1], r["w"][-1]
        if a == w:
            seen.setdefault(w, np.zeros(Vv))[r["t"][-1]] += 1
    tested = 0
    for w, counts in seen.items():
        if counts.sum() >= 400:
            want = _softmax(models[k - 1][w]) * counts.sum()
            assert st.chisquare(counts, want).pvalue > 1e-4, (w, counts, want)
            tested += 1
    assert tested >= 1


@pytest.mark.parametrize("k,final_bonus", [(4, False), (4, True), (5, False)])
def test_lossless(k, final_bonus):
    pin_lossless(Pp.verify_pipeline_sequence, k, final_bonus, seed=k + int(final_bonus))


@pytest.mark.parametrize("k", [3, 4])
def test_bonus_law(k):
    pin_bonus_law(Pp.verify_pipeline_sequence, k, seed=30 + k)


def pin_invariants(fn, k=5, n=300, seed=3):
    rng = np.random.default_rng(seed)
    Vv = 7
    for _ in range(n):
        g1 = int(rng.integers(1, 6))
        gs = [g1] + [int(rng.integers(1, 6)) for _ in range(2, k)]
        fb = bool(rng.integers(0, 2))
        models = [rng.normal(0, 1, (g1, Vv)), rng.normal(0, 1, (g1 + 1, Vv))]
        for s in range(2, k):
            models.append(rng.normal(0, 1, (gs[s - 1] + (1 if (fb and s == k - 1) else 0), Vv)))
        tokens = [int(x) for x in rng.integers(0, Vv, g1)]
        us = [rng.random(g1)] + [rng.random(gs[s - 1]) for s in range(2, k)]
        vs = list(rng.random(k - 1))
        r = fn(models, tokens, us, vs, 1.0, False, fb)
        assert r["t_valid"][0] == 1 and r["w"][0] == g1
        L = r["a"][0] + 1
        for s in range(2, k):
            assert r["w"][s - 1] == min(gs[s - 1], L)
            assert r["a"][s - 1] <= r["w"][s - 1]
            if r["a"][s - 1] < r["w"][s - 1]:
                assert r["t_valid"][s - 1] == 1
            L = r["a"][s - 1] + r["t_valid"][s - 1]
        assert r["committed"] == L
        assert r["r"][0] <= r["a"][0]
        for j in range(1, k - 1):
            assert r["r"][j] <= r["w"][j]
        for s in range(1, k):  # a rejection at stage s bounds every earlier buffer
            if r["a"][s - 1] < r["w"][s - 1]:
                assert all(r["r"][j] <= r["a"][s - 1] for j in range(0, s))


def test_invariants():
    pin_invariants(Pp.verify_pipeline_sequence)


# planted mistakes ---------------------------------------------------------

def _q_is_m0(models, tokens, us, vs, temperature, greedy, final_bonus):
    """Every stage s >= 2 tests against M_0's rows instead of M_{s-1}'s."""
    k = len(models)
    fake = list(models)
    for s in range(1, k - 1):
        rows = models[s].shape[0]
        fake[s] = np.vstack([models[0]] * (rows // models[0].shape[0] + 2))[:rows]
    r = Pp.verify_pipeline_sequence([models[0], models[1]] + fake[2:], tokens, us, vs, temperature, greedy,
                                    final_bonus) if k == 2 else None
    if r is not None:
        return r
    # stage 1 must still use M_1 as its p: run stage by stage
    out = Pp.verify_pipeline_sequence(models[:2], tokens, us[:1], vs[:1], temperature, greedy, False)
    buf = list(tokens[:out["a"][0]]) + [out["t"][0]]
    res = dict(a=[out["a"][0]], w=[out["w"][0]], t=[out["t"][0]], t_valid=[1])
    for s in range(2, k):
        rows = models[s].shape[0] - (1 if (final_bonus and s == k - 1) else 0)
        w = min(rows, len(buf))
        q = np.vstack([models[0]] * (w // models[0].shape[0] + 2))[:w]
        p = np.vstack([models[s][:w], models[s][-1:]])
        sub = Pp.verify_pipeline_sequence([q, p], buf[:w], [us[s - 1][:w]], [vs[s - 1]], temperature, greedy, False)
        a = sub["a"][0]
        if a < w:
            buf = buf[:a] + [sub["t"][0]]
            res["t"].append(sub["t"][0])
            res["t_valid"].append(1)
        else:
            buf = buf[:w]
            res["t"].append(-1)
            res["t_valid"].append(0)
        res["a"].append(a)
        res["w"].append(w)
    res["r"] = [0] * (k - 1)
    res["committed"] = len(buf)
    return res


def _rollback_own_stage_only(models, tokens, us, vs, temperature, greedy, final_bonus):
    r = Pp.verify_pipeline_sequence(models, tokens, us, vs, temperature, greedy, final_bonus)
    r["r"] = [r["a"][0]] + [r["w"][j] for j in range(1, len(r["r"]))]
    return r


def _wrong_bonus_row(models, tokens, us, vs, temperature, greedy, final_bonus):
    if final_bonus:
        last = models[-1]
        models = models[:-1] + [np.vstack([last[:-1], last[:1]])]  # the bonus row replaced by row 0
    return Pp.verify_pipeline_sequence(models, tokens, us, vs, temperature, greedy, final_bonus)


def test_planted_q_is_m0_is_caught():
    with pytest.raises(AssertionError):
        pin_lossless(_q_is_m0, 4, False, trials=5000, seed=11)


def test_planted_rollback_is_caught():
    with pytest.raises(AssertionError):
        pin_invariants(_rollback_own_stage_only)


def test_planted_bonus_row_is_caught():
    with pytest.raises(AssertionError):
        pin_bonus_law(_wrong_bonus_row, 3, seed=33)
