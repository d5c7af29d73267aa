"""Checks that tie the CPU oracle to what the pages and the mathematics fix.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
something outside itself: hand-worked examples (tests/golden/hand_examples.json),
closed forms from the PipeSpec review, exact probability laws derived here
from the accept / residual rule, textbook routines (searchsorted, argmax,
logsumexp) and statistical laws.  They take the oracle module as an argument
so that tests/test_oracle_mutations.py can plant a mistake in the oracle and
check that some pin catches it.
"""

from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
from scipy import special, stats

from oracle import closed_forms as cf

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------
# helpers (test-side arithmetic, independent of the oracle's code)
# --------------------------------------------------------------------------

def _arr(rows):
    return np.array([[-math.inf if x == "-inf" else float(x) for x in r] for r in rows])


def softmax(l, T=1.0):
    z = np.asarray(l, float) / T
    e = np.exp(z - z.max())
    return e / e.sum()


def logits_of(p):
    """Logits whose temperature-1 softmax is p (zeros become -inf)."""
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, float))


def chi2_pvalue(counts, probs):
    """Pearson chi-squared p-value with bins of expected count < 5 merged."""
    counts = np.asarray(counts, float)
    n = counts.sum()
    exp = np.asarray(probs, float) * n
    order = np.argsort(exp)
    c_m, e_m = [], []
    acc_c = acc_e = 0.0
    for i in order:
        acc_c += counts[i]
        acc_e += exp[i]
        if acc_e >= 5.0:
            c_m.append(acc_c)
            e_m.append(acc_e)
            acc_c = acc_e = 0.0
    if acc_e > 0:
        if e_m:
            c_m[-1] += acc_c
            e_m[-1] += acc_e
        else:
            c_m.append(acc_c)
            e_m.append(acc_e)
    if len(c_m) < 2:
        return 1.0
    return float(stats.chisquare(c_m, e_m).pvalue)


# --------------------------------------------------------------------------
# hand-worked examples
# --------------------------------------------------------------------------

def pin_hand_examples(V):
    with open(os.path.join(GOLDEN, "hand_examples.json")) as fh:
        ex = json.load(fh)
    for e in ex["chain"]:
        r = V.verify_chain_sequence(_arr(e["target"]), _arr(e["draft"]),
                                    e["tokens"], e["u"], e["v"], 1.0, e["greedy"])
        for k, want in e["expect"].items():
            got = r[k]
            ok = abs(got - want) < 1e-12 if isinstance(want, float) else got == want
            assert ok, f"hand example {e['name']}: {k} = {got}, expected {want}"
    for e in ex["tree"]:
        r = V.verify_tree_sequence(e["parent"], e["tokens"], _arr(e["target"]),
                                   _arr(e["draft"]), e["u"], e["v"], 1.0,
                                   e["greedy"], e["max_depth"])
        assert list(r["path"]) == e["expect"]["path"], f"hand example {e['name']}: path {r['path']}"
        assert r["out_token"] == e["expect"]["out_token"], \
            f"hand example {e['name']}: token {r['out_token']}"
        if "error" in e["expect"]:
            assert r["error"] == e["expect"]["error"], f"hand example {e['name']}: error {r['error']}"
    for e in ex["cascade"]:
        r = V.verify_cascade_sequence(_arr(e["l0"]), _arr(e["l1"]), _arr(e["l2"]),
                                      e["tokens"], e["u1"], e["v1"], e["u2"],
                                      e["v2"], 1.0, e["greedy"])
        for k, want in e["expect"].items():
            assert r[k] == want, f"hand example {e['name']}: {k} = {r[k]}, expected {want}"


# --------------------------------------------------------------------------
# textbook special cases
# --------------------------------------------------------------------------

def pin_inverse_cdf(V, seed=0):
    """inverse_cdf == searchsorted(cumsum(w), v*Z, 'right'), incl. exact
    boundaries and zero weights."""
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(300):
        n = int(rng.integers(1, 40))
        w = rng.random(n)
        w[rng.random(n) < 0.3] = 0.0
        if w.sum() == 0:
            w[0] = 1.0
        cases.append((w, float(rng.random())))
    # exact boundaries: v * Z equals a running sum
    w = np.array([1.0, 1.0, 1.0, 1.0])
    cases += [(w, 0.25), (w, 0.5), (w, 0.75), (w, 0.0)]
    cases += [(np.array([0.0, 2.0, 0.0, 2.0]), 0.5), (np.array([0.0, 0.5, 0.5]), 0.0)]
    for w, v in cases:
        y, Z, _ = V.inverse_cdf(w, v)
        c = np.cumsum(w)
        want = int(np.searchsorted(c, v * c[-1], side="right"))
        assert y == want, f"inverse_cdf({w}, {v}) = {y}, searchsorted gives {want}"
        assert w[y] > 0


def pin_greedy_argmax(V, seed=0):
    rng = np.random.default_rng(seed)
    for _ in range(300):
        n = int(rng.integers(1, 30))
        l = rng.integers(-3, 4, n).astype(float)  # many ties
        assert V.first_argmax(l) == int(np.argmax(l))


def pin_log_partition(V, seed=0):
    rng = np.random.default_rng(seed)
    for T in (0.3, 0.7, 1.0, 2.5):
        for _ in range(20):
            l = rng.normal(0, 3, int(rng.integers(1, 2000)))
            got = V.log_partition(l, T)
            want = float(special.logsumexp(l / T))
            assert abs(got - want) <= 1e-12 * max(1.0, abs(want)), (T, got, want)
            p = V.temperature_softmax(l, T)
            assert np.allclose(np.log(p), l / T - want, atol=1e-10)


def pin_onehot_accepts_all(V):
    """Sampling with p == q one-hot keeps every draft (r = 1)."""
    Vv, g = 7, 5
    rows = np.full((g + 1, Vv), -math.inf)
    toks = [3, 1, 4, 1, 5]
    for i, t in enumerate(toks):
        rows[i, t] = 0.0
    rows[g, 2] = 0.0
    r = V.verify_chain_sequence(rows, rows[:g].copy(), toks, [0.999] * g, 0.5, 0.9, False)
    assert r["accept_len"] == g and r["out_token"] == 2 and r["error"] == 0


def pin_nonfinite_rows(V):
    base = np.zeros((2, 4))
    for bad in (math.nan, math.inf):
        t = base.copy()
        t[1, 2] = bad
        r = V.verify_chain_sequence(t, base[:1], [0], [0.5], 0.5, 1.0, False)
        assert r["error"] & V.ERR_NONFINITE and r["accept_len"] == 0 and r["out_token"] == -1
    t = base.copy()
    t[0, :] = -math.inf
    r = V.verify_chain_sequence(t, base[:1], [0], [0.5], 0.5, 1.0, True)
    assert r["error"] & V.ERR_NONFINITE
    t = base.copy()
    t[0, 1] = -math.inf  # a masked entry is allowed
    r = V.verify_chain_sequence(t, base[:1], [0], [0.5], 0.5, 1.0, False)
    assert r["error"] == 0
    r = V.verify_chain_sequence(base, base[:1], [4], [0.5], 0.5, 1.0, False)
    assert r["error"] & V.ERR_TOKEN and r["out_token"] == -1


# --------------------------------------------------------------------------
# closed forms and statistical laws
# --------------------------------------------------------------------------

def pin_acceptance_probability(V, seed=0, n=20000, T=0.8):
    """P(keep) = sum_x q(x) min(1, p(x)/q(x)) = sum_x min(p(x), q(x))."""
    rng = np.random.default_rng(seed)
    Vv = 10
    P = rng.normal(0, 1.5, (2, Vv))
    Q = rng.normal(0, 1.5, (1, Vv))
    p, q = softmax(P[0], T), softmax(Q[0], T)
    alpha = float(np.minimum(p, q).sum())
    kept = 0
    for _ in range(n):
        d = int(rng.choice(Vv, p=q))
        r = V.verify_chain_sequence(P, Q, [d], [rng.random()], rng.random(), T, False)
        kept += r["accept_len"]
    se = math.sqrt(alpha * (1 - alpha) / n)
    assert abs(kept / n - alpha) < 4 * se, (kept / n, alpha)


def _alpha_rows(alpha, Vv=8):
    """p, q over Vv tokens with sum min(p, q) == alpha exactly."""
    c = np.zeros(Vv)
    c[2:] = np.arange(1, Vv - 1, dtype=float)
    c /= c.sum()
    p = alpha * c
    q = alpha * c
    p[0] += 1 - alpha
    q[1] += 1 - alpha
    return p, q


def pin_accept_length_law(V, alpha, gamma, n=3000, seed=0):
    """E[a + 1] = (1 - alpha^(gamma+1)) / (1 - alpha) and the law of a."""
    rng = np.random.default_rng(seed)
    p, q = _alpha_rows(alpha)
    P = np.tile(logits_of(p), (gamma + 1, 1))
    Q = np.tile(logits_of(q), (gamma, 1))
    counts = np.zeros(gamma + 1)
    for _ in range(n):
        d = rng.choice(len(q), size=gamma, p=q)
        r = V.verify_chain_sequence(P, Q, [int(x) for x in d], rng.random(gamma),
                                    rng.random(), 1.0, False)
        counts[r["accept_len"]] += 1
    pmf = np.array(cf.accept_length_pmf(alpha, gamma))
    ks = np.arange(gamma + 1) + 1.0
    mean, var = float((pmf * ks).sum()), float((pmf * ks ** 2).sum() - (pmf * ks).sum() ** 2)
    emp = float((counts * ks).sum() / n)
    assert abs(mean - cf.expected_tokens_per_round(alpha, gamma)) < 1e-12
    assert abs(emp - mean) < 4 * math.sqrt(var / n) + 1e-12, (alpha, gamma, emp, mean)
    assert chi2_pvalue(counts, pmf) > 1e-3, (alpha, gamma, counts, pmf)


def pin_rho_recurrence(V, alpha, gamma, steps=20000, seed=0):
    """Occupancy of the PipeSpec two-state chain driven by oracle outcomes
    converges to rho = alpha / (1 - alpha^(gamma+1) + alpha)."""
    rng = np.random.default_rng(seed)
    p, q = _alpha_rows(alpha)
    lp, lq = logits_of(p), logits_of(q)
    win = gamma + 1
    P_win, Q_win = np.tile(lp, (win + 1, 1)), np.tile(lq, (win, 1))
    P_one, Q_one = np.tile(lp, (2, 1)), np.tile(lq, (1, 1))
    state, occ = 0, 0
    for _ in range(steps):
        if state:
            d = rng.choice(len(q), size=win, p=q)
            r = V.verify_chain_sequence(P_win, Q_win, [int(x) for x in d],
                                        rng.random(win), rng.random(), 1.0, False)
            state = int(r["accept_len"] == win)
        else:
            d = int(rng.choice(len(q), p=q))
            r = V.verify_chain_sequence(P_one, Q_one, [d], [rng.random()],
                                        rng.random(), 1.0, False)
            state = int(r["accept_len"] == 1)
        occ += state
    rho = cf.rho_steady(alpha, gamma)
    lam = alpha ** win - alpha  # second eigenvalue of the two-state chain
    se = math.sqrt(rho * (1 - rho) / steps * (1 + lam) / (1 - lam))
    assert abs(occ / steps - rho) < 4 * se, (occ / steps, rho)
    # the recurrence iterated numerically reaches the same fixed point
    x = 0.0
    for _ in range(10000):
        x = cf.rho_step(x, alpha, gamma)
    assert abs(x - rho) < 1e-12


def pin_chain_grid_law(V, Vv=4, n=100, seed=3, T=1.0):
    """gamma = 1: the oracle's decisions over a midpoint grid of (u, v) match
    the exact law of the rule for every draft token, and the first emitted
    token is distributed as p_0 (lossless).

    Exact law for draft d at position 0 (r = p0(d)/q0(d)):
      keep with probability min(1, r), then the bonus y ~ p_1;
      reject with probability 1 - min(1, r), then y ~ max(0, p0 - q0) / Z.
    """
    rng = np.random.default_rng(seed)
    P = rng.normal(0, 1.2, (2, Vv))
    Q = rng.normal(0, 1.2, (1, Vv))
    p0, p1, q0 = softmax(P[0], T), softmax(P[1], T), softmax(Q[0], T)
    grid = (np.arange(n) + 0.5) / n
    first = np.zeros(Vv)
    tol = 1.0 / (2 * n) + 1.0 / n + 1e-12
    for d in range(Vv):
        freq = np.zeros((2, Vv))
        for u in grid:
            for v in grid:
                r = V.verify_chain_sequence(P, Q, [d], [u], v, T, False)
                freq[r["accept_len"], r["out_token"]] += 1
        freq /= n * n
        keep = min(1.0, p0[d] / q0[d])
        res = np.maximum(p0 - q0, 0.0)
        exact = np.vstack([(1 - keep) * res / res.sum(), keep * p1])
        assert np.abs(freq - exact).max() < tol, (d, freq, exact)
        first += q0[d] * np.where(np.arange(Vv) == d, freq[1].sum(), 0.0) + q0[d] * freq[0]
    assert np.abs(first - p0).max() < tol, (first, p0)


def pin_chain_lossless(V, seed=1, n=20000, Vv=16, gamma=3, T=0.9):
    """First emitted token ~ p_0; given that a second is emitted, it is ~ p_1."""
    rng = np.random.default_rng(seed)
    P = rng.normal(0, 1.5, (gamma + 1, Vv))
    Q = P[:gamma] * 0.7 + rng.normal(0, 0.8, (gamma, Vv))
    q = [softmax(Q[i], T) for i in range(gamma)]
    c0, c1 = np.zeros(Vv), np.zeros(Vv)
    for _ in range(n):
        d = [int(rng.choice(Vv, p=q[i])) for i in range(gamma)]
        r = V.verify_chain_sequence(P, Q, d, rng.random(gamma), rng.random(), T, False)
        emitted = d[: r["accept_len"]] + [r["out_token"]]
        c0[emitted[0]] += 1
        if len(emitted) > 1:
            c1[emitted[1]] += 1
    assert chi2_pvalue(c0, softmax(P[0], T)) > 1e-3
    assert chi2_pvalue(c1, softmax(P[1], T)) > 1e-3


def pin_tree_lossless(V, seed=2, n=12000, Vv=12, T=1.0):
    """Tree walk: the first emitted token follows the root target distribution.
    Children are drawn i.i.d. from q of their parent."""
    rng = np.random.default_rng(seed)
    parent = [-1, 0, 0, 0, 1, 1, 2, 4]
    N = len(parent)
    P = rng.normal(0, 1.5, (N, Vv))
    Q = P * 0.6 + rng.normal(0, 1.0, (N, Vv))
    q = [softmax(Q[i], T) for i in range(N)]
    counts = np.zeros(Vv)
    for _ in range(n):
        tok = [0] + [int(rng.choice(Vv, p=q[parent[i]])) for i in range(1, N)]
        r = V.verify_tree_sequence(parent, tok, P, Q, rng.random(N), rng.random(),
                                   T, False, 3)
        first = tok[r["path"][0]] if r["path"] else r["out_token"]
        counts[first] += 1
    assert chi2_pvalue(counts, softmax(P[0], T)) > 1e-3


def pin_tree_exact_law(V, Vv=3, T=1.0, seed=5):
    """Root with two children drawn i.i.d. from q: exact first-token law.

    For each pair of child tokens, the test enumerates the rule's branches with
    their exact probabilities (keep child 1 with min(1, r1); else keep child 2
    with min(1, r2') under the residual p'; else draw from the second
    residual).  Summed over the child draws this must be p_root (lossless),
    and the oracle, run on a fine grid of the uniforms, must match the
    per-draw law.
    """
    rng = np.random.default_rng(seed)
    parent = [-1, 0, 0]
    P = rng.normal(0, 1.0, (3, Vv))
    Q = rng.normal(0, 1.0, (3, Vv))
    p, q = softmax(P[0], T), softmax(Q[0], T)
    total = np.zeros(Vv)
    n = 20
    grid = (np.arange(n) + 0.5) / n
    for t1 in range(Vv):
        for t2 in range(Vv):
            k1 = min(1.0, p[t1] / q[t1])
            p1 = np.maximum(p - q, 0.0)
            p1 = p1 / p1.sum()
            k2 = min(1.0, p1[t2] / q[t2])
            p2 = np.maximum(p1 - q, 0.0)
            law = np.zeros(Vv)
            law[t1] += k1
            law[t2] += (1 - k1) * k2
            if p2.sum() > 0:
                law += (1 - k1) * (1 - k2) * p2 / p2.sum()
            total += q[t1] * q[t2] * law
            freq = np.zeros(Vv)
            for u1 in grid:
                for u2 in grid:
                    for v in grid:
                        r = V.verify_tree_sequence(parent, [0, t1, t2], P, Q,
                                                   [0.0, u1, u2], v, T, False, 1)
                        tok = [0, t1, t2][r["path"][0]] if r["path"] else r["out_token"]
                        freq[tok] += 1
            freq /= n ** 3
            assert np.abs(freq - law).max() < 2.0 / n + 1e-9, (t1, t2, freq, law)
    assert np.abs(total - p).max() < 1e-12, (total, p)


def pin_cascade_lossless(V, seed=4, n=12000, Vv=10, T=1.0):
    """The first token committed by the final stage follows M_2's row 0."""
    rng = np.random.default_rng(seed)
    g1, g2 = 4, 2
    L0 = rng.normal(0, 1.5, (g1, Vv))
    L1 = np.vstack([L0 * 0.8 + rng.normal(0, 0.7, (g1, Vv)), rng.normal(0, 1.5, (1, Vv))])
    L2 = L1[:g2] * 0.8 + rng.normal(0, 0.9, (g2, Vv))
    q0 = [softmax(L0[j], T) for j in range(g1)]
    counts = np.zeros(Vv)
    for _ in range(n):
        d = [int(rng.choice(Vv, p=q0[j])) for j in range(g1)]
        r = V.verify_cascade_sequence(L0, L1, L2, d, rng.random(g1), rng.random(),
                                      rng.random(g2), rng.random(), T, False)
        o1 = d[: r["a1"]] + [r["t1"]]
        first = o1[0] if r["a2"] >= 1 else r["t2"]
        counts[first] += 1
    assert chi2_pvalue(counts, softmax(L2[0], T)) > 1e-3


def pin_cascade_invariants(V, seed=6, trials=300):
    rng = np.random.default_rng(seed)
    Vv, g1, g2 = 9, 8, 4
    for t in range(trials):
        L0 = rng.normal(0, 1.5, (g1, Vv))
        L1 = np.vstack([L0 * 0.8 + rng.normal(0, 0.7, (g1, Vv)), rng.normal(0, 1.5, (1, Vv))])
        L2 = L1[:g2] * 0.8 + rng.normal(0, 0.9, (g2, Vv))
        mode = t % 3
        if mode == 1:
            L2 = L1[:g2].copy()      # M_2 == M_1: stage 2 keeps all w2
        elif mode == 2:
            L1[:g1] = L0             # M_1 == M_0: stage 1 keeps all g1
        d = [int(x) for x in rng.integers(0, Vv, g1)]
        r = V.verify_cascade_sequence(L0, L1, L2, d, rng.random(g1), rng.random(),
                                      rng.random(g2), rng.random(), 1.0, False)
        assert r["w2"] == min(g2, r["a1"] + 1)
        assert r["r0"] <= r["a1"] and r["r1"] <= r["w2"] and r["committed"] <= r["w2"]
        assert r["committed"] == r["a2"] + r["t2_valid"]
        if mode == 1:
            assert r["a2"] == r["w2"] and r["t2_valid"] == 0
        if mode == 2:
            assert r["a1"] == g1


def pin_tree_chain_shaped(V, seed=7, trials=200):
    """A tree in which every node has one child is a chain: same results."""
    rng = np.random.default_rng(seed)
    Vv, gamma = 11, 4
    for t in range(trials):
        greedy = bool(t % 2)
        P = rng.normal(0, 1.2, (gamma + 1, Vv))
        Q = P[:gamma] * 0.8 + rng.normal(0, 0.6, (gamma, Vv))
        d = [int(x) for x in rng.integers(0, Vv, gamma)]
        u, v = rng.random(gamma), rng.random()
        c = V.verify_chain_sequence(P, Q, d, u, v, 1.1, greedy)
        parent = [-1] + list(range(gamma))
        Qt = np.vstack([Q, np.zeros((1, Vv))])
        tr = V.verify_tree_sequence(parent, [0] + d, P, Qt, [0.0] + list(u), v, 1.1,
                                    greedy, gamma)
        assert len(tr["path"]) == c["accept_len"] and tr["out_token"] == c["out_token"]
        assert tr["path"] == list(range(1, c["accept_len"] + 1))


def pin_gamma_zero(V, seed=8):
    """gamma = 0: every round emits exactly one token (the bonus), matching
    E[tokens] = (1 - alpha)/(1 - alpha) = 1 (PipeSpec referee report, major
    comment 3)."""
    rng = np.random.default_rng(seed)
    P = rng.normal(0, 1, (1, 6))
    counts = np.zeros(6)
    for _ in range(3000):
        r = V.verify_chain_sequence(P, np.zeros((0, 6)), [], [], rng.random(), 1.0, False)
        assert r["accept_len"] == 0
        counts[r["out_token"]] += 1
    assert chi2_pvalue(counts, softmax(P[0])) > 1e-3
    for a in (0.05, 0.3, 0.6, 0.9):
        assert cf.expected_tokens_per_round(a, 0) == 1.0
        for g in (1, 2, 5, 8):
            assert cf.pipespec_expected_tokens(a, g) > 1.0
