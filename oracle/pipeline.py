"""k-model PipeSpec snapshot, written out step by step in float64 NumPy.

TEST INFRASTRUCTURE ONLY (see the package docstring): only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` call it.

Source: Pith review of "PipeSpec: Breaking Stage Dependencies in Hierarchical
LLM Decoding" (arXiv 2505.01572), "What carries the argument": a k-model
pipeline in which M_0 drafts into buffer O_0 and each later M_i reads
O_{i-1}, verifies it against its own prediction, appends the longest
matching prefix to O_i, and on a mismatch rolls every earlier buffer back to
the last verified token; "If this is right": more stages scale the benefit.
The accept and residual rule is the one the review's Circularity Check cites
(Leviathan et al.), as in ``oracle.verify``.

Readings (listed in the design notes as R14): one synchronous snapshot in
which every stage's window starts at the beginning of the buffer below it.
  * Stage 1 is the chain rule with p = M_1, q = M_0 over the g_1 drafted
    tokens; it always emits one token (the correction at the first
    rejection, else the bonus from M_1's row g_1): O_1 = d[:a_1] + [t_1].
  * Stage s >= 2 is the chain rule with p = M_s, q = M_{s-1} over the first
    w_s = min(g_s, len(O_{s-1})) tokens of O_{s-1}.  On a rejection at a_s it
    draws the correction t_s and O_s = O_{s-1}[:a_s] + [t_s].  When all w_s
    are kept it emits nothing, O_s = O_{s-1}[:w_s]; except the last stage
    when `final_bonus` is set, which then draws a bonus token from M_s's row
    w_s (that stage passes one more row).
  * Rollback: buffer O_j (j = 0 .. k-2) keeps r_j = min(L_j, a_s over every
    stage s > j that rejected), with L_0 = a_1 (what M_1 verified of O_0) and
    L_j = w_{j+1} for j >= 1 (what M_{j+1} consumed of O_j).
  * committed = len(O_{k-1}).
For k = 3 without the bonus this is ``oracle.verify.verify_cascade`` (r_0,
r_1 and committed as there); for k = 2 it is the chain rule
(``oracle.verify.verify_chain``: a_1, t_1, rollback a_1).
"""

from __future__ import annotations

import math

import numpy as np

from .verify import (ERR_NONFINITE, ERR_TOKEN, ERR_ZERO_MASS, accept_ratio, first_argmax, inverse_cdf, keeps,
                     residual, row_is_nonfinite, row_to_float64, temperature_softmax)


def verify_pipeline_sequence(models, tokens, us, vs, temperature, greedy, final_bonus):
    """One snapshot of the M_0 -> ... -> M_{k-1} pipeline for one sequence.

    models  list of k float64 arrays [rows_s, V]: models[0] has g_1 rows (M_0
            at the drafted positions; unused in greedy mode), models[1] g_1 + 1
            rows, models[s] (s >= 2) g_s rows, plus one for the last stage when
            final_bonus
    tokens  int [g_1], drafted by M_0
    us      list of k - 1 arrays: us[s-1] holds stage s's accept uniforms
    vs      list of k - 1 draw uniforms
    Returns dict(a, w, t, t_valid: lists over stages 1..k-1; r: list over
    buffers 0..k-2; committed, error, margin_u, margin_v, min_mass).
    """
    k = len(models)
    g1 = len(tokens)
    V = models[1].shape[1]
    gs = [g1] + [models[s].shape[0] - (1 if (final_bonus and s == k - 1) else 0) for s in range(2, k)]
    out = dict(a=[0] * (k - 1), w=[0] * (k - 1), t=[-1] * (k - 1), t_valid=[0] * (k - 1), r=[0] * (k - 1),
               committed=0, error=0, margin_u=math.inf, margin_v=math.inf, min_mass=math.inf)
    error = 0
    if any(t < 0 or t >= V for t in tokens):
        error |= ERR_TOKEN
    rows = [models[s][i] for s in range(0 if not greedy else 1, k) for i in range(models[s].shape[0])]
    if any(row_is_nonfinite(r) for r in rows):
        error |= ERR_NONFINITE
    if error:
        out["error"] = error
        return out

    probs = None if greedy else [
        [temperature_softmax(models[s][i], temperature) for i in range(models[s].shape[0])] for s in range(k)]

    def draw(weights, v, fallback):
        nonlocal error
        if weights is not fallback:  # a residual, formed after a rejection
            out["min_mass"] = min(out["min_mass"], float(np.sum(weights)))
        if not np.sum(weights) > 0.0:
            error |= ERR_ZERO_MASS
            weights = fallback
        tok, _, m = inverse_cdf(weights, float(v))
        out["margin_v"] = min(out["margin_v"], m)
        return tok

    buf = list(tokens)  # O_{s-1}
    rejected = []
    for s in range(1, k):
        g = gs[s - 1]
        w = g1 if s == 1 else min(g, len(buf))
        a = w
        for j in range(w):
            if greedy:
                ok = buf[j] == first_argmax(models[s][j])
            else:
                r = accept_ratio(probs[s][j][buf[j]], probs[s - 1][j][buf[j]])
                out["margin_u"] = min(out["margin_u"], abs(float(us[s - 1][j]) - r))
                ok = keeps(float(us[s - 1][j]), r)
            if not ok:
                a = j
                break
        bonus = s == 1 or (final_bonus and s == k - 1)
        if a < w:
            tok = first_argmax(models[s][a]) if greedy else draw(residual(probs[s][a], probs[s - 1][a]),
                                                                   vs[s - 1], probs[s][a])
            nxt, valid = buf[:a] + [tok], 1
            rejected.append((s, a))
        elif bonus:
            tok = first_argmax(models[s][w]) if greedy else draw(probs[s][w], vs[s - 1], probs[s][w])
            nxt, valid = buf[:w] + [tok], 1
        else:
            tok, nxt, valid = -1, buf[:w], 0
        out["a"][s - 1], out["w"][s - 1], out["t"][s - 1], out["t_valid"][s - 1] = a, w, tok, valid
        buf = nxt
    for j in range(k - 1):
        L = out["a"][0] if j == 0 else out["w"][j]
        out["r"][j] = min([L] + [a for s, a in rejected if s > j])
    out["committed"] = len(buf)
    out["error"] = error
    return out


def verify_pipeline(models, tokens, us, vs, temperature, greedy, final_bonus, dtype, V=None, base=None):
    """Batch wrapper.  models: list of k stored logit arrays [B, rows_s, ld]
    (models[0] may be None in greedy mode); tokens [B, g_1]; us: list of k - 1
    arrays [B, rows]; vs: list of k - 1 arrays [B]; base [k - 1, B] or None:
    buffer lengths before the snapshot, added to the rollback lengths (on a
    data error r_j = base_j).  Returns arrays a, w, t, t_valid [B, k-1], r
    [B, k-1], committed [B], error [B], margin_u, margin_v, min_mass [B]."""
    k = len(models)
    B = tokens.shape[0]
    V = models[1].shape[2] if V is None else V
    res = {n: np.zeros((B, k - 1), np.int64) for n in ("a", "w", "t", "t_valid", "r")}
    res.update(committed=np.zeros(B, np.int64), error=np.zeros(B, np.int64), margin_u=np.zeros(B),
               margin_v=np.zeros(B), min_mass=np.zeros(B))
    for b in range(B):
        ms = [None if (greedy and s == 0) else
              np.stack([row_to_float64(models[s][b, i, :V], dtype) for i in range(models[s].shape[1])])
              for s in range(k)]
        r = verify_pipeline_sequence(ms, [int(x) for x in tokens[b]],
                                     None if greedy else [u[b] for u in us],
                                     None if greedy else [v[b] for v in vs], temperature, greedy, final_bonus)
        for n in ("a", "w", "t", "t_valid", "r"):
            res[n][b] = r[n]
        for n in ("committed", "error", "margin_u", "margin_v", "min_mass"):
            res[n][b] = r[n]
        if base is not None:
            res["r"][b] += np.asarray([int(base[j][b]) for j in range(k - 1)])
    return res
