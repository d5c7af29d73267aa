"""Chain verification that consults rows in position order (the early exit).

TEST INFRASTRUCTURE ONLY (see the package docstring): only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` call it.

Source: Pith review of "PipeSpec" (arXiv 2505.01572), "What carries the
argument": a stage keeps the longest verified prefix of the buffer it reads;
the tokens after the first mismatch are rolled back without being used.  The
accept and residual rule is the one its Circularity Check cites, as in
``oracle.verify``.

Reading (R15 in the design notes): the verifier consults position i (target
row i, draft row i) only after positions 0 .. i-1 were kept; at the first
rejection a it consults nothing further except what the draw needs (rows a
for the residual); when every draft is kept it consults the bonus row.  The
decisions, the drawn token, the rollback and the residual mass are those of
the ordinary rule (``oracle.verify.verify_chain_sequence``) whenever every
consulted row is finite.  What differs:
  * a non-finite row is a data error only when it is consulted;
  * p(d_i) and q(d_i) exist only for consulted positions: NaN after a;
  * ``rows_read`` counts the logit rows consulted: 2 (a + 1) after a
    rejection at a, 2 gamma + 1 when every draft is kept.
Sampling mode only (greedy verification consults target rows only and has no
draft rows to skip).
"""

from __future__ import annotations

import math

import numpy as np

from .verify import (ERR_NONFINITE, ERR_TOKEN, ERR_ZERO_MASS, accept_ratio, inverse_cdf, keeps, residual,
                     row_is_nonfinite, row_to_float64, temperature_softmax)


def verify_chain_consulted_sequence(target, draft, tokens, u, v, temperature):
    gamma = len(tokens)
    V = target.shape[1]
    out = dict(accept_len=0, out_token=-1, error=0, p_at_draft=np.zeros(gamma), q_at_draft=np.zeros(gamma),
               resid_mass=0.0, margin_u=math.inf, margin_v=math.inf, rows_read=0, min_mass=math.inf)
    if any(t < 0 or t >= V for t in tokens):
        out["error"] = ERR_TOKEN
        return out
    p_at = np.full(gamma, np.nan)
    q_at = np.full(gamma, np.nan)
    a, rows, p, q = gamma, 0, None, None
    for i in range(gamma):
        rows += 2
        if row_is_nonfinite(target[i]) or row_is_nonfinite(draft[i]):
            out.update(error=ERR_NONFINITE, rows_read=rows)
            return out
        p = temperature_softmax(target[i], temperature)
        q = temperature_softmax(draft[i], temperature)
        p_at[i], q_at[i] = p[tokens[i]], q[tokens[i]]
        r = accept_ratio(p[tokens[i]], q[tokens[i]])
        out["margin_u"] = min(out["margin_u"], abs(float(u[i]) - r))
        if not keeps(float(u[i]), r):
            a = i
            break
    error = 0
    if a < gamma:
        weights = residual(p, q)
        out["min_mass"] = float(np.sum(weights))
        if not np.sum(weights) > 0.0:
            error |= ERR_ZERO_MASS
            weights = p
    else:
        rows += 1
        if row_is_nonfinite(target[gamma]):
            out.update(error=ERR_NONFINITE, rows_read=rows)
            return out
        weights = temperature_softmax(target[gamma], temperature)
    tok, Z, margin = inverse_cdf(weights, float(v))
    out.update(accept_len=a, out_token=tok, error=error, p_at_draft=p_at, q_at_draft=q_at, resid_mass=Z,
               margin_v=margin, rows_read=rows)
    return out


def verify_chain_consulted(target, draft, tokens, u, v, prefix_len, temperature, dtype, V=None):
    """Batch wrapper (rows converted to float64 only when consulted); the keys
    of ``oracle.verify.verify_chain`` plus rows_read [B]."""
    B, _, width = target.shape
    V = width if V is None else V
    gamma = tokens.shape[1]
    res = dict(accept_len=np.zeros(B, np.int64), out_token=np.zeros(B, np.int64),
               rollback_idx=np.zeros(B, np.int64), error=np.zeros(B, np.int64),
               p_at_draft=np.zeros((B, gamma)), q_at_draft=np.zeros((B, gamma)), resid_mass=np.zeros(B),
               margin_u=np.zeros(B), margin_v=np.zeros(B), rows_read=np.zeros(B, np.int64),
               min_mass=np.zeros(B))

    class Rows:  # converts a row when it is read
        def __init__(self, arr, n):
            self.arr, self.n = arr, n

        def __getitem__(self, i):
            return row_to_float64(self.arr[i, :V], dtype)

        @property
        def shape(self):
            return (self.n, V)

    for b in range(B):
        r = verify_chain_consulted_sequence(Rows(target[b], gamma + 1), Rows(draft[b], gamma),
                                            [int(t) for t in tokens[b]], u[b], v[b], temperature)
        for k in ("accept_len", "out_token", "error", "resid_mass", "margin_u", "margin_v", "rows_read",
                  "min_mass"):
            res[k][b] = r[k]
        res["p_at_draft"][b] = r["p_at_draft"]
        res["q_at_draft"][b] = r["q_at_draft"]
        res["rollback_idx"][b] = int(prefix_len[b]) + r["accept_len"]
    return res
