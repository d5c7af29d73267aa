"""Tree verification that consults only the rows of the nodes it walks.

TEST INFRASTRUCTURE ONLY (see the package docstring): only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` call it.

Source: "Accelerating LLM Inference with Staged Speculative Decoding"
(arXiv 2308.04623), abstract: the speculative batch is a tree; the walk from
the root keeps one child per level.  Pith review of "PipeSpec", "What
carries the argument": tokens after the first mismatch are never used.  The
accept and residual rule is ``oracle.verify.verify_tree_sequence``'s.

Reading (R18 in the design notes), the tree counterpart of the chain's
consulted mode (R15): the walk reads node n's rows only when it stands at n.
At a visited node it reads the target row (the children's distribution p, or
the argmax in greedy mode) and, in sampling mode when n has children, the
draft row (q for the children's tests); a leaf's draft row is not needed.
The path, the emitted token, the error bits for the zero-mass fallback and
the margins are those of the ordinary rule whenever every consulted row is
finite.  What differs:
  * a non-finite row is a data error only when it is consulted; the walk
    stops there with empty outputs, like the ordinary rule's error;
  * ``rows_read`` counts the rows consulted.
The tree's structure and its tokens are checked as in the ordinary rule
(malformed parents, depth above max_depth, tokens outside [0, V)).
"""

from __future__ import annotations

import math

import numpy as np

from .verify import (ERR_NONFINITE, ERR_PARENT, ERR_TOKEN, ERR_ZERO_MASS, accept_ratio, first_argmax,
                     inverse_cdf, keeps, residual, row_is_nonfinite, row_to_float64, temperature_softmax,
                     tree_depths)


def verify_tree_consulted_sequence(parent, tokens, target, draft, u, v, temperature, greedy, max_depth):
    """One tree (arguments as ``oracle.verify.verify_tree_sequence``; target
    and draft may be lazy row sources: only rows[i] and .shape are used).
    Returns dict(path, out_token, error, margin_u, margin_v, rows_read, min_mass)."""
    N, V = target.shape
    out = dict(path=[], out_token=-1, error=0, margin_u=math.inf, margin_v=math.inf, rows_read=0,
               min_mass=math.inf)
    error = 0
    depth = tree_depths([int(x) for x in parent])
    if depth is None or max(depth) > max_depth:
        error |= ERR_PARENT
    if any(not (0 <= int(tokens[i]) < V) for i in range(1, N)):
        error |= ERR_TOKEN
    if error:
        out["error"] = error
        return out
    children = [[] for _ in range(N)]
    for i in range(1, N):
        children[int(parent[i])].append(i)

    node, path, rows = 0, [], 0
    while True:
        kids = children[node]
        t_row = target[node]
        rows += 1
        if row_is_nonfinite(t_row):
            out.update(error=ERR_NONFINITE, rows_read=rows)
            return out
        if greedy:
            best = first_argmax(t_row)
            kept = next((c for c in kids if int(tokens[c]) == best), None)
            if kept is None:
                out.update(path=path, out_token=best, rows_read=rows)
                return out
            path.append(kept)
            node = kept
            continue
        p_node = temperature_softmax(t_row, temperature)
        p = p_node
        kept = None
        zero_mass = False
        if kids:
            d_row = draft[node]
            rows += 1
            if row_is_nonfinite(d_row):
                out.update(error=ERR_NONFINITE, rows_read=rows)
                return out
            q = temperature_softmax(d_row, temperature)
            for c in kids:
                t = int(tokens[c])
                r = accept_ratio(p[t], q[t])
                out["margin_u"] = min(out["margin_u"], abs(float(u[c]) - r))
                if keeps(float(u[c]), r):
                    kept = c
                    break
                nxt = residual(p, q)
                mass = float(np.sum(nxt))
                out["min_mass"] = min(out["min_mass"], mass)
                if not mass > 0.0:
                    zero_mass = True
                    break
                p = nxt / mass
        if kept is not None:
            path.append(kept)
            node = kept
            continue
        if zero_mass:
            error |= ERR_ZERO_MASS
            p = p_node
        tok, _, margin = inverse_cdf(p, float(v))
        out.update(path=path, out_token=tok, error=error, margin_v=margin, rows_read=rows)
        return out


def verify_tree_consulted(parent, tokens, target, draft, u, v, prefix_len, temperature, greedy, max_depth, dtype,
                          V=None):
    """Batch wrapper (rows converted to float64 only when consulted); the keys
    of ``oracle.verify.verify_tree`` plus rows_read [B]."""
    B, N, width = target.shape
    V = width if V is None else V
    res = dict(path_len=np.zeros(B, np.int64), path_nodes=-np.ones((B, max_depth + 1), np.int64),
               out_token=np.zeros(B, np.int64), rollback_idx=np.zeros(B, np.int64),
               error=np.zeros(B, np.int64), margin_u=np.zeros(B), margin_v=np.zeros(B),
               rows_read=np.zeros(B, np.int64), min_mass=np.zeros(B))

    class Rows:  # converts a row when it is read
        def __init__(self, arr):
            self.arr = arr

        def __getitem__(self, i):
            return row_to_float64(self.arr[i, :V], dtype)

        @property
        def shape(self):
            return (N, V)

    for b in range(B):
        r = verify_tree_consulted_sequence(parent[b], tokens[b], Rows(target[b]),
                                           None if greedy else Rows(draft[b]), None if greedy else u[b],
                                           None if greedy else v[b], temperature, greedy, max_depth)
        for k in ("out_token", "error", "margin_u", "margin_v", "rows_read", "min_mass"):
            res[k][b] = r[k]
        res["path_len"][b] = len(r["path"])
        if r["error"] & (ERR_TOKEN | ERR_PARENT | ERR_NONFINITE) == 0:
            nodes = [0] + list(r["path"])
            res["path_nodes"][b, :len(nodes)] = nodes
        res["rollback_idx"][b] = int(prefix_len[b]) + len(r["path"])
    return res
