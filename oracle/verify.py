"""Batched draft verification, written out step by step in float64 NumPy.

TEST INFRASTRUCTURE ONLY (see the package docstring): only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` call it.

Sources (the pages):
  * Pith review of "PipeSpec: Breaking Stage Dependencies in Hierarchical LLM
    Decoding" (arXiv 2505.01572).  "What carries the argument": each stage
    verifies the previous buffer against its own prediction, appends the
    longest matching prefix and, on a mismatch, rolls the earlier buffers back
    to the last verified token.  "Circularity Check": the acceptance formula is
    the one of Leviathan et al.  "Reading between the lines": the reported runs
    use greedy decoding (temperature 0).
  * "Accelerating LLM Inference with Staged Speculative Decoding"
    (arXiv 2308.04623), abstract: the speculative batch is restructured as a
    tree, and a second speculative stage is added.
  * Pith review of "CLaSp: In-Context Layer Skip for Self-Speculative Decoding"
    (arXiv 2505.24196), "Assumptions & free parameters": speculative sampling
    with a matching draft distribution is lossless.

The pages name the sampling rule only by citation.  The rule followed here is
the standard one they cite: a drafted token x is kept when u < min(1, p(x)/q(x))
for a uniform u, and at the first rejection a replacement is drawn from the
residual distribution max(0, p - q) renormalised; when every draft is kept, a
bonus token is drawn from the next target distribution.  p and q are the
temperature softmaxes of the target and draft logits.

Readings where the pages are silent (each also listed in the design notes):
  R1  the accept test is strict: u < min(1, r), u in [0, 1); so r >= 1 keeps.
  R2  q(x) == 0: r = +inf (keep) when p(x) > 0; both zero: reject.
  R3  a zero residual mass after a rejection: draw from p instead and set
      error bit ERR_ZERO_MASS.
  R4  greedy: ties in the argmax go to the lowest index; greedy ignores the
      temperature and compares raw logits.
  R5  the inverse CDF runs over ascending vocabulary index and returns the
      first y whose running sum exceeds v * Z (strictly).
  R6  u[b, i] is used only for the test at position i; one v per draw.
  R7  a row containing NaN or +inf, or with no finite entry, is a data error
      (ERR_NONFINITE); so is a drafted token outside [0, V) (ERR_TOKEN) and a
      malformed parent array (ERR_PARENT).  A sequence with a data error gets
      empty outputs (accept length 0, token -1, rollback = prefix length).
  R8  tree: row n of the target / draft logits is the distribution over the
      children of node n; node 0 is the root; children are tried in ascending
      node index; after a rejected sibling p becomes norm(max(0, p - q)) with
      q unchanged; a leaf draws its bonus from its own target row.
  R9  cascade: one synchronous snapshot of a 3-model pipeline; stage 2
      verifies the first min(gamma2, a1 + 1) tokens of the stage-1 output
      with p = M_2 and q = M_1 and draws no bonus when it keeps them all.

Every accept test and every inverse-CDF draw also records how close it came to
flipping (``margin_u`` = |u - r|; ``margin_v`` = distance of v*Z to the
nearest bracketing running sum, divided by Z) so that parity tests can set
aside decisions a faithful float32 implementation may legitimately take the
other way.  ``min_mass`` is the smallest mass of a residual distribution
max(0, p - q) formed after a rejection (inf when no rejection forms one): it
is exactly 0 when reading R3 applies, and a small positive value means the
residual is the difference of two nearly equal distributions, which a
float32 implementation resolves only to its rounding (the zero-mass fallback
and the draw may then go either way).
"""

from __future__ import annotations

import math

import numpy as np

ERR_TOKEN = 1
ERR_PARENT = 2
ERR_NONFINITE = 4
ERR_ZERO_MASS = 8


# --------------------------------------------------------------------------
# exact conversion of the stored logits
# --------------------------------------------------------------------------

def bf16_bits_to_float64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64, exactly.

    A bfloat16 value is the top half of a float32, so shifting the pattern
    into the high 16 bits of a 32-bit word gives the float32 with the same
    value; widening to float64 is exact.
    """
    wide = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return wide.view(np.float32).astype(np.float64)


def row_to_float64(row: np.ndarray, dtype: str) -> np.ndarray:
    """One stored logit row (float32 values or bfloat16 bits) as float64."""
    if dtype == "bf16":
        return bf16_bits_to_float64(row)
    if dtype == "f32":
        return np.asarray(row, dtype=np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# --------------------------------------------------------------------------
# per-row primitives
# --------------------------------------------------------------------------

def temperature_softmax(logits: np.ndarray, temperature: float) -> np.ndarray:
    """p(x) = exp(l(x)/T) / sum_y exp(l(y)/T), with the max subtracted first."""
    z = logits / float(temperature)
    z = z - np.max(z)
    e = np.exp(z)
    return e / np.sum(e)


def log_partition(logits: np.ndarray, temperature: float) -> float:
    """log sum_x exp(l(x)/T) = m + log sum_x exp(l(x)/T - m), m = max l/T."""
    z = logits / float(temperature)
    m = float(np.max(z))
    return m + math.log(float(np.sum(np.exp(z - m))))


def first_argmax(logits: np.ndarray) -> int:
    """Index of the largest logit; ties go to the lowest index (reading R4)."""
    best = np.max(logits)
    return int(np.flatnonzero(logits == best)[0])


def row_is_nonfinite(logits: np.ndarray) -> bool:
    """Reading R7: NaN or +inf anywhere, or no finite entry at all."""
    return bool(np.isnan(logits).any() or np.isposinf(logits).any()
                or not np.isfinite(logits).any())


def accept_ratio(p_tok: float, q_tok: float) -> float:
    """r = p(x)/q(x) with reading R2 for q(x) == 0."""
    if q_tok > 0.0:
        return p_tok / q_tok
    return math.inf if p_tok > 0.0 else 0.0


def keeps(u: float, ratio: float) -> bool:
    """The accept test u < min(1, r) (reading R1)."""
    return u < min(1.0, ratio)


def inverse_cdf(weights: np.ndarray, v: float) -> tuple[int, float, float]:
    """Draw from weights / sum(weights) with the uniform v (reading R5).

    Returns (index, Z, margin): the first y whose running sum C(y) exceeds
    v * Z, the total Z, and min(|v Z - C(y)|, |v Z - C(y-1)|) / Z.
    The running sums are taken in ascending index order.  Z must be > 0.
    """
    running = np.cumsum(weights)
    total = float(running[-1])
    target = float(v) * total
    above = np.flatnonzero(running > target)
    if above.size:
        y = int(above[0])
    else:  # only when v * Z rounds up to Z: take the last index with mass
        y = int(np.flatnonzero(weights > 0)[-1])
    below = float(running[y - 1]) if y > 0 else 0.0
    margin = min(abs(target - float(running[y])), abs(target - below)) / total
    return y, total, margin


def residual(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """Unnormalised residual max(0, p - q), drawn from after a rejection."""
    return np.maximum(p - q, 0.0)


# --------------------------------------------------------------------------
# chain verification
# --------------------------------------------------------------------------

def verify_chain_sequence(target, draft, tokens, u, v, temperature, greedy):
    """Verify one gamma-token draft chain.

    target  float64 [gamma+1, V]  target logits; row i scores position i,
                                  row gamma is the bonus position
    draft   float64 [gamma, V]    draft logits (ignored when greedy)
    tokens  int [gamma]           drafted tokens
    u       float [gamma]         accept uniforms (sampling only)
    v       float                 uniform for the one draw (sampling only)

    Returns a dict: accept_len, out_token, error, p_at_draft, q_at_draft,
    resid_mass, margin_u, margin_v, min_mass.
    """
    gamma = len(tokens)
    V = target.shape[1]
    out = dict(accept_len=0, out_token=-1, error=0,
               p_at_draft=np.zeros(gamma), q_at_draft=np.zeros(gamma),
               resid_mass=0.0, margin_u=math.inf, margin_v=math.inf,
               min_mass=math.inf)
    error = 0
    if any(t < 0 or t >= V for t in tokens):
        error |= ERR_TOKEN
    rows = [target[i] for i in range(gamma + 1)]
    if not greedy:
        rows += [draft[i] for i in range(gamma)]
    if any(row_is_nonfinite(r) for r in rows):
        error |= ERR_NONFINITE
    if error:
        out["error"] = error
        return out

    if greedy:
        # keep while the draft equals the target argmax; emit the target
        # argmax where the chain stops (reading R4)
        for i in range(gamma):
            best = first_argmax(target[i])
            if tokens[i] != best:
                out.update(accept_len=i, out_token=best)
                return out
        out.update(accept_len=gamma, out_token=first_argmax(target[gamma]))
        return out

    p_rows = [temperature_softmax(target[i], temperature) for i in range(gamma + 1)]
    q_rows = [temperature_softmax(draft[i], temperature) for i in range(gamma)]
    for i in range(gamma):
        out["p_at_draft"][i] = p_rows[i][tokens[i]]
        out["q_at_draft"][i] = q_rows[i][tokens[i]]

    a = gamma
    for i in range(gamma):
        r = accept_ratio(p_rows[i][tokens[i]], q_rows[i][tokens[i]])
        out["margin_u"] = min(out["margin_u"], abs(float(u[i]) - r))
        if not keeps(float(u[i]), r):
            a = i
            break
    if a < gamma:
        weights = residual(p_rows[a], q_rows[a])
        out["min_mass"] = float(np.sum(weights))
        if not np.sum(weights) > 0.0:  # reading R3
            error |= ERR_ZERO_MASS
            weights = p_rows[a]
    else:
        weights = p_rows[gamma]
    tok, mass, margin = inverse_cdf(weights, float(v))
    out.update(accept_len=a, out_token=tok, error=error, resid_mass=mass,
               margin_v=margin)
    return out


def verify_chain(target, draft, tokens, u, v, prefix_len, temperature,
                 greedy, dtype, V=None):
    """Batch wrapper: rows are converted to float64 one sequence at a time.

    target [B, gamma+1, ld] and draft [B, gamma, ld] hold float32 values or
    bfloat16 bits (``dtype``); only the first V = ``target.shape[2]`` columns
    are logits when ld is the full width.  Returns arrays per sequence plus
    rollback_idx = prefix_len + accept_len (the buffer length to keep;
    "What carries the argument": roll back to the last verified token).
    """
    B, _, width = target.shape
    V = width if V is None else V
    gamma = tokens.shape[1]
    res = dict(accept_len=np.zeros(B, np.int64), out_token=np.zeros(B, np.int64),
               rollback_idx=np.zeros(B, np.int64), error=np.zeros(B, np.int64),
               p_at_draft=np.zeros((B, gamma)), q_at_draft=np.zeros((B, gamma)),
               resid_mass=np.zeros(B), margin_u=np.zeros(B), margin_v=np.zeros(B),
               min_mass=np.zeros(B))
    for b in range(B):
        tgt = np.stack([row_to_float64(target[b, i, :V], dtype) for i in range(gamma + 1)])
        drf = None
        if not greedy:
            drf = np.stack([row_to_float64(draft[b, i, :V], dtype) for i in range(gamma)]) \
                if gamma else np.zeros((0, V))
        r = verify_chain_sequence(tgt, drf, [int(t) for t in tokens[b]],
                                  None if greedy else u[b],
                                  None if greedy else v[b], temperature, greedy)
        for k in ("accept_len", "out_token", "error", "resid_mass",
                  "margin_u", "margin_v", "min_mass"):
            res[k][b] = r[k]
        res["p_at_draft"][b] = r["p_at_draft"]
        res["q_at_draft"][b] = r["q_at_draft"]
        res["rollback_idx"][b] = int(prefix_len[b]) + r["accept_len"]
    return res


# --------------------------------------------------------------------------
# tree verification (Staged Speculative Decoding: the speculative batch as a tree)
# --------------------------------------------------------------------------

def tree_depths(parent):
    """Depth of every node, or None when the parent array is malformed.

    Well formed: parent[0] == -1 and 0 <= parent[i] < i for i >= 1.
    """
    n = len(parent)
    if n == 0 or parent[0] != -1:
        return None
    depth = [0] * n
    for i in range(1, n):
        p = parent[i]
        if p < 0 or p >= i:
            return None
        depth[i] = depth[p] + 1
    return depth


def verify_tree_sequence(parent, tokens, target, draft, u, v, temperature,
                         greedy, max_depth):
    """Walk one draft tree from the root (readings R8, R1-R7).

    parent  int [N]            parent[0] = -1; node 0 is the root
    tokens  int [N]            token of each node (tokens[0] unused)
    target  float64 [N, V]     row n: target logits over the children of n
    draft   float64 [N, V]     row n: draft logits over the children of n
    u       float [N]          u[c] is the uniform of node c's own test
    v       float              uniform for the final draw

    Sampling: at node n the children are tried in ascending index against the
    current distribution p (initially softmax of target row n).  A kept child
    becomes the new node.  A rejected child replaces p by norm(max(0, p - q))
    before the next sibling is tried.  When no child is kept the token is drawn
    from the current p (from p_n itself at a leaf).
    Greedy: the first child whose token equals the target argmax of row n is
    kept; otherwise the argmax is emitted.
    """
    N, V = target.shape
    out = dict(path=[], out_token=-1, error=0, margin_u=math.inf,
               margin_v=math.inf, min_mass=math.inf)
    error = 0
    depth = tree_depths([int(x) for x in parent])
    if depth is None or max(depth) > max_depth:
        error |= ERR_PARENT
    if any(not (0 <= int(tokens[i]) < V) for i in range(1, N)):
        error |= ERR_TOKEN
    rows = [target[i] for i in range(N)]
    if not greedy:
        rows += [draft[i] for i in range(N)]
    if any(row_is_nonfinite(r) for r in rows):
        error |= ERR_NONFINITE
    if error:
        out["error"] = error
        return out

    children = [[] for _ in range(N)]
    for i in range(1, N):
        children[int(parent[i])].append(i)

    node = 0
    path = []
    while True:
        kids = children[node]
        if greedy:
            best = first_argmax(target[node])
            kept = next((c for c in kids if int(tokens[c]) == best), None)
            if kept is None:
                out.update(path=path, out_token=best)
                return out
            path.append(kept)
            node = kept
            continue

        p_node = temperature_softmax(target[node], temperature)
        q = temperature_softmax(draft[node], temperature)
        p = p_node
        kept = None
        zero_mass = False
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
            if not mass > 0.0:  # reading R3
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
        out.update(path=path, out_token=tok, error=error, margin_v=margin)
        return out


def verify_tree(parent, tokens, target, draft, u, v, prefix_len, temperature,
                greedy, max_depth, dtype, V=None):
    """Batch wrapper for the tree walk.

    Returns path_len [B], path_nodes [B, max_depth+1] (root first, then the
    kept nodes, -1 padded; all -1 on a data error), out_token, rollback_idx
    (= prefix_len + path_len), error, margin_u, margin_v, min_mass.
    """
    B, N, width = target.shape
    V = width if V is None else V
    res = dict(path_len=np.zeros(B, np.int64),
               path_nodes=-np.ones((B, max_depth + 1), np.int64),
               out_token=np.zeros(B, np.int64), rollback_idx=np.zeros(B, np.int64),
               error=np.zeros(B, np.int64), margin_u=np.zeros(B),
               margin_v=np.zeros(B), min_mass=np.zeros(B))
    for b in range(B):
        tgt = np.stack([row_to_float64(target[b, i, :V], dtype) for i in range(N)])
        drf = None if greedy else np.stack(
            [row_to_float64(draft[b, i, :V], dtype) for i in range(N)])
        r = verify_tree_sequence(parent[b], tokens[b], tgt, drf,
                                 None if greedy else u[b],
                                 None if greedy else v[b], temperature, greedy,
                                 max_depth)
        res["error"][b] = r["error"]
        res["out_token"][b] = r["out_token"]
        res["margin_u"][b] = r["margin_u"]
        res["margin_v"][b] = r["margin_v"]
        res["min_mass"][b] = r["min_mass"]
        res["path_len"][b] = len(r["path"])
        if r["error"] & (ERR_TOKEN | ERR_PARENT | ERR_NONFINITE) == 0:
            nodes = [0] + list(r["path"])
            res["path_nodes"][b, :len(nodes)] = nodes
        res["rollback_idx"][b] = int(prefix_len[b]) + len(r["path"])
    return res


# --------------------------------------------------------------------------
# PipeSpec 3-model cascade, one synchronous snapshot (reading R9)
# --------------------------------------------------------------------------

def verify_cascade_sequence(l0, l1, l2, tokens, u1, v1, u2, v2, temperature,
                            greedy):
    """One snapshot of the M_0 -> M_1 -> M_2 pipeline for one sequence.

    l0  float64 [g1, V]     M_0 (draft) logits for the O_0 window
    l1  float64 [g1+1, V]   M_1 logits; row g1 is M_1's bonus position
    l2  float64 [g2, V]     M_2 logits for the first g2 positions
    tokens int [g1]         the O_0 window drafted by M_0

    Stage 1 ("What carries the argument": M_1 reads O_0 and verifies it
    against its own prediction) is the chain rule with p = M_1, q = M_0 and
    gives a1 and the correction / bonus t1; O_1 = tokens[:a1] + [t1].
    Stage 2 is the chain rule with p = M_2, q = M_1 over the first
    w2 = min(g2, a1 + 1) tokens of O_1; it draws a correction t2 on a
    rejection and no bonus otherwise (t2_valid = 0).  A final-stage mismatch
    rolls the earlier buffer back too: r0 = min(a1, a2) on a rejection, else
    a1; r1 = a2 on a rejection, else w2; committed = a2 + t2_valid.
    """
    g1 = len(tokens)
    g2 = l2.shape[0]
    V = l1.shape[1]
    out = dict(a1=0, t1=-1, a2=0, w2=0, t2=-1, t2_valid=0, r0=0, r1=0,
               committed=0, error=0, margin_u=math.inf, margin_v=math.inf,
               min_mass=math.inf)
    error = 0
    if any(t < 0 or t >= V for t in tokens):
        error |= ERR_TOKEN
    rows = [l1[i] for i in range(g1 + 1)] + [l2[i] for i in range(g2)]
    if not greedy:
        rows += [l0[i] for i in range(g1)]
    if any(row_is_nonfinite(r) for r in rows):
        error |= ERR_NONFINITE
    if error:
        out["error"] = error
        return out

    def note_u(u, r):
        out["margin_u"] = min(out["margin_u"], abs(float(u) - r))

    if greedy:
        a1 = g1
        for j in range(g1):
            if tokens[j] != first_argmax(l1[j]):
                a1 = j
                break
        t1 = first_argmax(l1[a1])
        o1 = list(tokens[:a1]) + [t1]
        w2 = min(g2, a1 + 1)
        a2 = w2
        for j in range(w2):
            if o1[j] != first_argmax(l2[j]):
                a2 = j
                break
        t2, t2_valid = (first_argmax(l2[a2]), 1) if a2 < w2 else (-1, 0)
    else:
        p0 = [temperature_softmax(l0[j], temperature) for j in range(g1)]
        p1 = [temperature_softmax(l1[j], temperature) for j in range(g1 + 1)]
        p2 = [temperature_softmax(l2[j], temperature) for j in range(g2)]
        # stage 1: M_1 verifies O_0 (q = M_0)
        a1 = g1
        for j in range(g1):
            r = accept_ratio(p1[j][tokens[j]], p0[j][tokens[j]])
            note_u(u1[j], r)
            if not keeps(float(u1[j]), r):
                a1 = j
                break
        weights = residual(p1[a1], p0[a1]) if a1 < g1 else p1[g1]
        if a1 < g1:
            out["min_mass"] = float(np.sum(weights))
        if not np.sum(weights) > 0.0:
            error |= ERR_ZERO_MASS
            weights = p1[a1]
        t1, _, m = inverse_cdf(weights, float(v1))
        out["margin_v"] = min(out["margin_v"], m)
        o1 = list(tokens[:a1]) + [t1]
        # stage 2: M_2 verifies the first w2 tokens of O_1 (q = M_1)
        w2 = min(g2, a1 + 1)
        a2 = w2
        for j in range(w2):
            r = accept_ratio(p2[j][o1[j]], p1[j][o1[j]])
            note_u(u2[j], r)
            if not keeps(float(u2[j]), r):
                a2 = j
                break
        if a2 < w2:
            weights = residual(p2[a2], p1[a2])
            out["min_mass"] = min(out["min_mass"], float(np.sum(weights)))
            if not np.sum(weights) > 0.0:
                error |= ERR_ZERO_MASS
                weights = p2[a2]
            t2, _, m = inverse_cdf(weights, float(v2))
            out["margin_v"] = min(out["margin_v"], m)
            t2_valid = 1
        else:
            t2, t2_valid = -1, 0

    rejected = a2 < w2
    out.update(a1=a1, t1=t1, a2=a2, w2=w2, t2=t2, t2_valid=t2_valid,
               r0=min(a1, a2) if rejected else a1,
               r1=a2 if rejected else w2,
               committed=a2 + t2_valid, error=error)
    return out


def verify_cascade(l0, l1, l2, tokens, u1, v1, u2, v2, base0, base1,
                   temperature, greedy, dtype, V=None):
    """Batch wrapper for the cascade; r0 / r1 are returned as absolute buffer
    lengths base0 + r0 and base1 + r1 (on a data error: base0 and base1)."""
    B, g1p1, width = l1.shape
    V = width if V is None else V
    g1 = g1p1 - 1
    g2 = l2.shape[1]
    keys = ("a1", "t1", "a2", "w2", "t2", "t2_valid", "r0", "r1",
            "committed", "error")
    res = {k: np.zeros(B, np.int64) for k in keys}
    res["margin_u"] = np.zeros(B)
    res["margin_v"] = np.zeros(B)
    res["min_mass"] = np.zeros(B)
    for b in range(B):
        m1 = np.stack([row_to_float64(l1[b, i, :V], dtype) for i in range(g1 + 1)])
        m2 = np.stack([row_to_float64(l2[b, i, :V], dtype) for i in range(g2)])
        m0 = None if greedy else np.stack(
            [row_to_float64(l0[b, i, :V], dtype) for i in range(g1)])
        r = verify_cascade_sequence(
            m0, m1, m2, [int(t) for t in tokens[b]],
            None if greedy else u1[b], None if greedy else v1[b],
            None if greedy else u2[b], None if greedy else v2[b],
            temperature, greedy)
        for k in keys:
            res[k][b] = r[k]
        res["margin_u"][b] = r["margin_u"]
        res["margin_v"][b] = r["margin_v"]
        res["min_mass"][b] = r["min_mass"]
        res["r0"][b] += int(base0[b])
        res["r1"][b] += int(base1[b])
    return res


# --------------------------------------------------------------------------
# helpers for input calibration and statistics
# --------------------------------------------------------------------------

def acceptance_rate(target_row, draft_row, temperature):
    """alpha = sum_x min(p(x), q(x)): the probability that a token drawn from
    q passes the accept test (sum_x q(x) min(1, p(x)/q(x)))."""
    p = temperature_softmax(target_row, temperature)
    q = temperature_softmax(draft_row, temperature)
    return float(np.sum(np.minimum(p, q)))
