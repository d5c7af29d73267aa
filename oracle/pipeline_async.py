"""PipeSpec stages at independent buffer offsets (the asynchronous snapshot).

TEST INFRASTRUCTURE ONLY (see the package docstring): only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` call it.

Source: Pith review of "PipeSpec: Breaking Stage Dependencies in Hierarchical
LLM Decoding" (arXiv 2505.01572), "What carries the argument": the k models
run without global synchronisation; M_0 keeps writing drafts to O_0, each
later M_i reads O_{i-1}, checks it against its own prediction, appends the
longest matching prefix to O_i, and a mismatch makes every earlier stage roll
its buffer back to the last verified token.  "What would settle it" and the
referee report's first comment: the analysis assumes a verifier always finds
a full window waiting in the buffer below it.

Reading (R17 in the design notes): one snapshot in which every stage s = 1 ..
k-1 verifies, at the same time and independently of the others, the w_s
tokens of O_{s-1} that follow what O_s already holds:
  * buffer lengths before the snapshot are l_0 .. l_{k-1}; stage s reads the
    window O_{s-1}[l_s : l_s + w_s], which must already be there
    (l_{s-1} >= l_s + w_s, the full-window assumption; otherwise the
    sequence is malformed: ERR_WINDOW and no change, the stages' own data
    errors reported beside it);
  * stage s is the chain rule with p = M_s and q = M_{s-1} at the window's
    positions (``oracle.verify.verify_chain_sequence``, M_s passing w_s + 1
    rows: the window's and the one after it);
  * emission: a stage emits the correction on a rejection.  When every
    window token is kept, stage 1 and (with `final_bonus`) the last stage
    emit the bonus drawn from M_s's row w_s, as in the synchronous snapshot
    (R14), but only when that position l_s + w_s is still empty in the
    buffer below once that buffer's own stage has appended in this snapshot
    (O_0 does not grow; O_{s-1} grows by a_{s-1} plus its emitted token): a
    bonus there would stand beside a token no verifier has checked, so the
    stage leaves the position to a later snapshot; middle stages emit
    nothing;
  * O_s grows to l_s + a_s (+1 when it emits); a rejection of stage s at
    position P_s = l_s + a_s rolls every earlier buffer back to at most P_s
    (the rejected token and everything after it were built on a token the
    verifier refused): r_j = min(new length of O_j, P_s over every stage
    s > j that rejected), with O_0's new length l_0 (M_0's own drafting is
    outside the snapshot);
  * committed = r_{k-1}, the final buffer's new length.
"""

from __future__ import annotations

import math

import numpy as np

from .verify import ERR_NONFINITE, ERR_TOKEN, row_to_float64, verify_chain_sequence

ERR_WINDOW = 32


def verify_pipeline_async_sequence(targets, drafts, windows, us, vs, lengths, temperature, greedy, final_bonus):
    """One sequence.

    targets  list over stages 1 .. k-1 of float64 [w_s + 1, V]: M_s at the
             window's positions and the one after it
    drafts   list of float64 [w_s, V]: M_{s-1} at the window's positions
             (ignored when greedy)
    windows  list of int lists: the tokens O_{s-1}[l_s : l_s + w_s]
    us, vs   per stage: accept uniforms [w_s] and the draw uniform
    lengths  l_0 .. l_{k-1}
    Returns dict(a, t, t_valid over stages; r over buffers 0 .. k-1 (r[k-1]
    is committed); committed, error, margin_u, margin_v, min_mass).
    """
    k = len(lengths)
    out = dict(a=[0] * (k - 1), t=[-1] * (k - 1), t_valid=[0] * (k - 1), r=list(lengths), committed=lengths[-1],
               error=0, margin_u=math.inf, margin_v=math.inf, min_mass=math.inf)
    malformed = any(l < 0 for l in lengths) or any(
        lengths[s - 1] < lengths[s] + len(windows[s - 1]) for s in range(1, k))
    stages = []
    error = ERR_WINDOW if malformed else 0
    for s in range(1, k):  # every stage is verified; its data errors are reported either way
        c = verify_chain_sequence(targets[s - 1], None if greedy else drafts[s - 1], windows[s - 1],
                                  None if greedy else us[s - 1], None if greedy else vs[s - 1], temperature,
                                  greedy)
        error |= c["error"]
        stages.append(c)
    if error & (ERR_TOKEN | ERR_NONFINITE | ERR_WINDOW):
        out["error"] = error
        return out
    new = [lengths[0]]
    cuts = []
    for s, c in enumerate(stages, start=1):
        w, a = len(windows[s - 1]), c["accept_len"]
        # new[s - 1]: the buffer below after its own stage's appends
        bonus = (s == 1 or (final_bonus and s == k - 1)) and new[s - 1] == lengths[s] + w
        emits = a < w or bonus
        out["a"][s - 1] = a
        out["t"][s - 1] = c["out_token"] if emits else -1
        out["t_valid"][s - 1] = int(emits)
        new.append(lengths[s] + a + int(emits))
        if a < w:
            cuts.append((s, lengths[s] + a))
        out["margin_u"] = min(out["margin_u"], c["margin_u"])
        out["min_mass"] = min(out["min_mass"], c["min_mass"])
        if emits:
            out["margin_v"] = min(out["margin_v"], c["margin_v"])
    out["r"] = [min([new[j]] + [P for s, P in cuts if s > j]) for j in range(k)]
    out["committed"] = out["r"][k - 1]
    out["error"] = error
    return out


def verify_pipeline_async(targets, drafts, windows, us, vs, lengths, temperature, greedy, final_bonus, dtype,
                          V=None):
    """Batch wrapper.  targets / drafts: per stage stored logit arrays
    [B, w_s + 1, ld] / [B, w_s, ld] (drafts may be None when greedy);
    windows: per stage int arrays [B, w_s]; us: per stage [B, w_s]; vs: per
    stage [B]; lengths [k, B].  Returns a, t, t_valid [B, k-1], r [B, k-1]
    (buffers 0 .. k-2), committed, error, margin_u, margin_v, min_mass [B]."""
    k = len(targets) + 1
    B = windows[0].shape[0]
    V = targets[0].shape[2] if V is None else V
    res = {n: np.zeros((B, k - 1), np.int64) for n in ("a", "t", "t_valid", "r")}
    res.update(committed=np.zeros(B, np.int64), error=np.zeros(B, np.int64), margin_u=np.zeros(B),
               margin_v=np.zeros(B), min_mass=np.zeros(B))

    def rows(arr, b):
        return np.stack([row_to_float64(arr[b, i, :V], dtype) for i in range(arr.shape[1])])

    for b in range(B):
        r = verify_pipeline_async_sequence(
            [rows(t, b) for t in targets], None if greedy else [rows(d, b) for d in drafts],
            [[int(x) for x in w[b]] for w in windows], None if greedy else [u[b] for u in us],
            None if greedy else [float(v[b]) for v in vs], [int(lengths[j][b]) for j in range(k)], temperature,
            greedy, final_bonus)
        for n in ("a", "t", "t_valid"):
            res[n][b] = r[n]
        res["r"][b] = r["r"][:k - 1]
        for n in ("committed", "error", "margin_u", "margin_v", "min_mass"):
            res[n][b] = r[n]
    return res
