"""Run the CUDA path and the CPU oracle on the same seeded workload and
compare them.

Parity rules (the tolerances are written here and used by every GPU test):
  * integer outputs (accept lengths, tokens, paths, rollback indices, error
    bits) must be identical, except for sequences with a decision the oracle
    reports as a near tie;
  * a near tie is an accept test with |u - p/q| < TOL_U, or an inverse-CDF
    draw whose target v*Z lies within TOL_V * Z of one of the two running
    sums that bracket the drawn index.  The float32 kernels compute p/q and
    the running sums with relative errors of a few 1e-7, so decisions inside
    these bands may legitimately go either way;
  * a residual distribution max(0, p - q) formed after a rejection whose
    float64 mass is positive but below Z_MIN is also set aside: float32
    weights carry a relative error of up to about 1e-6 that is common to a
    whole row (its rounded 1/s), so a residual of two nearly equal
    distributions is known only to about 1e-6 in absolute terms; below Z_MIN
    neither the zero-mass fallback (reading R3) nor the draw from the
    residual is decided by the inputs alone.  An exactly zero mass (R3
    proper) is not set aside: both sides must take the fallback;
  * error words are compared whole (the zero-mass bit 8 included) on every
    sequence not set aside; on every sequence the data-error bits must agree,
    and no sequence may carry bit 16 (a bounded wait that gave up);
  * float outputs (p(d), q(d), residual mass) within REL_F of the float64
    oracle, or within ABS_F in absolute terms for values below 1e-30
    (float32 flushes subnormal probabilities to zero).
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import verify as V

TOL_U = 1e-6
TOL_V = 1e-6
REL_F = 1e-5
ABS_F = 1e-30
MAX_FLAGGED = 0.25  # a parity run that sets aside more than this is not a test
Z_MIN = 1e-3
ERR_INTERNAL = 16


def set_aside(o, greedy):
    """Sequences whose outputs a faithful float32 implementation may take
    either way: near ties of an accept test or a draw, and residuals whose
    mass is positive but below Z_MIN (greedy decisions are exact)."""
    B = len(o["error"])
    if greedy:
        return np.zeros(B, bool)
    thin = (o["min_mass"] > 0.0) & (o["min_mass"] < Z_MIN)
    return (o["margin_u"] < TOL_U) | (o["margin_v"] < TOL_V) | thin


def compare_errors(g_err, o_err, flagged, hard):
    """Error words: the data-error bits `hard` on every sequence, the whole
    word on every sequence not set aside, and never bit 16."""
    g_err = np.asarray(g_err, np.int64)
    o_err = np.asarray(o_err, np.int64)
    assert not (g_err & ERR_INTERNAL).any(), f"a bounded wait gave up: {np.flatnonzero(g_err & ERR_INTERNAL)}"
    assert np.array_equal(g_err & hard, o_err & hard), (g_err, o_err)
    keep = ~flagged
    bad = np.flatnonzero(keep & (g_err != o_err))
    assert bad.size == 0, f"error words differ at {bad[:8]}: gpu {g_err[bad[:8]]} oracle {o_err[bad[:8]]}"


def dev_logits(arr: np.ndarray, dtype: str, device) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(arr, np.float32)).to(device)


def dev(arr, device, dt=None):
    t = torch.from_numpy(np.ascontiguousarray(arr))
    if dt is not None:
        t = t.to(dt)
    return t.to(device)


def to_np(out: dict) -> dict:
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def logits_view(t: torch.Tensor, V: int) -> torch.Tensor:
    return t[..., :V]


# --------------------------------------------------------------------------
# chain
# --------------------------------------------------------------------------

def chain_plan(w, device, greedy=None, workspace=None, consulted_only=False):
    from draft_verification_gb300 import ChainPlan
    s = w["spec"]
    greedy = s.greedy if greedy is None else greedy
    tgt = logits_view(dev_logits(w["target"], s.dtype, device), s.V)
    drf = logits_view(dev_logits(w["draft"], s.dtype, device), s.V)
    return ChainPlan(tgt, drf, dev(w["tokens"], device), dev(w["u"], device), dev(w["v"], device),
                     dev(w["prefix_len"], device), greedy=greedy, temperature=s.temperature,
                     workspace=workspace, consulted_only=consulted_only)


def gpu_chain(w, device, greedy=None, workspace=None, consulted_only=False):
    return to_np(chain_plan(w, device, greedy, workspace, consulted_only).run())


def oracle_chain(w, greedy=None):
    s = w["spec"]
    greedy = s.greedy if greedy is None else greedy
    return V.verify_chain(w["target"], w["draft"], w["tokens"], w["u"], w["v"], w["prefix_len"],
                          s.temperature, greedy, s.dtype, V=s.V)


def close(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    ok = np.abs(a - b) <= REL_F * np.abs(b)
    ok |= (np.abs(b) < 1e-30) & (np.abs(a) <= ABS_F)
    return ok


def compare_chain(g, o, greedy):
    B = len(o["accept_len"])
    flagged = set_aside(o, greedy)
    ok = ~flagged
    assert flagged.mean() <= MAX_FLAGGED, f"{flagged.sum()} of {B} sequences set aside"
    bad = np.flatnonzero(ok & ((g["accept_len"] != o["accept_len"]) | (g["out_token"] != o["out_token"])
                               | (g["rollback_idx"] != o["rollback_idx"])))
    assert bad.size == 0, (
        f"mismatch at {bad[:8]}: gpu a={g['accept_len'][bad[:8]]} t={g['out_token'][bad[:8]]}, "
        f"oracle a={o['accept_len'][bad[:8]]} t={o['out_token'][bad[:8]]} "
        f"margins u={o['margin_u'][bad[:8]]} v={o['margin_v'][bad[:8]]}")
    compare_errors(g["seq_error"], o["error"], flagged, V.ERR_TOKEN | V.ERR_NONFINITE)
    if not greedy:
        valid = (o["error"] & (V.ERR_TOKEN | V.ERR_NONFINITE)) == 0
        assert close(g["p_at_draft"][valid], o["p_at_draft"][valid]).all()
        assert close(g["q_at_draft"][valid], o["q_at_draft"][valid]).all()
        same = ok & valid & (g["accept_len"] == o["accept_len"])
        assert close(g["resid_mass"][same], o["resid_mass"][same]).all(), (
            g["resid_mass"][same], o["resid_mass"][same])
    return flagged


# --------------------------------------------------------------------------
# tree
# --------------------------------------------------------------------------

def gpu_tree(w, device, greedy=None, workspace=None, consulted_only=False):
    from draft_verification_gb300 import TreePlan
    s = w["spec"]
    greedy = s.greedy if greedy is None else greedy
    tgt = logits_view(dev_logits(w["target"], s.dtype, device), s.V)
    drf = logits_view(dev_logits(w["draft"], s.dtype, device), s.V)
    plan = TreePlan(dev(w["parent"], device), dev(w["tokens"], device), tgt, drf,
                    dev(w["u"], device), dev(w["v"], device), dev(w["prefix_len"], device),
                    max_depth=w["max_depth"], greedy=greedy, temperature=s.temperature,
                    workspace=workspace, consulted_only=consulted_only)
    return to_np(plan.run())


def oracle_tree(w, greedy=None):
    s = w["spec"]
    greedy = s.greedy if greedy is None else greedy
    return V.verify_tree(w["parent"], w["tokens"], w["target"], w["draft"], w["u"], w["v"],
                         w["prefix_len"], s.temperature, greedy, w["max_depth"], s.dtype, V=s.V)


def compare_tree(g, o, greedy):
    B = len(o["path_len"])
    flagged = set_aside(o, greedy)
    ok = ~flagged
    assert flagged.mean() <= MAX_FLAGGED, f"{flagged.sum()} of {B} sequences set aside"
    bad = np.flatnonzero(ok & ((g["path_len"] != o["path_len"]) | (g["out_token"] != o["out_token"])
                               | (g["rollback_idx"] != o["rollback_idx"])
                               | (g["path_nodes"] != o["path_nodes"]).any(axis=1)))
    assert bad.size == 0, (f"mismatch at {bad[:8]}: gpu {g['path_nodes'][bad[:4]]} {g['out_token'][bad[:4]]}"
                           f" oracle {o['path_nodes'][bad[:4]]} {o['out_token'][bad[:4]]}")
    compare_errors(g["seq_error"], o["error"], flagged, V.ERR_TOKEN | V.ERR_PARENT | V.ERR_NONFINITE)
    return flagged


# --------------------------------------------------------------------------
# cascade
# --------------------------------------------------------------------------

CASCADE_KEYS = ("a1", "t1", "a2", "w2", "t2", "t2_valid", "r0", "r1", "committed")


def gpu_cascade(w, device, greedy=None):
    from draft_verification_gb300 import CascadePlan
    s = w["spec"]
    greedy = s.greedy if greedy is None else greedy
    l0 = logits_view(dev_logits(w["l0"], s.dtype, device), s.V)
    l1 = logits_view(dev_logits(w["l1"], s.dtype, device), s.V)
    l2 = logits_view(dev_logits(w["l2"], s.dtype, device), s.V)
    plan = CascadePlan(l0, l1, l2, dev(w["tokens"], device), dev(w["u1"], device),
                       dev(w["v1"], device), dev(w["u2"], device), dev(w["v2"], device),
                       dev(w["base0"], device), dev(w["base1"], device), greedy=greedy,
                       temperature=s.temperature)
    return to_np(plan.run())


def oracle_cascade(w, greedy=None):
    s = w["spec"]
    greedy = s.greedy if greedy is None else greedy
    return V.verify_cascade(w["l0"], w["l1"], w["l2"], w["tokens"], w["u1"], w["v1"], w["u2"],
                            w["v2"], w["base0"], w["base1"], s.temperature, greedy, s.dtype, V=s.V)


def compare_cascade(g, o, greedy):
    B = len(o["a1"])
    flagged = set_aside(o, greedy)
    ok = ~flagged
    assert flagged.mean() <= MAX_FLAGGED, f"{flagged.sum()} of {B} sequences set aside"
    for k in CASCADE_KEYS:
        bad = np.flatnonzero(ok & (g[k] != o[k]))
        assert bad.size == 0, f"{k} mismatch at {bad[:8]}: gpu {g[k][bad[:8]]} oracle {o[k][bad[:8]]}"
    compare_errors(g["seq_error"], o["error"], flagged, V.ERR_TOKEN | V.ERR_NONFINITE)
    return flagged
