"""The fused LM head and row statistics (spec_verify_chain_lm_head) against
the float64 oracle of oracle/lm_head.py.

The kernel's logits are float32 sums of d bfloat16 products formed on the
tensor cores, so each differs from the exact product by rounding: at most
about d * 2^-24 * sum_k |h_k w_k| (the worst case of a d-term float32 sum),
in practice far less.  The tests measure that error on the logits the kernel
stores (sampling mode keeps them for the draw) and check it against the
worst-case bound; decisions are then compared exactly except where the
measured error could flip them:
  * an accept test with |u - r| below TOL_U + 4 e / T * max(1, r): the
    ratio r = p / q moves by at most 4 e / T in log space (two logits and two
    row sums, each off by at most e);
  * a draw whose v * Z lies within TOL_V + 8 e / (T Z) of a running sum, or
    a residual thinner than 16 e / T (its mass is then mostly rounding);
  * in greedy mode a tested row whose two largest exact logits are closer
    than 4 e.
e is the measured maximum logit error of the call; the same rules as the
stored-logit parity tests otherwise (tests/gpu_helpers.py).
"""

import numpy as np
import pytest
import torch

from oracle import lm_head as LH
from oracle import verify as V
from workloads import synth

from . import gpu_helpers as H

pytestmark = pytest.mark.gpu

BASE = synth.LM_HEAD_SPECS["lm_head_chain_b64_g5_v128256_d4096_bf16"]
W = synth.with_sizes


def _bf16_dev(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def run(w, device, greedy=None):
    from draft_verification_gb300 import LmHeadChainPlan
    s = w["spec"]
    greedy = s.greedy if greedy is None else greedy
    plan = LmHeadChainPlan(_bf16_dev(w["h_target"], device), _bf16_dev(w["h_draft"], device),
                           _bf16_dev(w["w_target"], device), _bf16_dev(w["w_draft"], device),
                           H.dev(w["tokens"], device), H.dev(w["u"], device), H.dev(w["v"], device),
                           H.dev(w["prefix_len"], device), greedy=greedy, temperature=s.temperature)
    out = H.to_np(plan.run())
    logits = None
    if not greedy:
        logits = (plan.target_logits().cpu().numpy().astype(np.float64),
                  plan.draft_logits().cpu().numpy().astype(np.float64) if s.gamma else None)
    return out, logits


def exact(w, seqs):
    ht, hd = LH.bf16_values(w["h_target"][seqs]), LH.bf16_values(w["h_draft"][seqs])
    if "_w64" not in w:  # the heads as float64, converted once per workload
        wt = LH.bf16_values(w["w_target"])
        wd = wt if w["w_draft"] is w["w_target"] else LH.bf16_values(w["w_draft"])
        w["_w64"] = (wt, wd)
    return (ht, hd) + w["_w64"]


def logit_error(w, logits, seqs):
    """Measured max |gpu - exact| over the sampled sequences' rows, and the
    worst-case float32 bound of a d-term sum of those rows."""
    ht, hd, wt, wd = exact(w, seqs)
    err, bound = 0.0, 0.0
    for x, wmat, g in ((ht, wt, logits[0]), (hd, wd, logits[1])):
        if g is None:
            continue
        wabs = np.abs(wmat)
        for i, b in enumerate(seqs):
            ex = x[i] @ wmat.T
            err = max(err, float(np.abs(g[b] - ex).max()))
            d = x.shape[2]
            bound = max(bound, d * 2.0 ** -24 * float((np.abs(x[i]) @ wabs.T).max()))
    return err, bound


def oracle(w, seqs, greedy):
    s = w["spec"]
    ht, hd, wt, wd = exact(w, seqs)
    return LH.verify_chain_from_hidden(ht, hd, wt, wd, w["tokens"][seqs], w["u"][seqs], w["v"][seqs],
                                       w["prefix_len"][seqs], s.temperature, greedy)


def compare_sampling(g, o, seqs, err, T):
    r = np.where(o["q_at_draft"] > 0, o["p_at_draft"] / np.maximum(o["q_at_draft"], 1e-300), np.inf)
    rmax = np.maximum(1.0, np.nan_to_num(r, posinf=1e30).max(axis=1)) if r.shape[1] else np.ones(len(seqs))
    Z = np.where(o["resid_mass"] > 0, o["resid_mass"], 1.0)
    flagged = ((o["margin_u"] < H.TOL_U + 4 * err / T * rmax)
               | (o["margin_v"] < H.TOL_V + 8 * err / (T * Z))
               | ((o["min_mass"] > 0) & (o["min_mass"] < max(H.Z_MIN, 16 * err / T))))
    assert flagged.mean() <= H.MAX_FLAGGED, f"{flagged.sum()} of {len(seqs)} set aside (e = {err:.3g})"
    ok = ~flagged
    for k in ("accept_len", "out_token", "rollback_idx"):
        bad = np.flatnonzero(ok & (g[k][seqs] != o[k]))
        assert bad.size == 0, (k, seqs[bad[:8]], g[k][seqs][bad[:8]], o[k][bad[:8]])
    H.compare_errors(g["seq_error"][seqs], o["error"], flagged, V.ERR_TOKEN | V.ERR_NONFINITE)
    tol = H.REL_F + 4 * err / T
    valid = o["error"] == 0
    for k in ("p_at_draft", "q_at_draft"):
        a, b = g[k][seqs][valid], o[k][valid]
        assert (np.abs(a - b) <= tol * np.abs(b) + H.ABS_F).all(), k
    same = ok & valid & (g["accept_len"][seqs] == o["accept_len"])
    a, b = g["resid_mass"][seqs][same], o["resid_mass"][same]
    # each weight p or q is off by at most 2 e / T relative, so a mass built
    # from at most two unit-mass distributions by at most 4 e / T absolute
    assert (np.abs(a - b) <= H.REL_F * np.abs(b) + 4 * err / T + H.ABS_F).all()
    return flagged


def compare_greedy(g, o, w, seqs, err):
    ht, _, wt, _ = exact(w, seqs)
    flagged = np.zeros(len(seqs), bool)
    for i in range(len(seqs)):
        a = int(o["accept_len"][i])
        ex = ht[i][: a + 1] @ wt.T
        top2 = np.sort(ex, axis=1)[:, -2:]
        flagged[i] = (top2[:, 1] - top2[:, 0] < 4 * err).any()
    ok = ~flagged
    for k in ("accept_len", "out_token", "rollback_idx"):
        bad = np.flatnonzero(ok & (g[k][seqs] != o[k]))
        assert bad.size == 0, (k, seqs[bad[:8]], g[k][seqs][bad[:8]], o[k][bad[:8]])
    assert (g["seq_error"][seqs] == 0).all()


CASES = [
    W(BASE, name="v1000_d256_g4", B=3, gamma=4, V=1000, d_target=256, d_draft=256),
    W(BASE, name="v5000_dt200_dd104_g3", B=5, gamma=3, V=5000, d_target=200, d_draft=104),
    W(BASE, name="rows180_v3001_d128", B=30, gamma=5, V=3001, d_target=128, d_draft=128, temperature=1.0),
    W(BASE, name="rows560_two_row_blocks", B=80, gamma=6, V=3000, d_target=128, d_draft=64),
    W(BASE, name="g0_bonus_only", B=6, gamma=0, V=2000, d_target=64, d_draft=64),
    W(BASE, name="v40000_d1024_T1.3", B=4, gamma=5, V=40000, d_target=1024, d_draft=1024, temperature=1.3),
]


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_lm_head_chain_small(cuda_device, spec):
    w = synth.make(spec, seed=3)
    g, logits = run(w, cuda_device)
    seqs = np.arange(spec.B)
    err, bound = logit_error(w, logits, seqs)
    assert err <= bound, (err, bound)
    compare_sampling(g, oracle(w, seqs, False), seqs, err, spec.temperature)
    # greedy on the same inputs: the same GEMM, argmaxes only, no logits stored
    gg, _ = run(w, cuda_device, greedy=True)
    compare_greedy(gg, oracle(w, seqs, True), w, seqs, err)


def test_lm_head_chain_full_size_sampled(cuda_device):
    # the measured workload (B = 64, gamma = 5, V = 128256, d = 4096) in its
    # launch configuration; every output of 8 sampled sequences is checked
    w = synth.make(BASE, seed=0)
    g, logits = run(w, cuda_device)
    seqs = np.array([0, 9, 17, 26, 35, 44, 53, 63])
    err, bound = logit_error(w, logits, seqs)
    assert err <= bound, (err, bound)
    flagged = compare_sampling(g, oracle(w, seqs, False), seqs, err, BASE.temperature)
    assert not flagged.all()
    assert (g["seq_error"] == 0).all() and g["error_word"][0] == 0
    gg, _ = run(w, cuda_device, greedy=True)
    compare_greedy(gg, oracle(w, seqs, True), w, seqs, err)


def test_lm_head_matches_stored_logit_path(cuda_device):
    # the fused path's decisions equal spec_verify_chain's on the logits the
    # head kernel stored (float32 rows): same walk, same statistics up to the
    # order of the row sums, so outputs agree except at near ties
    spec = W(BASE, B=6, gamma=4, V=9000, d_target=512, d_draft=512)
    w = synth.make(spec, seed=8)
    g, logits = run(w, cuda_device)
    tw = dict(kind="chain", spec=synth.with_sizes(synth.SPECS["sampling_chain_b32_g8_v32000_bf16"], B=spec.B,
                                                  gamma=spec.gamma, V=spec.V, dtype="f32",
                                                  temperature=spec.temperature),
              target=logits[0].astype(np.float32), draft=logits[1].astype(np.float32), tokens=w["tokens"],
              u=w["u"], v=w["v"], prefix_len=w["prefix_len"])
    gc = H.gpu_chain(tw, cuda_device)
    oc = H.oracle_chain(tw)
    flagged = H.set_aside(oc, False)
    for k in ("accept_len", "out_token", "rollback_idx"):
        assert np.array_equal(g[k][~flagged], gc[k][~flagged]), k
