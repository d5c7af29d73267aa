"""The fused LM head and row statistics (spec_verify_chain_lm_head) against
the float64 oracle of oracle/lm_head.py.

The kernel's logits are float32 sums of d bfloat16 products formed on the
tensor cores, so each differs from the exact product by rounding.  The
tests check that in two steps:
  1. the logits the kernel stores (sampling mode keeps them for the draw)
     are within the worst-case error of a d-term float32 sum,
     d * 2^-24 * sum_k |h_k w_k|, of the exact products;
  2. the verification on those logits is the oracle's: the float64 oracle
     run on the kernel's own float32 logits must give the GPU's decisions,
     tokens and error words, with the stored-logit tests' near-tie rules
     (tests/gpu_helpers.py), and the oracle on the exact products must give
     the same wherever the two oracles agree.  Where they differ, the
     rounding of the products itself moved a decision; such sequences are
     set aside, and they must stay rare.
Greedy calls store no logits; their GEMM is the same launch geometry as the
sampling call's, so its logits are the same bits, and the greedy result must
equal the argmax rule on the stored logits exactly.
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


def oracle_on_kernel_logits(w, logits, seqs, greedy):
    """The chain oracle on the kernel's float32 logits (converted exactly)."""
    s = w["spec"]
    tgt = np.ascontiguousarray(logits[0][seqs], np.float32)
    drf = (np.ascontiguousarray(logits[1][seqs], np.float32) if logits[1] is not None
           else np.zeros((len(seqs), 0, s.V), np.float32))
    return V.verify_chain(tgt, drf, w["tokens"][seqs], w["u"][seqs], w["v"][seqs], w["prefix_len"][seqs],
                          s.temperature, greedy, "f32")


DECISIONS = ("accept_len", "out_token", "rollback_idx")


def compare(g, w, logits, seqs, greedy, err):
    s = w["spec"]
    o_exact = oracle(w, seqs, greedy)
    o_kern = oracle_on_kernel_logits(w, logits, seqs, greedy)
    moved = np.zeros(len(seqs), bool)
    for k in DECISIONS:
        moved |= o_exact[k] != o_kern[k]
    assert moved.mean() <= H.MAX_FLAGGED, f"rounding of the products moved {moved.sum()} of {len(seqs)}"
    flagged = H.set_aside(o_kern, greedy) | moved
    assert flagged.mean() <= H.MAX_FLAGGED, f"{flagged.sum()} of {len(seqs)} set aside"
    ok = ~flagged
    for k in DECISIONS:
        bad = np.flatnonzero(ok & (g[k][seqs] != o_kern[k]))
        assert bad.size == 0, (k, seqs[bad[:8]], g[k][seqs][bad[:8]], o_kern[k][bad[:8]])
        assert np.array_equal(o_kern[k][ok], o_exact[k][ok])
    H.compare_errors(g["seq_error"][seqs], o_kern["error"], flagged, V.ERR_TOKEN | V.ERR_NONFINITE)
    if not greedy:
        valid = o_kern["error"] == 0
        for k in ("p_at_draft", "q_at_draft"):
            assert H.close(g[k][seqs][valid], o_kern[k][valid]).all(), k
            # and against the exact products, within what e moves a probability
            a, b = g[k][seqs][valid], o_exact[k][valid]
            assert (np.abs(a - b) <= (H.REL_F + 4 * err / s.temperature) * np.abs(b) + H.ABS_F).all(), k
        same = ok & valid
        assert H.close(g["resid_mass"][seqs][same], o_kern["resid_mass"][same]).all()
    return flagged, moved


CASES = [
    W(BASE, name="v1000_d256_g4", B=3, gamma=4, V=1000, d_target=256, d_draft=256),
    W(BASE, name="v5000_dt200_dd104_g3", B=5, gamma=3, V=5000, d_target=200, d_draft=104),
    W(BASE, name="rows180_v3001_d128", B=30, gamma=5, V=3001, d_target=128, d_draft=128, temperature=1.0),
    W(BASE, name="rows560_two_row_blocks", B=80, gamma=6, V=3000, d_target=128, d_draft=64),
    # 270 / 216 rows: CTA pairs, chunks of 144 / 112 rows partly past the
    # last row, a ragged vocabulary tile and a ragged last K step
    W(BASE, name="pairs_rows270_v5001_d200", B=54, gamma=4, V=5001, d_target=200, d_draft=200),
    W(BASE, name="g0_bonus_only", B=6, gamma=0, V=2000, d_target=64, d_draft=64),
    W(BASE, name="v40000_d1024_T1.3", B=4, gamma=5, V=40000, d_target=1024, d_draft=1024, temperature=1.3),
    # the interface's limits: the largest vocabulary (one partial per CTA and
    # row, one CTA per SM, merged by the walk's warp-per-row form; d = 8 is
    # one K step, mostly zero-filled by the copy engine) and the widest
    # hidden state (1024 K steps per tile)
    W(BASE, name="vmax_2097152_d8", B=2, gamma=1, V=2097152, d_target=8, d_draft=8),
    W(BASE, name="dmax_65536_v1000", B=2, gamma=2, V=1000, d_target=65536, d_draft=65536),
]


def check(w, device, seqs):
    g, logits = run(w, device)
    err, bound = logit_error(w, logits, seqs)
    assert err <= bound, (err, bound)
    compare(g, w, logits, seqs, False, err)
    # greedy on the same inputs: the same GEMM, argmaxes only, no logits stored
    gg, _ = run(w, device, greedy=True)
    _, moved = compare(gg, w, logits, seqs, True, err)
    o_kern = oracle_on_kernel_logits(w, logits, seqs, True)
    for k in DECISIONS:  # argmaxes of the same float32 values: exact
        assert np.array_equal(gg[k][seqs], o_kern[k]), k
    return g


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_lm_head_chain_small(cuda_device, spec):
    w = synth.make(spec, seed=3)
    check(w, cuda_device, np.arange(spec.B))


def test_lm_head_chain_full_size_sampled(cuda_device):
    # the measured workload (B = 64, gamma = 5, V = 128256, d = 4096) in its
    # launch configuration; every output of 8 sampled sequences is checked
    w = synth.make(BASE, seed=0)
    g = check(w, cuda_device, np.array([0, 9, 17, 26, 35, 44, 53, 63]))
    assert (g["seq_error"] == 0).all() and g["error_word"][0] == 0


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


@pytest.mark.parametrize("B", [6, 64], ids=["single_cta", "cta_pairs"])
def test_lm_head_data_errors(cuda_device, B):
    # a drafted token out of range, and NaN hidden states (their logit rows
    # are NaN): those sequences get the data-error bits and empty outputs,
    # the others are unaffected (B = 64: 256 target rows, the CTA-pair kernel)
    spec = W(BASE, B=B, gamma=3, V=3000, d_target=128, d_draft=128)
    w = synth.make(spec, seed=21)
    nan = synth.bf16_from_float32(np.array([np.nan], np.float32))[0]
    w["tokens"][1, 2] = spec.V
    w["h_target"][3, 1, 5] = nan
    w["h_draft"] = w["h_draft"].copy()
    w["h_draft"][4, 0, 7] = nan
    for greedy in (False, True):
        g, _ = run(w, cuda_device, greedy=greedy)
        o = oracle(w, np.arange(spec.B), greedy)
        want = {1: V.ERR_TOKEN, 3: V.ERR_NONFINITE, 4: 0 if greedy else V.ERR_NONFINITE}
        for b, bit in want.items():
            assert g["seq_error"][b] == bit == o["error"][b], (greedy, b, g["seq_error"][b], o["error"][b])
            if bit:
                assert g["accept_len"][b] == 0 and g["out_token"][b] == -1
        ok = np.array([b not in want or want[b] == 0 for b in range(spec.B)])
        flagged = H.set_aside(o, greedy)
        for k in DECISIONS:
            assert np.array_equal(g[k][ok & ~flagged], o[k][ok & ~flagged]), (greedy, k)


@pytest.mark.parametrize("B", [4, 64], ids=["single_cta", "cta_pairs"])
def test_lm_head_wait_gives_up_with_internal_error(cuda_device, B):
    # The head's copy-timeout test hook: every stage of the head kernel
    # expects 16 bytes that never come, so its MMA issuers' bounded waits
    # give up (about 65 ms, then a bounded wait for the stages already
    # issued).  Every row comes out non-finite, so every sequence reports
    # SPEC_ERR_NONFINITE with empty outputs, and the head sets
    # SPEC_ERR_INTERNAL in the error word.  B = 4: 16 target rows, single
    # CTAs; B = 64: 256 rows, CTA pairs (both CTAs of a pair give up, and the
    # even one waits for the odd one's copies before either leaves).
    # Afterwards the same calls, hook off, are correct.
    from draft_verification_gb300 import _lib
    lib = _lib.lib()
    spec = W(BASE, B=B, gamma=3, V=3000 if B == 64 else 5001, d_target=128 if B == 64 else 256,
             d_draft=128 if B == 64 else 256)
    w = synth.make(spec, seed=23)
    for greedy in (False, True):
        assert lib.spec_test_inject_head_copy_timeout(1) == _lib.SPEC_OK
        try:
            g, _ = run(w, cuda_device, greedy=greedy)
        finally:
            assert lib.spec_test_inject_head_copy_timeout(0) == _lib.SPEC_OK
        assert (g["seq_error"] == _lib.ERR_NONFINITE).all(), (greedy, g["seq_error"])
        assert g["error_word"][0] & _lib.ERR_INTERNAL, (greedy, g["error_word"])
        assert (g["accept_len"] == 0).all() and (g["out_token"] == -1).all()
        assert np.array_equal(g["rollback_idx"], w["prefix_len"])
    check(w, cuda_device, np.arange(spec.B))


@pytest.mark.parametrize("B,V,ties", [(2, 40000, [230, 300, 35000, 39999]), (128, 75776, [100, 260, 35000, 39999])],
                         ids=["single_cta", "cta_pairs"])
def test_lm_head_greedy_ties_go_to_the_lowest_index(cuda_device, B, V, ties):
    # Identical weight rows give bit-identical logits (same operands, same
    # accumulation order in every column), so each hidden row's maximum is
    # an exact tie between those vocabulary entries and the greedy argmax
    # must be the lowest of them (the first-index rule of the oracle's
    # argmax).  With V = 40000 and 4 rows the head kernel's tiles are 144
    # entries wide and one CTA of a 152-SM part owns tiles 1 and 2; its first
    # epilogue half sees entry 300 (tile 2) and its second half entry 230
    # (tile 1), so the merge of the two halves must pick 230.  With 256 rows
    # (B = 128) and V = 75776 the CTA-pair kernel runs (on a 152-SM part its
    # 296 tiles balance better over 76 pairs than the single-CTA tiles over
    # 152 CTAs): the even CTA of the first pair holds
    # entries 0-127 (tile 0) and 256-383 (tile 1); its lane quarter 0 sees 260
    # and its quarter 3 sees 100, and the per-row merge of the quarters (in
    # quarter order) must pick 100.
    from draft_verification_gb300 import LmHeadChainPlan
    rng = np.random.default_rng(5)
    g, d = 1, 64
    h = synth.bf16_from_float32((np.abs(rng.normal(size=(B, g + 1, d))) + 0.5).astype(np.float32))
    w = synth.bf16_from_float32((0.01 * rng.normal(size=(V, d))).astype(np.float32))
    w[ties] = synth.bf16_from_float32(np.ones(d, np.float32))
    tokens = np.full((B, g), 7, np.int32)  # never the argmax: the first test rejects
    zeros = np.zeros((B, g), np.float32)
    plan = LmHeadChainPlan(_bf16_dev(h, cuda_device), _bf16_dev(h[:, :g], cuda_device), _bf16_dev(w, cuda_device),
                           _bf16_dev(w, cuda_device), H.dev(tokens, cuda_device), H.dev(zeros, cuda_device),
                           H.dev(np.zeros(B, np.float32), cuda_device), H.dev(np.zeros(B, np.int32), cuda_device),
                           greedy=True)
    out = H.to_np(plan.run())
    assert (out["seq_error"] == 0).all()
    assert (out["accept_len"] == 0).all()
    assert (out["out_token"] == min(ties)).all(), out["out_token"]
