"""CLaSp layer selection on the GPU against the oracle.

Two checks per case:
  * sequences whose oracle decisions on the backtracked path are all further
    than TOL_COS from a tie must give the oracle's skip mask exactly and its
    score D(L, M) within TOL_SCORE;
  * every sequence's full decision table must be valid: replaying the DP in
    float64 along the GPU's own decisions, each decision whose two cosines
    differ by more than TOL_COS is the larger-cosine one (the tie rule: keep),
    states outside the reachable band are marked 255, the mask is the
    backtracking of the table from (L, M), and the score is the replayed
    cosine of g(L, M).  Near-ties may go either way; they are counted.

Tolerances: the kernels keep states in float32, form the product from a
two-term bfloat16 split (about 16 significant bits of the input) with float32
accumulation and sum the cosines' dot products in float32; a float32
emulation of that arithmetic stays within 1e-7 of the float64 cosines over 32
layers of width 4096, and float32 sums of 4096 products add about 1e-6.
TOL_COS = 2e-5 leaves an order of magnitude over that; TOL_SCORE = 1e-5.
"""

import numpy as np
import pytest
import torch

from oracle import clasp as K
from workloads import synth

from . import gpu_helpers as H

pytestmark = pytest.mark.gpu

TOL_COS = 2e-5
TOL_SCORE = 1e-5
BASE = synth.CLASP_SPECS["clasp_b16_l32_d4096_m12_bf16"]


def gpu_clasp(w, device, choices=True):
    from draft_verification_gb300 import ClaspPlan
    hidden = torch.from_numpy(w["hidden"]).to(device)
    weights = torch.from_numpy(w["weights"].view(np.int16)).to(device).view(torch.bfloat16)
    plan = ClaspPlan(hidden, weights, w["spec"].M, choices=choices)
    out = plan.run()
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def band(i, L, M):
    return max(0, M - (L - i)), min(i, M)


def validate(h, Ws, M, choice, mask, score):
    """The checks of the second bullet above for one sequence; returns the
    number of near-tie decisions."""
    L = len(Ws)
    g = {(0, 0): h[0]}
    near = 0
    for i in range(1, L + 1):
        W = np.asarray(Ws[i - 1], np.float64)
        lo, hi = band(i, L, M)
        row = choice[i - 1]
        assert (row[:lo] == 255).all() and (row[hi + 1:] == 255).all(), (i, row)
        for j in range(lo, hi + 1):
            c = int(row[j])
            assert c in (0, 1), (i, j, c)
            ck = cs = None
            if j <= i - 1:
                k = K.layer(W, g[(i - 1, j)])
                ck = K.cosine(h[i], k)
            if j >= 1:
                s = g[(i - 1, j - 1)]
                cs = K.cosine(h[i], s)
            if ck is None:
                assert c == 1, (i, j)
            elif cs is None:
                assert c == 0, (i, j)
            elif abs(cs - ck) > TOL_COS:
                assert c == int(cs > ck), (i, j, cs, ck)
            else:
                near += 1
            g[(i, j)] = s if c else k
    j, want = M, np.zeros(L, np.int64)
    for i in range(L, 0, -1):
        want[i - 1] = choice[i - 1, j]
        j -= want[i - 1]
    assert j == 0
    assert np.array_equal(mask, want)
    assert abs(float(score) - K.cosine(h[L], g[(L, M)])) <= TOL_SCORE
    return near


def check(w, g, sequences=None):
    s = w["spec"]
    Wv = synth.clasp_weight_values(w)
    seqs = range(s.B) if sequences is None else sequences
    flagged = 0
    for b in seqs:
        h = w["hidden"][b].astype(np.float64)
        mask, score, margin = K.clasp_dp(h, Wv, s.M)
        validate(h, Wv, s.M, g["choice"][b], g["skip_mask"][b], g["score"][b])
        if margin < TOL_COS:
            flagged += 1
            continue
        assert np.array_equal(g["skip_mask"][b], mask), (b, g["skip_mask"][b], mask)
        assert abs(float(g["score"][b]) - score) <= TOL_SCORE, (b, g["score"][b], score)
        assert int(g["skip_mask"][b].sum()) == s.M
    assert flagged <= H.MAX_FLAGGED * len(seqs), f"{flagged} of {len(seqs)} sequences set aside"


CASES = [
    synth.with_sizes(BASE, name="b6_l8_d64_m3", B=6, L=8, d=64, M=3),
    synth.with_sizes(BASE, name="b5_l12_d256_m5", B=5, L=12, d=256, M=5),
    synth.with_sizes(BASE, name="b4_l10_d520_m4_ragged", B=4, L=10, d=520, M=4),
    synth.with_sizes(BASE, name="b4_l9_d1032_m0_keep_all", B=4, L=9, d=1032, M=0),
    synth.with_sizes(BASE, name="b3_l5_d9000_m2_beyond_registers", B=3, L=5, d=9000, M=2),
    synth.with_sizes(BASE, name="b4_l7_d136_m7_skip_all", B=4, L=7, d=136, M=7),
    synth.with_sizes(BASE, name="b3_l1_d8_m0", B=3, L=1, d=8, M=0),
    synth.with_sizes(BASE, name="b3_l1_d8_m1", B=3, L=1, d=8, M=1),
    synth.with_sizes(BASE, name="b130_l6_d32_m2_two_blocks", B=130, L=6, d=32, M=2),
    synth.with_sizes(BASE, name="b4_l6_d272_m2", B=4, L=6, d=272, M=2),
    synth.with_sizes(BASE, name="b8_l16_d1024_m6_scale05", B=8, L=16, d=1024, M=6, scale=0.5, tau=0.2),
]


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_clasp_small(cuda_device, spec):
    w = synth.make(spec, seed=3)
    check(w, gpu_clasp(w, cuda_device))


def test_clasp_extremes_have_closed_forms(cuda_device):
    # M = L skips every layer: score cos(h_L, h_0); M = 0 keeps every layer
    for M in (0, 6):
        spec = synth.with_sizes(BASE, B=4, L=6, d=128, M=M)
        w = synth.make(spec, seed=8)
        g = gpu_clasp(w, cuda_device)
        assert (g["skip_mask"] == (1 if M else 0)).all()
        if M:
            for b in range(spec.B):
                h = w["hidden"][b].astype(np.float64)
                assert abs(float(g["score"][b]) - K.cosine(h[-1], h[0])) <= TOL_SCORE


def test_clasp_full_size(cuda_device):
    # the whole batch on the GPU; the oracle on a sample of its sequences
    w = synth.make(BASE, seed=0)
    g = gpu_clasp(w, cuda_device)
    check(w, g, sequences=[0, 3, 7, 10, 15])


def test_clasp_is_deterministic_and_choice_is_optional(cuda_device):
    spec = synth.with_sizes(BASE, B=6, L=12, d=512, M=5)
    w = synth.make(spec, seed=4)
    a = gpu_clasp(w, cuda_device)
    b = gpu_clasp(w, cuda_device)
    c = gpu_clasp(w, cuda_device, choices=False)
    for k in ("skip_mask", "score"):
        assert a[k].tobytes() == b[k].tobytes() == c[k].tobytes(), k
    assert a["choice"].tobytes() == b["choice"].tobytes()
    assert "choice" not in c


def test_clasp_graph_replays(cuda_device):
    # one call captured in a CUDA graph (cuBLAS products included) and
    # replayed on new hidden states copied into the same buffer
    from draft_verification_gb300 import ClaspPlan
    spec = synth.with_sizes(BASE, B=5, L=10, d=512, M=4)
    ws = [synth.make(spec, seed=30 + i) for i in range(3)]
    w0 = ws[0]
    hidden = torch.from_numpy(w0["hidden"]).to(cuda_device)
    weights = torch.from_numpy(w0["weights"].view(np.int16)).to(cuda_device).view(torch.bfloat16)
    plan = ClaspPlan(hidden, weights, spec.M, choices=True)
    stream = torch.cuda.Stream(cuda_device)
    plan.run(stream)  # the first call on the device creates the cuBLAS handle: outside the capture
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        plan.run(stream)
    for w in ws[1:] + ws[:1]:
        w = dict(w, weights=w0["weights"])  # the weights stay bound; only the hidden states change
        hidden.copy_(torch.from_numpy(w["hidden"]).to(cuda_device))
        graph.replay()
        torch.cuda.synchronize()
        check(w, {k: v.cpu().numpy() for k, v in plan.out.items()})
