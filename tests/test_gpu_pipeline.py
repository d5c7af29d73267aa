"""k-model pipeline on the GPU against the oracle, sequence by sequence.

Sequences whose accept or draw uniform lies within the oracle's tolerance of
a decision boundary are set aside (as for the other sampling paths); every
other output must match exactly.  k = 3 without the bonus is also checked
against the three-model cascade entry point, bit for bit.
"""

import numpy as np
import pytest

from oracle import pipeline as Pp
from oracle import verify as V
from workloads import synth

from . import gpu_helpers as H

pytestmark = pytest.mark.gpu

BASE = synth.PIPELINE_SPECS["pipeline4_b128_g8_g6_g4_v128256_bf16"]
KEYS = ("a", "w", "t", "t_valid", "r", "committed")


def gpu_pipeline(w, device, greedy=None):
    from draft_verification_gb300 import PipelinePlan
    s = w["spec"]
    greedy = s.greedy if greedy is None else greedy
    models = [None if (greedy and i == 0) else H.logits_view(H.dev_logits(m, s.dtype, device), s.V)
              for i, m in enumerate(w["models"])]
    plan = PipelinePlan(models, H.dev(w["tokens"], device), s.windows,
                        [H.dev(u, device) for u in w["us"]], [H.dev(v, device) for v in w["vs"]],
                        H.dev(w["base"], device), greedy=greedy, temperature=s.temperature,
                        final_bonus=s.final_bonus)
    return H.to_np(plan.run())


def oracle_pipeline(w, greedy=None):
    s = w["spec"]
    greedy = s.greedy if greedy is None else greedy
    return Pp.verify_pipeline(w["models"], w["tokens"], w["us"], w["vs"], s.temperature, greedy, s.final_bonus,
                              s.dtype, V=s.V, base=w["base"])


def compare(g, o, greedy):
    B = len(o["committed"])
    flagged = H.set_aside(o, greedy)
    ok = ~flagged
    assert flagged.mean() <= H.MAX_FLAGGED, f"{flagged.sum()} of {B} sequences set aside"
    for k in KEYS:
        gk, ok_k = g[k], o[k]
        diff = (gk != ok_k) if gk.ndim == 1 else (gk != ok_k).any(axis=1)
        bad = np.flatnonzero(ok & diff)
        assert bad.size == 0, f"{k} mismatch at {bad[:8]}: gpu {gk[bad[:4]]} oracle {ok_k[bad[:4]]}"
    H.compare_errors(g["seq_error"], o["error"], flagged, V.ERR_TOKEN | V.ERR_NONFINITE)


CASES = [
    synth.with_sizes(BASE, name="k2_v9001", B=10, windows=(5,), V=9001, a=(0.9,), s=(0.6,)),
    synth.with_sizes(BASE, name="k3_v12000_pad3", B=10, windows=(6, 4), V=12000, a=(0.9, 0.9), s=(0.5, 1.0), pad=3),
    synth.with_sizes(BASE, name="k4_v20000", B=12, V=20000),
    synth.with_sizes(BASE, name="k4_bonus_v20000", B=12, V=20000, final_bonus=True),
    synth.with_sizes(BASE, name="k5_bonus_v7000", B=12, windows=(8, 6, 4, 3), V=7000, a=(0.9,) * 4,
                     s=(0.465, 1.0, 1.0, 1.0), final_bonus=True),
    synth.with_sizes(BASE, name="k8_v3000", B=8, windows=(6, 5, 5, 4, 4, 3, 3), V=3000, a=(0.95,) * 7,
                     s=(0.4,) * 7),
    synth.with_sizes(BASE, name="k4_f32_v4001", B=8, V=4001, dtype="f32"),
    synth.with_sizes(BASE, name="k4_greedy_v16000", B=10, V=16000, greedy=True, final_bonus=True),
    synth.with_sizes(BASE, name="k6_greedy_v5000", B=10, windows=(8, 7, 6, 5, 4), V=5000, a=(0.95,) * 5,
                     s=(0.3,) * 5, greedy=True),
]


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_pipeline_small(cuda_device, spec):
    w = synth.make(spec, seed=7)
    compare(gpu_pipeline(w, cuda_device), oracle_pipeline(w), spec.greedy)


def test_pipeline_full_size(cuda_device):
    w = synth.make(BASE, seed=0)
    compare(gpu_pipeline(w, cuda_device), oracle_pipeline(w), False)
    compare(gpu_pipeline(w, cuda_device, greedy=True), oracle_pipeline(w, greedy=True), True)


@pytest.mark.parametrize("greedy", [False, True])
def test_k3_equals_the_cascade_entry(cuda_device, greedy):
    spec = synth.with_sizes(synth.SPECS["cascade_b128_g8_g4_v128256_bf16"], B=16, V=11000, greedy=greedy)
    cw = synth.make(spec, seed=12)
    gc = H.gpu_cascade(cw, cuda_device)
    pspec = synth.with_sizes(BASE, B=16, windows=(spec.gamma1, spec.gamma2), V=spec.V, greedy=greedy)
    pw = dict(kind="pipeline", spec=pspec, models=[cw["l0"], cw["l1"], cw["l2"]], tokens=cw["tokens"],
              us=[cw["u1"], cw["u2"]], vs=[cw["v1"], cw["v2"]], base=np.stack([cw["base0"], cw["base1"]]))
    gp = gpu_pipeline(pw, cuda_device)
    assert np.array_equal(gp["a"], np.stack([gc["a1"], gc["a2"]], 1))
    assert np.array_equal(gp["t"][:, 0], gc["t1"])
    assert np.array_equal(gp["t"][:, 1], gc["t2"])
    assert np.array_equal(gp["t_valid"][:, 1], gc["t2_valid"])
    assert np.array_equal(gp["w"][:, 1], gc["w2"])
    assert np.array_equal(gp["r"], np.stack([gc["r0"], gc["r1"]], 1))
    assert np.array_equal(gp["committed"], gc["committed"])


def test_pipeline_data_errors(cuda_device):
    spec = synth.with_sizes(BASE, B=5, V=3000)
    w = synth.make(spec, seed=9)
    w["tokens"][1, 2] = spec.V
    nan = synth.bf16_from_float32(np.array([np.nan], np.float32))[0]
    w["models"][2][3, 1, 5] = nan
    for greedy in (False, True):
        g = gpu_pipeline(w, cuda_device, greedy=greedy)
        o = oracle_pipeline(w, greedy=greedy)
        compare(g, o, greedy)
        assert g["seq_error"][1] & 1 and g["seq_error"][3] & 4
        assert (g["r"][1] == w["base"][:, 1]).all() and g["committed"][1] == 0
