"""The seeded input generators (no GPU)."""

import json
import os

import numpy as np
import pytest
import torch

from oracle.verify import acceptance_rate, row_to_float64
from workloads import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 3, 100000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, -2.5e-39], np.float32)])
    ours = synth.bf16_from_float32(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(synth.float32_from_bf16(ours),
                          torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_specs_match_recorded_calibration():
    with open(os.path.join(GOLDEN, "calibration.json")) as fh:
        cal = json.load(fh)
    for name, rec in cal.items():
        spec = synth.SPECS[name]
        for k in ("a", "s", "a01", "s01", "a12", "s12"):
            if k in rec:
                assert getattr(spec, k) == pytest.approx(rec[k], abs=1e-12), (name, k)
        for k in ("alpha", "alpha01", "alpha12"):
            if k in rec:
                tgt = {"alpha": "alpha_target", "alpha01": "alpha01_target",
                       "alpha12": "alpha12_target"}[k]
                assert abs(rec[k] - getattr(spec, tgt)) < 0.01, (name, k)


def test_deterministic_and_in_range():
    for name, spec in synth.SPECS.items():
        small = synth.with_sizes(spec, B=2, V=min(spec.V, 3001))
        a, b = synth.make(small, seed=3), synth.make(small, seed=3)
        for k in a:
            if isinstance(a[k], np.ndarray):
                assert np.array_equal(a[k], b[k]), (name, k)
        toks = a["tokens"] if a["kind"] != "tree" else a["tokens"][:, 1:]
        assert toks.min() >= 0 and toks.max() < small.V


@pytest.mark.parametrize("name", ["sampling_chain_b32_g8_v32000_bf16",
                                  "sampling_chain_b64_g5_v128256_bf16_a60"])
def test_alpha_near_target_on_fresh_seed(name):
    spec = synth.SPECS[name]
    w = synth.make(synth.with_sizes(spec, B=1), seed=11)
    al = [acceptance_rate(row_to_float64(w["target"][0, i], spec.dtype),
                          row_to_float64(w["draft"][0, i], spec.dtype), spec.temperature)
          for i in range(spec.gamma)]
    assert abs(np.mean(al) - spec.alpha_target) < 0.05


def test_tree_topology_reading():
    parent = synth.tree_topology()
    assert len(parent) == 64 and parent[0] == -1
    assert all(0 <= parent[i] < i for i in range(1, 64))
    depth = np.zeros(64, int)
    for i in range(1, 64):
        depth[i] = depth[parent[i]] + 1
    assert list(np.bincount(depth)) == [1, 4, 9, 11, 13, 13, 13]
    assert int((np.bincount(parent[1:], minlength=64) == 0).sum()) == 18


def test_clasp_workload_is_seeded_and_shaped():
    spec = synth.with_sizes(synth.CLASP_SPECS["clasp_b16_l32_d4096_m12_bf16"], B=3, L=5, d=64, M=2)
    a, b, c = synth.make(spec, seed=1), synth.make(spec, seed=1), synth.make(spec, seed=2)
    assert a["weights"].shape == (5, 64, 64) and a["weights"].dtype == np.uint16
    assert a["hidden"].shape == (3, 6, 64) and a["hidden"].dtype == np.float32
    assert np.array_equal(a["weights"], b["weights"]) and np.array_equal(a["hidden"], b["hidden"])
    assert not np.array_equal(a["hidden"], c["hidden"])
    assert np.isfinite(a["hidden"]).all()
    # weights are bf16 values of N(0, scale^2 / d): sample sd near scale / sqrt(d)
    wv = synth.clasp_weight_values(a)
    assert abs(wv.std() * np.sqrt(64) / spec.scale - 1) < 0.05
