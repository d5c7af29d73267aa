"""Consulted-only chain verification on the GPU against the oracle."""

import numpy as np
import pytest

from oracle import consulted as Cn
from oracle import verify as V
from workloads import synth

from . import gpu_helpers as H

pytestmark = pytest.mark.gpu

S = synth.SPECS


def oracle(w):
    s = w["spec"]
    return Cn.verify_chain_consulted(w["target"], w["draft"], w["tokens"], w["u"], w["v"], w["prefix_len"],
                                     s.temperature, s.dtype, V=s.V)


def compare(g, o):
    B = len(o["accept_len"])
    flagged = H.set_aside(o, False)
    ok = ~flagged
    assert flagged.mean() <= H.MAX_FLAGGED
    for k in ("accept_len", "out_token", "rollback_idx"):
        bad = np.flatnonzero(ok & (g[k] != o[k]))
        assert bad.size == 0, (k, bad[:8], g[k][bad[:4]], o[k][bad[:4]])
    H.compare_errors(g["seq_error"], o["error"], flagged, V.ERR_TOKEN | V.ERR_NONFINITE)
    fine = ok & (o["error"] == 0)
    for k in ("p_at_draft", "q_at_draft"):
        gn, on = np.isnan(g[k][fine]), np.isnan(o[k][fine])
        assert np.array_equal(gn, on), k
        assert H.close(g[k][fine][~gn], o[k][fine][~on]).all(), k
    assert H.close(g["resid_mass"][fine], o["resid_mass"][fine]).all()


SMALL = [
    synth.with_sizes(S["sampling_chain_b64_g5_v128256_bf16_a05"], name="a05_v20000", B=24, V=20000),
    synth.with_sizes(S["sampling_chain_b64_g5_v128256_bf16_a60"], name="a60_v20001_pad3", B=24, V=20001, pad=3),
    synth.with_sizes(S["sampling_chain_b64_g5_v128256_bf16_a90"], name="a90_v9000", B=24, V=9000),
    synth.with_sizes(S["sampling_chain_b32_g8_v32000_bf16"], name="g8_f32_v5003", B=12, V=5003, dtype="f32"),
    synth.with_sizes(S["sampling_chain_b32_g8_v32000_bf16"], name="g1_v3000", B=10, gamma=1, V=3000),
]


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: s.name)
def test_consulted_small(cuda_device, spec):
    w = synth.make(spec, seed=8)
    g = H.gpu_chain(w, cuda_device, consulted_only=True)
    o = oracle(w)
    compare(g, o)
    # the ordinary mode makes the same decisions on finite inputs (its row
    # statistics are summed in another order, so not at near ties)
    d = H.gpu_chain(w, cuda_device)
    keep = ~H.set_aside(o, False)
    for k in ("accept_len", "out_token", "rollback_idx", "seq_error"):
        assert np.array_equal(g[k][keep], d[k][keep]), k


@pytest.mark.parametrize("name", ["sampling_chain_b64_g5_v128256_bf16_a05", "sampling_chain_b64_g5_v128256_bf16_a60"])
def test_consulted_full_size(cuda_device, name):
    w = synth.make(S[name], seed=0)
    compare(H.gpu_chain(w, cuda_device, consulted_only=True), oracle(w))


def test_consulted_nonfinite_rows(cuda_device):
    spec = synth.with_sizes(S["sampling_chain_b64_g5_v128256_bf16_a60"], B=18, V=4000)
    w = synth.make(spec, seed=6)
    o0 = V.verify_chain(w["target"], w["draft"], w["tokens"], w["u"], w["v"], w["prefix_len"], spec.temperature,
                        False, spec.dtype, V=spec.V)
    g_ = spec.gamma
    nan = synth.bf16_from_float32(np.array([np.nan], np.float32))[0]
    for b in range(spec.B):
        a = int(o0["accept_len"][b])
        if b % 3 == 0 and a + 1 < g_:
            w["draft"][b, a + 1, 7] = nan          # never read
        elif b % 3 == 1:
            w["target"][b, min(a, g_), 3] = nan    # read
        elif a > 0:
            w["draft"][b, 0, 1] = nan              # read
    g = H.gpu_chain(w, cuda_device, consulted_only=True)
    o = oracle(w)
    compare(g, o)
    assert (g["seq_error"][0::3] & 4 == 0).all()
