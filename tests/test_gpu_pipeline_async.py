"""Asynchronous PipeSpec snapshot on the GPU against the oracle.

Sequences whose accept or draw uniform lies within the oracle's tolerance of
a decision boundary (any stage) are set aside as for the other sampling
paths; every other output must match exactly.  Greedy runs compare every
sequence.
"""

import numpy as np
import pytest

from oracle import pipeline_async as A
from oracle import verify as V
from workloads import synth

from . import gpu_helpers as H

pytestmark = pytest.mark.gpu

BASE = synth.PIPELINE_ASYNC_SPECS["pipeline4_async_b128_g8_g6_g4_v128256_bf16"]
KEYS = ("a", "t", "t_valid", "r", "committed")


def gpu_async(w, device, greedy=None, length=None):
    from draft_verification_gb300 import PipelineAsyncPlan
    s = w["spec"]
    greedy = s.greedy if greedy is None else greedy
    tg = [H.logits_view(H.dev_logits(x, s.dtype, device), s.V) for x in w["targets"]]
    dr = None if greedy else [H.logits_view(H.dev_logits(x, s.dtype, device), s.V) for x in w["drafts"]]
    plan = PipelineAsyncPlan(tg, dr, [H.dev(t, device) for t in w["tokens"]],
                             H.dev(w["length"] if length is None else length, device),
                             None if greedy else [H.dev(u, device) for u in w["us"]],
                             None if greedy else [H.dev(v, device) for v in w["vs"]], greedy=greedy,
                             temperature=s.temperature, final_bonus=s.final_bonus)
    return H.to_np(plan.run())


def oracle_async(w, greedy=None, length=None):
    s = w["spec"]
    greedy = s.greedy if greedy is None else greedy
    return A.verify_pipeline_async(w["targets"], None if greedy else w["drafts"], w["tokens"], w["us"], w["vs"],
                                   w["length"] if length is None else length, s.temperature, greedy,
                                   s.final_bonus, s.dtype, V=s.V)


def compare(g, o, greedy):
    B = len(o["committed"])
    flagged = H.set_aside(o, greedy)
    assert flagged.mean() <= H.MAX_FLAGGED, f"{flagged.sum()} of {B} sequences set aside"
    ok = ~flagged
    for k in KEYS:
        gk, ok_k = g[k], o[k]
        diff = (gk != ok_k) if gk.ndim == 1 else (gk != ok_k).any(axis=1)
        bad = np.flatnonzero(ok & diff)
        assert bad.size == 0, f"{k} mismatch at {bad[:8]}: gpu {gk[bad[:4]]} oracle {ok_k[bad[:4]]}"
    H.compare_errors(g["seq_error"], o["error"], flagged, V.ERR_TOKEN | V.ERR_NONFINITE | A.ERR_WINDOW)


CASES = [
    synth.with_sizes(BASE, name="k2_v9001", B=12, windows=(5,), V=9001),
    synth.with_sizes(BASE, name="k3_v12000_pad3", B=10, windows=(6, 4), V=12000, pad=3),
    synth.with_sizes(BASE, name="k4_v20000", B=16, V=20000),
    synth.with_sizes(BASE, name="k4_bonus_full_windows_v20000", B=16, V=20000, final_bonus=True, extra=0),
    synth.with_sizes(BASE, name="k5_bonus_v7000", B=14, windows=(8, 6, 4, 3), V=7000, a=(0.9,) * 4,
                     s=(0.465, 1.0, 1.0, 1.0), final_bonus=True, extra=1),
    synth.with_sizes(BASE, name="k8_v3000", B=10, windows=(6, 5, 5, 4, 4, 3, 3), V=3000, a=(0.95,) * 7,
                     s=(0.4,) * 7, extra=1),
    synth.with_sizes(BASE, name="k4_f32_v4001", B=10, V=4001, dtype="f32"),
    synth.with_sizes(BASE, name="k4_greedy_v16000", B=12, V=16000, greedy=True, final_bonus=True, extra=1),
    synth.with_sizes(BASE, name="k6_greedy_v5000", B=12, windows=(8, 7, 6, 5, 4), V=5000, a=(0.95,) * 5,
                     s=(0.3,) * 5, greedy=True, extra=0),
]


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_pipeline_async_small(cuda_device, spec):
    w = synth.make(spec, seed=7)
    compare(gpu_async(w, cuda_device), oracle_async(w), spec.greedy)


def test_pipeline_async_full_size(cuda_device):
    w = synth.make(BASE, seed=0)
    compare(gpu_async(w, cuda_device), oracle_async(w), False)
    compare(gpu_async(w, cuda_device, greedy=True), oracle_async(w, greedy=True), True)


def test_pipeline_async_malformed_windows_and_data_errors(cuda_device):
    spec = synth.with_sizes(BASE, B=6, V=3000)
    w = synth.make(spec, seed=9)
    length = w["length"].copy()
    length[0, 1] = length[1, 1] + spec.windows[0] - 1   # stage 1's window does not fit in O_0
    length[3, 2] = -1                                   # a negative length
    w["tokens"][1][4, 0] = spec.V                       # a token outside the vocabulary
    nan = synth.bf16_from_float32(np.array([np.nan], np.float32))[0]
    w["targets"][2][5, 1, 7] = nan                      # a non-finite row in stage 3
    for greedy in (False, True):
        g = gpu_async(w, cuda_device, greedy=greedy, length=length)
        o = oracle_async(w, greedy=greedy, length=length)
        compare(g, o, greedy)
        assert g["seq_error"][1] & A.ERR_WINDOW and g["seq_error"][2] & A.ERR_WINDOW
        assert g["seq_error"][4] & V.ERR_TOKEN and g["seq_error"][5] & V.ERR_NONFINITE
        for b in (1, 2, 4, 5):
            assert (g["r"][b] == length[:-1, b]).all() and g["committed"][b] == length[-1, b]
            assert (g["t"][b] == -1).all() and (g["a"][b] == 0).all()
        assert g["error_word"][0] & (A.ERR_WINDOW | V.ERR_TOKEN | V.ERR_NONFINITE) == (
            A.ERR_WINDOW | V.ERR_TOKEN | V.ERR_NONFINITE)


@pytest.mark.parametrize("greedy", [False, True])
def test_two_models_equal_the_chain_entry(cuda_device, greedy):
    # k = 2 is one chain verification with prefix l_1: same accept length and
    # token, committed = the chain's rollback index + 1 when the window ends O_0
    spec = synth.with_sizes(BASE, B=16, windows=(6,), V=11000, greedy=greedy, extra=0)
    w = synth.make(spec, seed=12)
    g = gpu_async(w, cuda_device)
    from draft_verification_gb300 import ChainPlan
    tgt = H.logits_view(H.dev_logits(w["targets"][0], spec.dtype, cuda_device), spec.V)
    drf = H.logits_view(H.dev_logits(w["drafts"][0], spec.dtype, cuda_device), spec.V)
    c = H.to_np(ChainPlan(tgt, drf, H.dev(w["tokens"][0], cuda_device), H.dev(w["us"][0], cuda_device),
                          H.dev(w["vs"][0], cuda_device), H.dev(w["length"][1], cuda_device), greedy=greedy,
                          temperature=spec.temperature).run())
    assert np.array_equal(g["a"][:, 0], c["accept_len"])
    assert np.array_equal(g["t"][:, 0], c["out_token"])
    assert np.array_equal(g["committed"], c["rollback_idx"] + 1)


def test_pipeline_async_graph_replays(cuda_device):
    # one call (per-stage chains with their batch-group streams, then the
    # combine) captured in a CUDA graph and replayed on new inputs
    import torch
    from draft_verification_gb300 import PipelineAsyncPlan
    spec = synth.with_sizes(BASE, B=40, V=9000, final_bonus=True, extra=1)
    ws = [synth.make(spec, seed=40 + i) for i in range(3)]
    w0 = ws[0]
    tg = [H.logits_view(H.dev_logits(x, spec.dtype, cuda_device), spec.V) for x in w0["targets"]]
    dr = [H.logits_view(H.dev_logits(x, spec.dtype, cuda_device), spec.V) for x in w0["drafts"]]
    tok = [H.dev(t, cuda_device) for t in w0["tokens"]]
    us = [H.dev(u, cuda_device) for u in w0["us"]]
    vs = [H.dev(v, cuda_device) for v in w0["vs"]]
    length = H.dev(w0["length"], cuda_device)
    plan = PipelineAsyncPlan(tg, dr, tok, length, us, vs, temperature=spec.temperature, final_bonus=True)
    stream = torch.cuda.Stream(cuda_device)
    plan.run(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        plan.run(stream)
    for w in ws[1:] + ws[:1]:
        for dst, src in zip(tg, w["targets"]):
            dst.copy_(H.logits_view(H.dev_logits(src, spec.dtype, cuda_device), spec.V))
        for dst, src in zip(dr, w["drafts"]):
            dst.copy_(H.logits_view(H.dev_logits(src, spec.dtype, cuda_device), spec.V))
        for dst, src in zip(tok + us + vs, w["tokens"] + w["us"] + w["vs"]):
            dst.copy_(H.dev(src, cuda_device))
        length.copy_(H.dev(w["length"], cuda_device))
        plan.out["error_word"].zero_()
        graph.replay()
        torch.cuda.synchronize()
        compare(H.to_np(plan.out), oracle_async(w), False)
