"""The bounded waits' give-up path, and grouped calls replayed from a graph.

A wait that runs out must end the walk with SPEC_ERR_INTERNAL and empty
outputs, never a hang or a fault, and leave the GPU usable.  The library's
test hook (spec_test_inject_copy_timeout) makes every bulk-copy stage of a
residual pass expect 16 bytes that never come: the copies themselves land,
only the stage's barrier phase stays open, so its wait gives up after its
poll limit (about 65 ms) with nothing in flight.
"""

import numpy as np
import pytest
import torch

from workloads import synth

from . import gpu_helpers as H

pytestmark = pytest.mark.gpu

S = synth.SPECS
W = synth.with_sizes


def test_copy_wait_gives_up_with_internal_error(cuda_device):
    from draft_verification_gb300 import _lib
    lib = _lib.lib()
    # V = 1504: one pass tile, so each sequence's walk is a single CTA, and
    # 16-byte aligned rows, so the residual pass takes the bulk-copy path
    spec = W(S["sampling_chain_b32_g8_v32000_bf16"], B=4, gamma=3, V=1504)
    w = synth.make(spec, seed=40)
    assert lib.spec_test_inject_copy_timeout(1) == _lib.SPEC_OK
    try:
        g = H.gpu_chain(w, cuda_device)
    finally:
        assert lib.spec_test_inject_copy_timeout(0) == _lib.SPEC_OK
    assert (g["seq_error"] == _lib.ERR_INTERNAL).all(), g["seq_error"]
    assert g["error_word"][0] == _lib.ERR_INTERNAL
    assert (g["accept_len"] == 0).all() and (g["out_token"] == -1).all()
    assert np.array_equal(g["rollback_idx"], w["prefix_len"])
    # the context is intact: the same call, hook off, matches the oracle
    H.compare_chain(H.gpu_chain(w, cuda_device), H.oracle_chain(w), False)


def test_grouped_chain_graph_replays(cuda_device):
    # B = 64 rows of 128256 logits: the call runs as four batch groups on the
    # calling thread's side streams, forked from and joined into the capture
    # stream; the captured fork / join must order every group, replay after
    # replay, with new inputs copied into the captured buffers
    import draft_verification_gb300 as dv
    spec = S["sampling_chain_b64_g5_v128256_bf16_a60"]
    ws = [synth.make(spec, seed=50 + i) for i in range(2)]
    plan = H.chain_plan(ws[0], cuda_device)
    stream = torch.cuda.Stream(cuda_device)
    plan.run(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        plan.run(stream)
    tgt, drf = plan.keep[0], plan.keep[1]
    for w in ws[1:] + ws[:1]:
        tgt.copy_(H.logits_view(H.dev_logits(w["target"], spec.dtype, cuda_device), spec.V))
        drf.copy_(H.logits_view(H.dev_logits(w["draft"], spec.dtype, cuda_device), spec.V))
        for k, x in (("tokens", 2), ("u", 3), ("v", 4), ("prefix_len", 5)):
            plan.keep[x].copy_(H.dev(w[k], cuda_device))
        plan.out["error_word"].zero_()
        graph.replay()
        torch.cuda.synchronize()
        H.compare_chain(H.to_np(plan.out), H.oracle_chain(w), False)
    assert dv.workspace_bytes("chain", 64, 5, 128256) <= plan.workspace.numel()


def test_grouped_tree_graph_replays(cuda_device):
    # 16 trees of 64 nodes at V = 50257 (206 MB of logits): the call runs as
    # four batch groups of four trees on the side streams; replayed from a
    # graph with new inputs copied into the captured buffers
    from draft_verification_gb300 import TreePlan
    spec = S["tree_b16_n64_v50257_bf16"]
    ws = [synth.make(spec, seed=60 + i) for i in range(2)]
    w0 = ws[0]
    plan = TreePlan(H.dev(w0["parent"], cuda_device), H.dev(w0["tokens"], cuda_device),
                    H.logits_view(H.dev_logits(w0["target"], spec.dtype, cuda_device), spec.V),
                    H.logits_view(H.dev_logits(w0["draft"], spec.dtype, cuda_device), spec.V),
                    H.dev(w0["u"], cuda_device), H.dev(w0["v"], cuda_device), H.dev(w0["prefix_len"], cuda_device),
                    max_depth=w0["max_depth"], temperature=spec.temperature)
    stream = torch.cuda.Stream(cuda_device)
    plan.run(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        plan.run(stream)
    for w in ws[1:] + ws[:1]:
        for k, x in (("parent", 0), ("tokens", 1), ("u", 4), ("v", 5), ("prefix_len", 6)):
            plan.keep[x].copy_(H.dev(w[k], cuda_device))
        plan.keep[2].copy_(H.logits_view(H.dev_logits(w["target"], spec.dtype, cuda_device), spec.V))
        plan.keep[3].copy_(H.logits_view(H.dev_logits(w["draft"], spec.dtype, cuda_device), spec.V))
        plan.out["error_word"].zero_()
        graph.replay()
        torch.cuda.synchronize()
        H.compare_tree(H.to_np(plan.out), H.oracle_tree(w), False)
