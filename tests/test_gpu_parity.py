"""CUDA path vs the CPU oracle, element by element, on seeded inputs.

Small shapes span several 8192-element statistics chunks and 2048-element
walker tiles with ragged tails, misaligned row strides, both dtypes, both
modes and several temperatures; the five measured workloads run at their full
sizes, in the launch configuration the benchmark uses, with every sequence
checked against the oracle.
"""

import math

import numpy as np
import pytest
import torch

from workloads import synth

from . import gpu_helpers as H

pytestmark = pytest.mark.gpu

S = synth.SPECS
W = synth.with_sizes

CHAIN_SMALL = [
    W(S["sampling_chain_b32_g8_v32000_bf16"], name="bf16_v20011_g5_pad3", B=12, gamma=5, V=20011, pad=3),
    W(S["sampling_chain_b32_g8_v32000_bf16"], name="bf16_v7_g3", B=9, gamma=3, V=7),
    W(S["sampling_chain_b32_g8_v32000_bf16"], name="bf16_v1_g2", B=3, gamma=2, V=1),
    W(S["sampling_chain_b32_g8_v32000_bf16"], name="bf16_v16387_g1_T1.6", B=10, gamma=1, V=16387,
      temperature=1.6),
    W(S["sampling_chain_b32_g8_v32000_bf16"], name="bf16_g0_bonus_only", B=6, gamma=0, V=9000),
    W(S["sampling_chain_b64_g5_v128256_bf16_a60"], name="bf16_v40000_g8_T0.7_pad5", B=6, gamma=8,
      V=40000, pad=5),
    W(S["sampling_chain_b32_g8_v32000_bf16"], name="f32_v5003_g3_pad1", B=8, gamma=3, V=5003,
      dtype="f32", pad=1),
    W(S["sampling_chain_b32_g8_v32000_bf16"], name="f32_v12000_g32", B=3, gamma=32, V=12000, dtype="f32"),
    W(S["greedy_chain_b4_g4_v1000_f32"], name="greedy_f32_v4097_pad2", B=7, gamma=6, V=4097, pad=2),
    W(S["greedy_chain_b4_g4_v1000_f32"], name="greedy_bf16_v50257", B=5, gamma=4, V=50257, dtype="bf16"),
    # the interface's limits: the largest vocabulary (128 statistics chunks
    # per row; a low temperature concentrates the softmax on a few tokens, so
    # that draws and accept tests do not fall within the near-tie margins,
    # which a flat distribution over 2^21 tokens would) and the largest batch
    # (65535 sequences of a tiny vocabulary: launch grids 65535 deep, one
    # single-CTA cluster per sequence)
    W(S["sampling_chain_b32_g8_v32000_bf16"], name="bf16_vmax_2097152_g2", B=2, gamma=2, V=2097152,
      temperature=0.05),
    W(S["sampling_chain_b32_g8_v32000_bf16"], name="bf16_bmax_65535_v16_g1", B=65535, gamma=1, V=16),
    W(S["greedy_chain_b4_g4_v1000_f32"], name="greedy_f32_bmax_65535_v16", B=65535, gamma=1, V=16),
]


@pytest.mark.parametrize("spec", CHAIN_SMALL, ids=lambda s: s.name)
def test_chain_small(cuda_device, spec):
    w = synth.make(spec, seed=5)
    H.compare_chain(H.gpu_chain(w, cuda_device), H.oracle_chain(w), spec.greedy)


@pytest.mark.parametrize("name", [
    "greedy_chain_b4_g4_v1000_f32",
    "sampling_chain_b32_g8_v32000_bf16",
    "sampling_chain_b64_g5_v128256_bf16_a05",
    "sampling_chain_b64_g5_v128256_bf16_a30",
    "sampling_chain_b64_g5_v128256_bf16_a60",
    "sampling_chain_b64_g5_v128256_bf16_a90",
])
def test_chain_full_size(cuda_device, name):
    spec = S[name]
    w = synth.make(spec, seed=0)
    g = H.gpu_chain(w, cuda_device)
    H.compare_chain(g, H.oracle_chain(w), spec.greedy)
    if not spec.greedy:
        # greedy rule on the same sampling inputs (draft logits not read)
        H.compare_chain(H.gpu_chain(w, cuda_device, greedy=True), H.oracle_chain(w, greedy=True), True)


def test_chain_batch_groups_ragged(cuda_device):
    # B = 37 rows of 128256 logits is large enough to be split into two
    # groups of sequences (18 and 19) on library streams; every sequence,
    # including those at the group boundary, must match the oracle, and a
    # data error in the second group must stay with its sequence
    spec = W(S["sampling_chain_b64_g5_v128256_bf16_a60"], B=37)
    w = synth.make(spec, seed=9)
    w["tokens"][20, 2] = spec.V  # out of range, in the second group
    g = H.gpu_chain(w, cuda_device)
    H.compare_chain(g, H.oracle_chain(w), False)
    assert g["seq_error"][20] == 1 and (np.delete(g["seq_error"], 20) & 1).sum() == 0


def test_chain_workspace_reused_across_shapes(cuda_device):
    # one workspace (sized for the largest call) serves chain and tree calls
    # of different sizes, dtypes and modes in turn: whatever an earlier call
    # left in it never passes for the current call's statistics
    import draft_verification_gb300 as dv
    big = W(S["sampling_chain_b32_g8_v32000_bf16"], B=24, gamma=6, V=40000)
    tree = W(S["tree_b16_n64_v50257_bf16"], B=3, V=5000, n_nodes=20, branching=(3, 3, 2))
    need = max(dv.workspace_bytes("chain", 24, 6, 40000), dv.workspace_bytes("tree", 3, 20, 5000))
    ws = torch.zeros(need, dtype=torch.uint8, device=cuda_device)
    calls = [(big, 1), (W(big, B=5, V=9000), 2), (big, 3), (tree, 4), (W(big, greedy=True), 5),
             (W(big, B=7, gamma=3, dtype="f32", V=12001), 6), (big, 7)]
    for spec, seed in calls:
        w = synth.make(spec, seed=seed)
        if w["kind"] == "tree":
            H.compare_tree(H.gpu_tree(w, cuda_device, workspace=ws), H.oracle_tree(w), False)
        else:
            H.compare_chain(H.gpu_chain(w, cuda_device, workspace=ws), H.oracle_chain(w), spec.greedy)


def test_chain_graph_replays(cuda_device):
    # a call captured once in a CUDA graph and replayed on new inputs copied
    # into the same buffers (the way the benchmark runs it): every replay is
    # verified against the oracle
    spec = W(S["sampling_chain_b64_g5_v128256_bf16_a60"], B=12)
    ws = [synth.make(spec, seed=20 + i) for i in range(3)]
    plan = H.chain_plan(ws[0], cuda_device)
    tgt, drf = plan.keep[0], plan.keep[1]
    stream = torch.cuda.Stream(cuda_device)
    plan.run(stream)  # first call outside the capture
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        plan.run(stream)
    for w in ws[1:] + ws[:1]:
        tgt.copy_(H.logits_view(H.dev_logits(w["target"], spec.dtype, cuda_device), spec.V))
        drf.copy_(H.logits_view(H.dev_logits(w["draft"], spec.dtype, cuda_device), spec.V))
        for k, x in (("tokens", 2), ("u", 3), ("v", 4), ("prefix_len", 5)):
            plan.keep[x].copy_(H.dev(w[k], cuda_device))
        graph.replay()
        torch.cuda.synchronize()
        H.compare_chain(H.to_np(plan.out), H.oracle_chain(w), False)


def test_chain_data_errors(cuda_device):
    spec = W(S["sampling_chain_b32_g8_v32000_bf16"], B=6, gamma=4, V=3000)
    w = synth.make(spec, seed=2)
    nan, pinf, ninf = (synth.bf16_from_float32(np.array([x], np.float32))[0]
                       for x in (math.nan, math.inf, -math.inf))
    w["target"][1, 2, 17] = nan
    w["draft"][2, 0, 2999] = pinf
    w["target"][3, 4, :] = ninf
    w["tokens"][4, 2] = spec.V
    w["target"][5, 1, :100] = ninf  # masked entries are allowed
    for greedy in (False, True):
        g = H.gpu_chain(w, cuda_device, greedy=greedy)
        o = H.oracle_chain(w, greedy=greedy)
        H.compare_chain(g, o, greedy)
        bad = (o["error"] & 5) != 0
        assert (g["out_token"][bad] == -1).all() and (g["accept_len"][bad] == 0).all()
        assert g["error_word"][0] == np.bitwise_or.reduce(g["seq_error"])


def test_chain_equal_distributions_keep_everything(cuda_device):
    spec = W(S["sampling_chain_b32_g8_v32000_bf16"], B=4, gamma=6, V=5000)
    w = synth.make(spec, seed=3)
    w["draft"][:] = w["target"][:, :6]
    g = H.gpu_chain(w, cuda_device)
    assert (g["accept_len"] == 6).all()
    H.compare_chain(g, H.oracle_chain(w), False)


def test_chain_deterministic(cuda_device):
    w = synth.make(W(S["sampling_chain_b64_g5_v128256_bf16_a60"], B=8), seed=4)
    a = H.gpu_chain(w, cuda_device)
    b = H.gpu_chain(w, cuda_device)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


TREE_SMALL = [
    W(S["tree_b16_n64_v50257_bf16"], name="tree_v3001_n64", B=6, V=3001),
    W(S["tree_b16_n64_v50257_bf16"], name="tree_v12289_n20_pad1", B=5, V=12289, n_nodes=20, pad=1,
      branching=(3, 3, 2, 2)),
    W(S["tree_b16_n64_v50257_bf16"], name="tree_f32_v999_n40", B=4, V=999, dtype="f32", n_nodes=40),
    W(S["tree_b16_n64_v50257_bf16"], name="tree_wide_root", B=4, V=4000, n_nodes=9, branching=(8,)),
    W(S["tree_b16_n64_v50257_bf16"], name="tree_greedy_v20000", B=6, V=20000, greedy=True),
    # the interface's limits: the most nodes (1024, a binary tree ten levels
    # deep) and the largest vocabulary (at a low temperature, as for chains)
    W(S["tree_b16_n64_v50257_bf16"], name="tree_nmax_1024_v64", B=2, V=64, n_nodes=1024, branching=(2,) * 10),
    W(S["tree_b16_n64_v50257_bf16"], name="tree_greedy_nmax_1024_v64", B=2, V=64, n_nodes=1024,
      branching=(2,) * 10, greedy=True),
    W(S["tree_b16_n64_v50257_bf16"], name="tree_vmax_2097152_n6", B=1, V=2097152, n_nodes=6, branching=(2, 2),
      temperature=0.05),
]


@pytest.mark.parametrize("spec", TREE_SMALL, ids=lambda s: s.name)
def test_tree_small(cuda_device, spec):
    w = synth.make(spec, seed=6)
    H.compare_tree(H.gpu_tree(w, cuda_device), H.oracle_tree(w), spec.greedy)


def test_tree_full_size(cuda_device):
    spec = S["tree_b16_n64_v50257_bf16"]
    w = synth.make(spec, seed=0)
    H.compare_tree(H.gpu_tree(w, cuda_device), H.oracle_tree(w), False)
    H.compare_tree(H.gpu_tree(w, cuda_device, greedy=True), H.oracle_tree(w, greedy=True), True)


def test_tree_data_errors(cuda_device):
    spec = W(S["tree_b16_n64_v50257_bf16"], B=6, V=2000, n_nodes=12, branching=(3, 2, 2))
    w = synth.make(spec, seed=8)
    w["parent"][1, 5] = 7          # parent after child
    w["parent"][2, 0] = 0          # root with a parent
    w["tokens"][3, 4] = -2         # token out of range
    nan = synth.bf16_from_float32(np.array([math.nan], np.float32))[0]
    w["draft"][4, 3, 9] = nan
    w["max_depth"] = w["max_depth"]  # sequence 5 stays valid
    for greedy in (False, True):
        H.compare_tree(H.gpu_tree(w, cuda_device, greedy=greedy), H.oracle_tree(w, greedy=greedy), greedy)
    w["max_depth"] = 1             # every tree is deeper than allowed
    g = H.gpu_tree(w, cuda_device)
    assert (g["seq_error"] & 2).all() and (g["path_nodes"] == -1).all()


def test_tree_root_only_and_chain_shaped(cuda_device):
    chain = W(S["sampling_chain_b32_g8_v32000_bf16"], B=8, gamma=5, V=7000)
    w = synth.make(chain, seed=9)
    gc = H.gpu_chain(w, cuda_device)
    N = 6
    tw = dict(kind="tree", spec=W(S["tree_b16_n64_v50257_bf16"], V=7000, temperature=chain.temperature),
              parent=np.tile(np.arange(-1, N - 1, dtype=np.int32), (8, 1)),
              tokens=np.concatenate([np.zeros((8, 1), np.int32), w["tokens"]], axis=1),
              target=w["target"], draft=np.concatenate([w["draft"], w["draft"][:, :1]], axis=1),
              u=np.concatenate([np.zeros((8, 1), np.float32), w["u"]], axis=1), v=w["v"],
              prefix_len=w["prefix_len"], max_depth=N - 1)
    gt = H.gpu_tree(tw, cuda_device)
    assert np.array_equal(gt["path_len"], gc["accept_len"])
    assert np.array_equal(gt["out_token"], gc["out_token"])
    H.compare_tree(gt, H.oracle_tree(tw), False)
    root = dict(tw, parent=tw["parent"][:, :1], tokens=tw["tokens"][:, :1], target=w["target"][:, :1],
                draft=w["draft"][:, :1], u=tw["u"][:, :1], max_depth=0)
    H.compare_tree(H.gpu_tree(root, cuda_device), H.oracle_tree(root), False)


CASCADE_SMALL = [
    W(S["cascade_b128_g8_g4_v128256_bf16"], name="cascade_v9001_pad7", B=10, V=9001, pad=7),
    W(S["cascade_b128_g8_g4_v128256_bf16"], name="cascade_g3_g4_v30000", B=8, gamma1=3, gamma2=4, V=30000),
    W(S["cascade_b128_g8_g4_v128256_bf16"], name="cascade_f32_v4000", B=6, V=4000, dtype="f32"),
    W(S["cascade_b128_g8_g4_v128256_bf16"], name="cascade_greedy_v16000", B=8, V=16000, greedy=True),
    # the largest vocabulary the interface accepts (at a low temperature, as
    # for chains)
    W(S["cascade_b128_g8_g4_v128256_bf16"], name="cascade_vmax_2097152", B=2, V=2097152, temperature=0.05),
]


@pytest.mark.parametrize("spec", CASCADE_SMALL, ids=lambda s: s.name)
def test_cascade_small(cuda_device, spec):
    w = synth.make(spec, seed=10)
    H.compare_cascade(H.gpu_cascade(w, cuda_device), H.oracle_cascade(w), spec.greedy)


def test_cascade_full_size(cuda_device):
    spec = S["cascade_b128_g8_g4_v128256_bf16"]
    w = synth.make(spec, seed=0)
    g = H.gpu_cascade(w, cuda_device)
    H.compare_cascade(g, H.oracle_cascade(w), False)
    assert (g["r0"] - w["base0"] <= g["a1"]).all() and (g["committed"] <= g["w2"]).all()
    H.compare_cascade(H.gpu_cascade(w, cuda_device, greedy=True), H.oracle_cascade(w, greedy=True), True)


def test_host_buffers_end_to_end(cuda_device):
    """CPU tensors in, CPU tensors out, through the public call."""
    import draft_verification_gb300 as dv
    spec = W(S["sampling_chain_b32_g8_v32000_bf16"], B=4, V=9000)
    w = synth.make(spec, seed=12)
    to_bf16 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    out = dv.verify_chain(to_bf16(w["target"]), to_bf16(w["draft"]), torch.from_numpy(w["tokens"]),
                          torch.from_numpy(w["u"]), torch.from_numpy(w["v"]),
                          torch.from_numpy(w["prefix_len"]), temperature=spec.temperature)
    torch.cuda.synchronize()
    assert out["accept_len"].device.type == "cpu"
    g = {k: v.numpy() for k, v in out.items()}
    H.compare_chain(g, H.oracle_chain(w), False)
