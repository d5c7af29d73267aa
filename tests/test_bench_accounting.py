"""bench.py's work accounting on the CPU: the units and algorithmic bytes
(or flops) that every reported rate and roofline fraction divides by."""

import itertools

import numpy as np
import pytest

import bench
from workloads import synth


def _reachable_keep_states(L, M):
    """States (i - 1, j) whose layer i - 1 is applied in the DP, counted by
    brute force: j keeps layer i - 1 (j <= i - 1) and (i, j) can still end at
    (L, M) with at most one skip per remaining layer (M - j <= L - i)."""
    n = 0
    for i in range(1, L + 1):
        for j in range(0, min(i, M) + 1):
            if j <= i - 1 and M - j <= L - i:
                n += 1
    return n


@pytest.mark.parametrize("L,M", [(32, 12), (8, 0), (8, 8), (5, 2), (1, 0), (1, 1), (12, 11)])
def test_clasp_columns_count_the_reachable_kept_states(L, M):
    spec = synth.with_sizes(synth.CLASP_SPECS["clasp_b16_l32_d4096_m12_bf16"], B=3, L=L, M=M)
    assert bench.clasp_columns(spec) == 2 * 3 * _reachable_keep_states(L, M)


def test_clasp_columns_and_bytes_of_the_workload():
    spec = synth.CLASP_SPECS["clasp_b16_l32_d4096_m12_bf16"]
    assert bench.clasp_columns(spec) == 8320
    assert bench.clasp_bytes(spec) == 32 * 4096 * 4096 * 2 + 16 * 33 * 4096 * 4
    assert bench.clasp_flops(spec) == 2 * 4096 * 4096 * 8320


def test_clasp_band_matches_brute_force_reachability():
    # the kernels evaluate max(0, M - (L - i)) <= j <= min(i, M); brute force
    # over skip sets: (i, j) lies on some path that ends at (L, M)
    for L, M in [(6, 2), (7, 7), (5, 0), (9, 4)]:
        reach = set()
        for S in itertools.combinations(range(L), M):
            j = 0
            reach.add((0, 0))
            for i in range(1, L + 1):
                j += (i - 1) in S
                reach.add((i, j))
        for i in range(L + 1):
            band = {j for j in range(max(0, M - (L - i)), min(i, M) + 1)}
            assert band == {j for (ii, j) in reach if ii == i}, (L, M, i)


def test_async_bytes_and_tokens():
    spec = synth.PIPELINE_ASYNC_SPECS["pipeline4_async_b128_g8_g6_g4_v128256_bf16"]
    assert bench.async_rows(spec) == (9 + 8) + (7 + 6) + (5 + 4)
    assert bench.async_bytes(spec) == 128 * 39 * 128256 * 2
    assert bench.async_tokens(spec) == 128 * 18
    g = synth.with_sizes(spec, greedy=True, dtype="f32")
    assert bench.async_bytes(g) == 128 * (9 + 7 + 5) * 128256 * 4


def test_async_workload_layout_is_consistent():
    spec = synth.with_sizes(synth.PIPELINE_ASYNC_SPECS["pipeline4_async_b128_g8_g6_g4_v128256_bf16"], B=5, V=300)
    w = synth.make(spec, seed=4)
    L = w["length"]
    assert L.shape == (4, 5) and (L >= 0).all()
    for s in range(1, 4):
        gap = L[s - 1] - L[s] - spec.windows[s - 1]
        assert (gap >= 0).all() and (gap <= spec.extra).all()
        assert w["targets"][s - 1].shape == (5, spec.windows[s - 1] + 1, 300)
        assert w["drafts"][s - 1].shape == (5, spec.windows[s - 1], 300)
        assert ((w["tokens"][s - 1] >= 0) & (w["tokens"][s - 1] < 300)).all()
    again = synth.make(spec, seed=4)
    assert all(np.array_equal(a, b) for a, b in zip(w["tokens"], again["tokens"]))


def _stats_launches_per_call(name, calls):
    """Statistics-kernel launches per call in a committed ncu launch list."""
    import os
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles",
                        f"launches_{name}.md")
    for line in open(path):
        if line.startswith("| stats_kernel"):
            return int(line.split("|")[2]) // calls
    raise AssertionError(name)


@pytest.mark.parametrize("name,per_call", [("sampling_chain_b32_g8_v32000_bf16", 2),
                                           ("sampling_chain_b64_g5_v128256_bf16_a60", 8),
                                           ("greedy_chain_b4_g4_v1000_f32", 2)])
def test_chain_launches_per_call_match_the_launch_lists(name, per_call):
    spec = synth.SPECS[name]
    w = dict(kind="chain", spec=spec)
    assert bench.launches_per_call(w) == per_call
    # the launch lists (5 calls each) saw one statistics kernel per group
    assert 2 * _stats_launches_per_call(name, 5) == per_call


def test_async_launches_per_call_match_the_launch_list():
    spec = synth.PIPELINE_ASYNC_SPECS["pipeline4_async_b128_g8_g6_g4_v128256_bf16"]
    assert bench.async_launches_per_call(spec) == 3 * 8 + 1
    assert 2 * _stats_launches_per_call(spec.name, 5) + 1 == bench.async_launches_per_call(spec)


def test_consulted_and_lm_head_launch_counts():
    # a consulted-only chain or tree call is one walk kernel (a small tree
    # call is one group: statistics and walk); the LM-head chain is one head
    # kernel per head plus the walk
    import bench
    from workloads import synth
    chain = synth.make(synth.with_sizes(synth.SPECS["sampling_chain_b64_g5_v128256_bf16_a05"], B=2, V=100), seed=0)
    tree = synth.make(synth.with_sizes(synth.SPECS["tree_b16_n64_v50257_bf16"], B=2, V=100), seed=0)
    old = bench.CONSULTED
    try:
        bench.CONSULTED = True
        assert bench.launches_per_call(chain) == 1 and bench.launches_per_call(tree) == 1
        bench.CONSULTED = False
        assert bench.launches_per_call(chain) == 2 and bench.launches_per_call(tree) == 2
    finally:
        bench.CONSULTED = old
    spec = synth.LM_HEAD_SPECS["lm_head_chain_b64_g5_v128256_d4096_bf16"]
    assert bench.lm_head_flops(spec) == 2 * 128256 * (64 * 6 * 4096 + 64 * 5 * 4096)
    assert bench.lm_head_bytes(spec) == 2 * 128256 * 4096 * 2 + 64 * (6 + 5) * 4096 * 2


def test_tree_launches_per_call_follow_the_grouping_rule():
    # trees are grouped like chains, with at least 4 trees and 40 MB of
    # logits per group: the full tree workload (16 trees, 206 MB) runs as 4
    # groups, 8 trees of 2 x 64 rows at V = 50257 (103 MB) as 2
    spec = synth.SPECS["tree_b16_n64_v50257_bf16"]
    w = synth.make(synth.with_sizes(spec, V=100), seed=0)
    n = w["parent"].shape[1]
    assert bench.chain_groups(16, 2 * n, 50257, 2, min_seqs=4) == 4
    assert bench.chain_groups(8, 2 * n, 50257, 2, min_seqs=4) == 2
    assert bench.chain_groups(3, 2 * n, 50257, 2, min_seqs=4) == 1
    w = dict(kind="tree", spec=spec, parent=w["parent"])
    assert bench.launches_per_call(w) == 8
