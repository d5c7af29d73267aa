"""Cache compaction on the GPU against the oracle, byte for byte."""

import numpy as np
import pytest
import torch

from oracle import compact as K
from workloads import synth

from . import gpu_helpers as H

pytestmark = pytest.mark.gpu

BASE = synth.COMPACT_SPECS["tree_kv_compact_b16_n64_d6_w131072"]


def gpu_compact(w, device):
    import draft_verification_gb300 as dv
    spec = w["spec"]
    W = spec.row_bytes
    tree = torch.from_numpy(w["tree_rows"]).to(device)[:, :, :W]
    cache = torch.from_numpy(w["cache"]).to(device)[:, :, :W]
    err = dv.compact_tree_path(tree, cache, H.dev(w["path_nodes"], device), H.dev(w["path_len"], device),
                               H.dev(w["prefix_len"], device))
    torch.cuda.synchronize()
    return cache.cpu().numpy(), err.cpu().numpy()


def oracle_compact(w):
    W = w["spec"].row_bytes
    out, err = K.compact_tree_path(w["tree_rows"][:, :, :W], w["cache"][:, :, :W], w["path_nodes"],
                                   w["path_len"], w["prefix_len"])
    return out, err


def check(w, device):
    W = w["spec"].row_bytes
    g, ge = gpu_compact(w, device)
    o, oe = oracle_compact(w)
    assert np.array_equal(ge, oe), (ge, oe)
    assert np.array_equal(g, o)
    return g


CASES = [
    synth.with_sizes(BASE, name="w64_vec", B=9, row_bytes=64),
    synth.with_sizes(BASE, name="w40_bytes", B=7, row_bytes=40),
    synth.with_sizes(BASE, name="w4096_pad16_vec", B=5, row_bytes=4096, pad=16),
    synth.with_sizes(BASE, name="w4096_pad8_bytes", B=5, row_bytes=4096, pad=8),
    synth.with_sizes(BASE, name="w40000_3chunks_bytes", B=4, row_bytes=40000),
    synth.with_sizes(BASE, name="w65536_4chunks_vec", B=6, row_bytes=65536, keep=0.95),
    synth.with_sizes(BASE, name="depth12_keep1", B=3, row_bytes=1024, max_depth=12, keep=1.0,
                     branching=(2,) * 12, n_nodes=100),
]


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_compact_small(cuda_device, spec):
    check(synth.make(spec, seed=3), cuda_device)


def test_compact_full_size(cuda_device):
    w = synth.make(BASE, seed=0)
    check(w, cuda_device)


def test_compact_edge_cases(cuda_device):
    w = synth.make(synth.with_sizes(BASE, B=6, row_bytes=256, keep=0.9), seed=5)
    pn, pl, pre = w["path_nodes"], w["path_len"], w["prefix_len"]
    C = w["cache"].shape[1]
    pn[0, :] = -1                       # verifier data error: skipped, no bit
    pl[0] = 0
    pn[1, :] = -1                       # root only
    pn[1, 0] = 0
    pl[1] = 0
    pn[2, 1] = 64                       # node outside the tree
    pl[2] = max(int(pl[2]), 1)
    pre[3] = C - int(pl[3])             # last row one past the cache end
    pl[4] = pn.shape[1]                 # longer than max_depth
    pre[5] = 0                          # writes at the cache start
    g = check(w, cuda_device)
    assert np.array_equal(g[0], w["cache"][0, :, :256])


def test_verify_then_compact(cuda_device):
    # the paths of a GPU tree verification (which matches the oracle's)
    # compacted on the GPU equal the oracle's compaction of the same paths
    tw = synth.make(synth.with_sizes(synth.SPECS["tree_b16_n64_v50257_bf16"], B=8, V=4001), seed=11)
    gv = H.gpu_tree(tw, cuda_device)
    ov = H.oracle_tree(tw)
    H.compare_tree(gv, ov, False)
    W = 512
    rng = np.random.default_rng(4)
    rows = rng.integers(0, 256, (8, 64, W), dtype=np.uint8)
    cache = rng.integers(0, 256, (8, 40, W), dtype=np.uint8)
    prefix = rng.integers(0, 30, 8).astype(np.int32)
    spec = synth.with_sizes(BASE, B=8, row_bytes=W)
    gw = dict(spec=spec, tree_rows=rows, cache=cache, path_nodes=gv["path_nodes"].astype(np.int32),
              path_len=gv["path_len"].astype(np.int32), prefix_len=prefix)
    g, ge = gpu_compact(gw, cuda_device)
    o, oe = K.compact_tree_path(rows, cache, gw["path_nodes"], gw["path_len"], prefix)
    assert np.array_equal(ge, oe) and np.array_equal(g, o)
