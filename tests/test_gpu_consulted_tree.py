"""Consulted-only tree verification on the GPU against oracle/consulted_tree.py.

The walk computes the statistics of a node's rows only when it stands at the
node, so a NaN planted in the rows of a node off the walked path must not
flag the sequence, while one in a walked node's rows must.  Decisions,
paths, tokens and rollbacks must equal the oracle's (near ties set aside as
in tests/gpu_helpers.py) and the ordinary mode's.
"""

import numpy as np
import pytest

from oracle import consulted_tree as CT
from oracle import verify as V
from workloads import synth

from . import gpu_helpers as H

pytestmark = pytest.mark.gpu

S = synth.SPECS
W = synth.with_sizes


def oracle(w, greedy=None):
    s = w["spec"]
    greedy = s.greedy if greedy is None else greedy
    return CT.verify_tree_consulted(w["parent"], w["tokens"], w["target"], w["draft"], w["u"], w["v"],
                                    w["prefix_len"], s.temperature, greedy, w["max_depth"], s.dtype, V=s.V)


CASES = [
    W(S["tree_b16_n64_v50257_bf16"], name="tree_v3001_n64", B=6, V=3001),
    W(S["tree_b16_n64_v50257_bf16"], name="tree_v12289_n20_pad1", B=5, V=12289, n_nodes=20, pad=1,
      branching=(3, 3, 2, 2)),
    W(S["tree_b16_n64_v50257_bf16"], name="tree_f32_v999_n40", B=4, V=999, dtype="f32", n_nodes=40),
    W(S["tree_b16_n64_v50257_bf16"], name="tree_v70000_streamed", B=3, V=70000),
    W(S["tree_b16_n64_v50257_bf16"], name="tree_greedy_v20000", B=6, V=20000, greedy=True),
    W(S["tree_b16_n64_v50257_bf16"], name="tree_greedy_v300001_direct", B=2, V=300001, greedy=True, pad=3),
]


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_tree_consulted_small(cuda_device, spec):
    w = synth.make(spec, seed=16)
    g = H.gpu_tree(w, cuda_device, consulted_only=True)
    o = oracle(w)
    flagged = H.compare_tree(g, o, spec.greedy)
    d = H.gpu_tree(w, cuda_device)  # the ordinary mode, same inputs
    keep = ~flagged
    for k in ("path_len", "out_token", "rollback_idx", "seq_error"):
        assert np.array_equal(g[k][keep], d[k][keep]), k


def test_tree_consulted_full_size(cuda_device):
    spec = S["tree_b16_n64_v50257_bf16"]
    w = synth.make(spec, seed=0)
    o = oracle(w)
    H.compare_tree(H.gpu_tree(w, cuda_device, consulted_only=True), o, False)
    # the walk reads the rows of a few nodes of the 64: the oracle counts them
    assert o["rows_read"].mean() < 0.2 * 2 * 64
    H.compare_tree(H.gpu_tree(w, cuda_device, greedy=True, consulted_only=True), oracle(w, greedy=True), True)


def test_tree_consulted_nonfinite_only_when_read(cuda_device):
    spec = W(S["tree_b16_n64_v50257_bf16"], B=8, V=4000)
    w = synth.make(spec, seed=17)
    o0 = V.verify_tree(w["parent"], w["tokens"], w["target"], w["draft"], w["u"], w["v"], w["prefix_len"],
                       spec.temperature, False, w["max_depth"], spec.dtype, V=spec.V)
    nan = synth.bf16_from_float32(np.array([np.nan], np.float32))[0]
    N = w["parent"].shape[1]
    for b in range(spec.B):
        path = [int(x) for x in o0["path_nodes"][b] if x >= 0]
        off = [n for n in range(N) if n not in path]
        if b % 2 == 0:
            w["target"][b, off[-1], 11] = nan       # a node the walk never stands at
            w["draft"][b, off[-2], 5] = nan
        else:
            w["target"][b, path[-1], 2] = nan       # the last node of the walk
    g = H.gpu_tree(w, cuda_device, consulted_only=True)
    o = oracle(w)
    H.compare_tree(g, o, False)
    assert (g["seq_error"][0::2] & V.ERR_NONFINITE == 0).all()
    assert (g["seq_error"][1::2] & V.ERR_NONFINITE != 0).all()
