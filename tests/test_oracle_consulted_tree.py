"""The consulted-rows tree oracle against the ordinary tree oracle (no GPU).

Pins:
  * on finite inputs the path, token, rollback, error bits and margins equal
    the ordinary rule's (oracle.verify, pinned in tests/pins.py), in sampling
    and greedy mode;
  * rows_read equals a count made from the ordinary rule's path and the
    tree's structure: one target row per visited node (the root and the kept
    nodes), plus, in sampling mode, one draft row per visited node that has
    children;
  * a non-finite row is an error exactly when it is consulted: rows of nodes
    off the path never are, and neither is the draft row of the leaf a walk
    ends on.
Planted mistakes (errors raised for rows off the path, a leaf's draft row
counted) must fail a pin.
"""

import numpy as np
import pytest

from oracle import consulted_tree as Ct
from oracle import verify as V
from workloads import synth

TREE = synth.SPECS["tree_b16_n64_v50257_bf16"]


def _case(seed, greedy=False, B=12, V_=700):
    spec = synth.with_sizes(TREE, B=B, V=V_, greedy=greedy)
    return spec, synth.make(spec, seed=seed)


def _ordinary(spec, w):
    return V.verify_tree(w["parent"], w["tokens"], w["target"], w["draft"], w["u"], w["v"], w["prefix_len"],
                         spec.temperature, spec.greedy, w["max_depth"], spec.dtype, V=spec.V)


def _run(fn, spec, w):
    return fn(w["parent"], w["tokens"], w["target"], w["draft"], w["u"], w["v"], w["prefix_len"],
              spec.temperature, spec.greedy, w["max_depth"], spec.dtype, V=spec.V)


def pin_equal_on_finite(fn):
    for seed in range(3):
        for greedy in (False, True):
            spec, w = _case(seed, greedy)
            o = _ordinary(spec, w)
            c = _run(fn, spec, w)
            for k in ("path_len", "path_nodes", "out_token", "rollback_idx", "error"):
                assert np.array_equal(c[k], o[k]), (k, seed, greedy)
            if not greedy:
                assert np.array_equal(c["margin_u"], o["margin_u"]) and np.array_equal(c["margin_v"], o["margin_v"])
            parent = w["parent"][0]
            has_kids = np.zeros(len(parent), bool)
            has_kids[parent[1:]] = True
            for b in range(spec.B):
                visited = o["path_nodes"][b][o["path_nodes"][b] >= 0]
                want = len(visited) + (0 if greedy else int(has_kids[visited].sum()))
                assert c["rows_read"][b] == want, (b, c["rows_read"][b], want)


def pin_nonfinite_only_when_consulted(fn):
    spec, w = _case(5, B=8)
    # equal target and draft rows: every ratio is 1, so the walk keeps a
    # child at every level and ends on a leaf (the case-2 sequences)
    for b in range(2, spec.B, 4):
        w["target"][b] = w["draft"][b]
    o = _ordinary(spec, w)
    parent = w["parent"][0]
    N = len(parent)
    has_kids = np.zeros(N, bool)
    has_kids[parent[1:]] = True
    nan = synth.bf16_from_float32(np.array([np.nan], np.float32))[0]
    expect = np.zeros(spec.B, np.int64)
    for b in range(spec.B):
        visited = [int(n) for n in o["path_nodes"][b] if n >= 0]
        off = [n for n in range(N) if n not in visited]
        last = visited[-1]
        case = b % 4
        if case == 0 and off:                      # a node off the path: never read
            w["target"][b, off[-1], 3] = nan
            w["draft"][b, off[0], 5] = nan
        elif case == 1:                            # a visited node's target row
            w["target"][b, visited[0], 2] = nan
            expect[b] = V.ERR_NONFINITE
        elif case == 2:                            # the leaf the walk ends on: its draft row is not needed
            assert not has_kids[last]
            w["draft"][b, last, 1] = nan
        elif case == 3 and has_kids[visited[0]]:   # a visited internal node's draft row
            w["draft"][b, visited[0], 4] = nan
            expect[b] = V.ERR_NONFINITE
    c = _run(fn, spec, w)
    assert np.array_equal(c["error"] & V.ERR_NONFINITE, expect), (c["error"], expect)
    ok = expect == 0
    assert np.array_equal(c["path_nodes"][ok], o["path_nodes"][ok])
    assert np.array_equal(c["out_token"][ok], o["out_token"][ok])


PINS = [pin_equal_on_finite, pin_nonfinite_only_when_consulted]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(Ct.verify_tree_consulted)


def _flag_everything(*args, **kw):
    r = Ct.verify_tree_consulted(*args, **kw)
    target, draft, dtype, V_ = args[2], args[3], args[10], kw.get("V")
    for b in range(target.shape[0]):
        rows = [V.row_to_float64(target[b, i, :V_], dtype) for i in range(target.shape[1])]
        rows += [V.row_to_float64(draft[b, i, :V_], dtype) for i in range(draft.shape[1])]
        if any(V.row_is_nonfinite(x) for x in rows):
            r["error"][b] |= V.ERR_NONFINITE
    return r


def _leaf_draft_counted(*args, **kw):
    r = Ct.verify_tree_consulted(*args, **kw)
    parent = args[0][0]
    has_kids = np.zeros(len(parent), bool)
    has_kids[parent[1:]] = True
    for b in range(len(r["rows_read"])):
        nodes = r["path_nodes"][b][r["path_nodes"][b] >= 0]
        if len(nodes) and not has_kids[nodes[-1]] and not args[8]:
            r["rows_read"][b] += 1
    return r


@pytest.mark.parametrize("mutant", [_flag_everything, _leaf_draft_counted], ids=lambda m: m.__name__)
def test_planted_mistake_is_caught(mutant):
    caught = False
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught = True
            break
    assert caught
