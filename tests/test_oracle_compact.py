"""The compaction oracle against what fixes it independently (no GPU).

Pins:
  * structure: every node row carries its own (sequence, node) identity; after
    compaction the identities read back from positions prefix .. prefix + L
    must form a root path of the tree (node 0 first, each node's parent the
    one before it), which is checked against the parent array, not against
    the oracle's gather;
  * a chain-shaped tree whose kept path is nodes 0..L reduces to a plain slice
    copy (NumPy slicing);
  * every byte outside the written positions is unchanged;
  * the edge cases of the reading: empty path (root only), verifier errors,
    malformed paths and destinations.
Planted mistakes (an off-by-one destination, a reversed path, a dropped
prefix, the root left out) must each fail one of the pins.
"""

import numpy as np
import pytest

from oracle import compact as K
from workloads import synth


def _identity_rows(B, N, W):
    # row (b, n) = bytes of the 16-bit numbers (b, n) repeated, so a row
    # names itself
    rows = np.zeros((B, N, W), np.uint8)
    for b in range(B):
        for n in range(N):
            word = np.array([b, n], np.uint16).view(np.uint8)
            rows[b, n] = np.resize(word, W)
    return rows


def _decode(row):
    b, n = row[:4].view(np.uint16)
    return int(b), int(n)


def _random_paths(parent, B, D, rng):
    N = len(parent)
    children = [[] for _ in range(N)]
    for n in range(1, N):
        children[parent[n]].append(n)
    nodes = -np.ones((B, D + 1), np.int32)
    plen = np.zeros(B, np.int32)
    for b in range(B):
        node, path = 0, [0]
        want = int(rng.integers(0, D + 1))
        while len(path) <= want and children[node]:
            node = int(rng.choice(children[node]))
            path.append(node)
        nodes[b, :len(path)] = path
        plen[b] = len(path) - 1
    return nodes, plen


def _case(seed=0, B=12, W=40, D=6):
    rng = np.random.default_rng(seed)
    parent = synth.tree_topology()
    N = len(parent)
    rows = _identity_rows(B, N, W)
    nodes, plen = _random_paths(parent, B, D, rng)
    prefix = rng.integers(0, 20, B).astype(np.int32)
    C = int(prefix.max()) + D + 3
    cache = rng.integers(0, 256, (B, C, W), dtype=np.uint8)
    return parent, rows, cache, nodes, plen, prefix


def pin_structure(fn):
    parent, rows, cache, nodes, plen, prefix = _case()
    out, err = fn(rows, cache, nodes, plen, prefix)
    assert (err == 0).all()
    for b in range(rows.shape[0]):
        ids = [_decode(out[b, prefix[b] + i]) for i in range(plen[b] + 1)]
        assert all(sb == b for sb, _ in ids)
        path = [n for _, n in ids]
        assert path[0] == 0
        assert all(parent[path[i]] == path[i - 1] for i in range(1, len(path)))
        assert len(path) == plen[b] + 1


def pin_untouched(fn):
    _, rows, cache, nodes, plen, prefix = _case(seed=1)
    out, _ = fn(rows, cache, nodes, plen, prefix)
    for b in range(rows.shape[0]):
        keep = np.ones(cache.shape[1], bool)
        keep[prefix[b]:prefix[b] + plen[b] + 1] = False
        assert np.array_equal(out[b, keep], cache[b, keep])


def pin_chain_is_slice(fn):
    rng = np.random.default_rng(2)
    B, N, W, D = 5, 9, 24, 8
    rows = rng.integers(0, 256, (B, N, W), dtype=np.uint8)
    plen = rng.integers(0, D + 1, B).astype(np.int32)
    nodes = -np.ones((B, D + 1), np.int32)
    for b in range(B):
        nodes[b, :plen[b] + 1] = np.arange(plen[b] + 1)
    prefix = rng.integers(0, 7, B).astype(np.int32)
    cache = rng.integers(0, 256, (B, 20, W), dtype=np.uint8)
    out, err = fn(rows, cache, nodes, plen, prefix)
    assert (err == 0).all()
    for b in range(B):
        L = plen[b] + 1
        assert np.array_equal(out[b, prefix[b]:prefix[b] + L], rows[b, :L])


def pin_edge_cases(fn):
    _, rows, cache, nodes, plen, prefix = _case(seed=3, B=6)
    nodes, plen, prefix = nodes.copy(), plen.copy(), prefix.copy()
    nodes[0, :] = -1                      # the verifier flagged a data error
    plen[0] = 0
    nodes[1, :] = -1                      # root only: one row
    nodes[1, 0] = 0
    plen[1] = 0
    nodes[2, 1] = rows.shape[1]           # a node outside the tree
    plen[2] = max(plen[2], 1)
    prefix[3] = cache.shape[1] - plen[3]  # one row past the end of the cache
    plen[4] = nodes.shape[1]              # longer than max_depth
    out, err = fn(rows, cache, nodes, plen, prefix)
    assert list(err) == [0, 0, K.ERR_PATH, K.ERR_PATH, K.ERR_PATH, 0]
    for b in (0, 2, 3, 4):
        assert np.array_equal(out[b], cache[b])
    assert np.array_equal(out[1, prefix[1]], rows[1, 0])
    assert np.array_equal(np.delete(out[1], prefix[1], 0), np.delete(cache[1], prefix[1], 0))


PINS = [pin_structure, pin_untouched, pin_chain_is_slice, pin_edge_cases]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(K.compact_tree_path)


def _mutant(shift=0, reverse=False, no_prefix=False, skip_root=False):
    def fn(rows, cache, nodes, plen, prefix):
        out = cache.copy()
        err = np.zeros(rows.shape[0], np.int64)
        for b in range(rows.shape[0]):
            if nodes[b, 0] < 0:
                continue
            L = int(plen[b]) + 1
            if L > nodes.shape[1] or prefix[b] + L > cache.shape[1] or (nodes[b, :L] >= rows.shape[1]).any():
                err[b] = K.ERR_PATH
                continue
            path = list(nodes[b, :L])
            if reverse:
                path = path[::-1]
            if skip_root:
                path = path[1:]
            base = 0 if no_prefix else int(prefix[b])
            for i, n in enumerate(path):
                d = base + i + shift
                if d < cache.shape[1]:
                    out[b, d] = rows[b, n]
        return out, err
    return fn


@pytest.mark.parametrize("mutant", [dict(shift=1), dict(reverse=True), dict(no_prefix=True), dict(skip_root=True)],
                         ids=lambda m: next(iter(m)))
def test_planted_mistake_is_caught(mutant):
    fn = _mutant(**mutant)
    caught = False
    for pin in PINS:
        try:
            pin(fn)
        except AssertionError:
            caught = True
            break
    assert caught
