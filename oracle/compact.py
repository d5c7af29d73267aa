"""Cache compaction after a tree verification, written out plainly.

TEST INFRASTRUCTURE ONLY (see the package docstring): only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` call it.

Sources (the pages):
  * "Accelerating LLM Inference with Staged Speculative Decoding"
    (arXiv 2308.04623), abstract: the speculative batch is a tree.
  * Pith review of "PipeSpec" (arXiv 2505.01572), "What carries the
    argument": after verification each buffer keeps the longest verified
    prefix and is rolled back to the last verified token.

Reading (listed in the design notes as R13): a tree verification pass
computes a cache row (the per-layer keys and values of one token, W bytes)
for every node of the tree; only the root path the verifier kept survives.
Compaction copies the kept path into the sequence's contiguous cache: the
root node's row goes to position prefix_len, the i-th kept node's row to
position prefix_len + i.  Everything else in the cache is left as it was.
A sequence the verifier marked as a data error (path_nodes[b, 0] == -1)
is skipped.  A path that names a node outside [0, N), a path length outside
[0, max_depth], or a destination outside [0, C) is malformed: the sequence
is skipped and gets error bit 2 (the bit of a malformed tree).
"""

from __future__ import annotations

import numpy as np

ERR_PATH = 2


def compact_tree_path(tree_rows, cache, path_nodes, path_len, prefix_len=None):
    """Compact every sequence's kept path; returns (new cache, error bits).

    tree_rows  uint8 [B, N, W]   one row per tree node
    cache      uint8 [B, C, W]   contiguous cache (not modified; a copy is returned)
    path_nodes int   [B, D+1]    root first, then the kept nodes, -1 padded
    path_len   int   [B]         kept nodes (the root not counted)
    prefix_len int   [B] or None tokens before the window (None: all 0)
    """
    tree_rows = np.asarray(tree_rows, np.uint8)
    out = np.array(cache, dtype=np.uint8, copy=True)
    B, N, W = tree_rows.shape
    C = out.shape[1]
    D1 = path_nodes.shape[1]
    err = np.zeros(B, np.int64)
    for b in range(B):
        if path_nodes[b, 0] < 0:  # the verifier reported a data error
            continue
        n_rows = int(path_len[b]) + 1
        base = 0 if prefix_len is None else int(prefix_len[b])
        if not 1 <= n_rows <= D1:
            err[b] = ERR_PATH
            continue
        nodes = [int(path_nodes[b, i]) for i in range(n_rows)]
        if any(not 0 <= n < N for n in nodes) or base < 0 or base + n_rows > C:
            err[b] = ERR_PATH
            continue
        for i, n in enumerate(nodes):
            out[b, base + i, :] = tree_rows[b, n, :]
    return out, err
