"""CLaSp layer-selection dynamic program, written out plainly.

TEST INFRASTRUCTURE ONLY (see the package docstring): only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` call it.

Source: Pith review of "CLaSp: In-Context Layer Skip for Self-Speculative
Decoding" (arXiv 2505.24196), "What carries the argument": g(i, j) is the best
hidden state obtainable by skipping j of the first i layers, scored by cosine
similarity to the full model's hidden state h_i; the recurrence compares
keeping versus skipping layer i - 1, and a backtracking pass recovers the skip
set S*.  Referee report, minor comments 1 and 4: the transition is
D(i, j) = max{cos(h_i, g(i-1, j-1)), cos(h_i, f_{i-1}(g(i-1, j)))}, and the
paper's backtracking compares state vectors instead of storing decisions.

Readings (R16 in the design notes):
  * g(0, 0) = h_0; states exist for 0 <= j <= min(i, M).  At j = 0 only the
    kept branch exists, at j = i only the skipped one (g(i, i) = h_0).
  * Both branches: the one with the larger cosine wins; a tie keeps the layer.
  * Backtracking follows the stored decisions from (L, M).
  * The layer functions of the synthetic workload are residual linear maps
    f_l(x) = x + W_l x with bfloat16 weights and the product taken at full
    precision (float64 here).  Rounding x to bfloat16 before the product was
    rejected: the rounding of each layer's input is then decided by noise far
    below the bfloat16 step, and a float32 and a float64 run of the same
    skip path drift apart by about 5e-3 relative after 32 layers, so no two
    implementations would agree on the decisions.
"""

from __future__ import annotations

import numpy as np


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 -> nearest bfloat16 (ties to even), as float64
    (used to make bfloat16 weights in tests)."""
    f = np.asarray(x, np.float64).astype(np.float32)
    bits = f.view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
    return ((bits + rounding) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.dot(a, b) / (np.linalg.norm(a) * np.linalg.norm(b)))


def layer(W: np.ndarray, x: np.ndarray) -> np.ndarray:
    """f(x) = x + W x, W float64 values of bfloat16 weights [d, d] (out, in)."""
    return x + W @ x


def clasp_dp(h, Ws, M):
    """One sequence.  h float64 [L+1, d] (h_0 .. h_L), Ws list of L float64
    [d, d] matrices, M skips (0 <= M <= L).  Returns (skip mask int [L],
    D(L, M), the smallest |cos keep - cos skip| over the decisions taken on
    the path: the tie margin)."""
    L = len(Ws)
    g = {(0, 0): np.asarray(h[0], np.float64)}
    choice = {}
    gap = {}
    for i in range(1, L + 1):
        W = np.asarray(Ws[i - 1], np.float64)
        for j in range(0, min(i, M) + 1):
            cands = []
            if j <= i - 1:  # keep layer i - 1
                k = layer(W, g[(i - 1, j)])
                cands.append((cosine(h[i], k), 0, k))
            if j >= 1:      # skip layer i - 1
                s = g[(i - 1, j - 1)]
                cands.append((cosine(h[i], s), 1, s))
            if len(cands) == 2:
                (ck, _, kk), (cs, _, ss) = cands
                skip = cs > ck
                g[(i, j)] = ss if skip else kk
                choice[(i, j)] = int(skip)
                gap[(i, j)] = abs(cs - ck)
            else:
                g[(i, j)] = cands[0][2]
                choice[(i, j)] = cands[0][1]
                gap[(i, j)] = np.inf
    mask = np.zeros(L, np.int64)
    j, margin = M, np.inf
    for i in range(L, 0, -1):
        margin = min(margin, gap[(i, j)])
        if choice[(i, j)]:
            mask[i - 1] = 1
            j -= 1
    return mask, cosine(h[L], g[(L, M)]), margin


def apply_skips(h0, Ws, mask):
    """The hidden state after the full stack with the masked layers skipped."""
    x = np.asarray(h0, np.float64)
    for l, W in enumerate(Ws):
        if not mask[l]:
            x = layer(W, x)
    return x


def clasp_batch(h, Ws, M):
    """h [B, L+1, d]; Ws [L, d, d] (float values of the bf16 weights; each
    layer is taken to float64 as the DP reaches it).
    Returns mask [B, L], score [B], margin [B]."""
    B, L = h.shape[0], len(Ws)
    mask = np.zeros((B, L), np.int64)
    score = np.zeros(B)
    margin = np.zeros(B)
    for b in range(B):
        mask[b], score[b], margin[b] = clasp_dp(np.asarray(h[b], np.float64), Ws, M)
    return mask, score, margin
