"""Seeded synthetic workloads for batched draft verification.

Shapes follow the five workloads the verification step is measured on:

  greedy chain      B=4,   gamma=4,  V=1000,   float32, temperature ignored
  sampling chain    B=32,  gamma=8,  V=32000,  bfloat16, T=1.0, alpha ~ 0.7
  sampling chain    B=64,  gamma=5,  V=128256, bfloat16, T=0.7,
                    alpha in {0.05, 0.3, 0.6, 0.9}
  tree              B=16,  64 nodes (depth 6, branching 4/3/2/2/1/1),
                    V=50257, bfloat16, T=1.0, alpha ~ 0.7
  cascade           B=128, gamma1=8, gamma2=4, V=128256, bfloat16, T=1.0,
                    alpha(M0,M1) ~ 0.8, alpha(M1,M2) ~ 0.6

The vocabulary sizes stand in for the LLaMA-2 (32000), LLaMA-3 (128256) and
GPT-2 (50257) families the pages use; the pages' datasets are not needed
because the verification step consumes logits only.

Logit model: draft logits Q ~ N(0, sigma_q^2); target logits
P = a * Q + N(0, s^2).  Values are rounded to the stored dtype before anything
reads them.  Drafted tokens are drawn from the draft softmax at the workload's
temperature with the Gumbel-max trick (argmax of Q/T plus Gumbel noise), so
that drafts follow q as speculative sampling assumes; the greedy workload
drafts the draft argmax instead.  The noise scales were chosen by bisection on
seeded calibration batches (tests/golden/make_calibration.py, which records
the achieved mean acceptance next to each value) so that the mean acceptance
sum_x min(p, q) lands near the stated alpha.

Everything is NumPy on the host; callers move arrays to the device.
"""

from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np


# --------------------------------------------------------------------------
# bfloat16 storage
# --------------------------------------------------------------------------

def bf16_from_float32(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even.

    Inputs here are finite, so no NaN special case is needed.
    """
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
    return ((bits + rounding) >> np.uint32(16)).astype(np.uint16)


def float32_from_bf16(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 values (exact)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_from_float32(x) if dtype == "bf16" else np.ascontiguousarray(x, np.float32)


def _values(stored: np.ndarray, dtype: str) -> np.ndarray:
    return float32_from_bf16(stored) if dtype == "bf16" else stored


def _gumbel_argmax(rng: np.random.Generator, scaled: np.ndarray) -> np.ndarray:
    """argmax over the last axis of scaled + Gumbel(0, 1) noise."""
    uni = rng.random(scaled.shape, dtype=np.float32)
    with np.errstate(divide="ignore"):
        g = -np.log(-np.log(uni))
    return np.argmax(scaled + g, axis=-1)


# --------------------------------------------------------------------------
# specs
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class ChainSpec:
    name: str
    B: int
    gamma: int
    V: int
    dtype: str            # "f32" | "bf16"
    greedy: bool
    temperature: float
    sigma_q: float        # draft logit scale
    a: float              # target = a * draft + noise
    s: float              # target noise scale
    alpha_target: float | None = None
    pad: int = 0          # row stride = V + pad elements


@dataclass(frozen=True)
class TreeSpec:
    name: str
    B: int
    V: int
    dtype: str
    greedy: bool
    temperature: float
    sigma_q: float
    a: float
    s: float
    branching: tuple = (4, 3, 2, 2, 1, 1)
    n_nodes: int = 64
    alpha_target: float | None = None
    pad: int = 0


@dataclass(frozen=True)
class CascadeSpec:
    name: str
    B: int
    gamma1: int
    gamma2: int
    V: int
    dtype: str
    greedy: bool
    temperature: float
    sigma_q: float
    a01: float
    s01: float
    a12: float
    s12: float
    alpha01_target: float | None = None
    alpha12_target: float | None = None
    pad: int = 0


# Calibrated noise scales: see tests/golden/calibration.json for the achieved
# mean acceptance of each value.
SPECS = {
    "greedy_chain_b4_g4_v1000_f32": ChainSpec(
        "greedy_chain_b4_g4_v1000_f32", B=4, gamma=4, V=1000, dtype="f32",
        greedy=True, temperature=1.0, sigma_q=2.0, a=1.0, s=0.5),
    "sampling_chain_b32_g8_v32000_bf16": ChainSpec(
        "sampling_chain_b32_g8_v32000_bf16", B=32, gamma=8, V=32000,
        dtype="bf16", greedy=False, temperature=1.0, sigma_q=2.0, a=0.9,
        s=0.748, alpha_target=0.7),
    "sampling_chain_b64_g5_v128256_bf16_a05": ChainSpec(
        "sampling_chain_b64_g5_v128256_bf16_a05", B=64, gamma=5, V=128256,
        dtype="bf16", greedy=False, temperature=0.7, sigma_q=2.0, a=0.0535,
        s=1.9971, alpha_target=0.05),
    "sampling_chain_b64_g5_v128256_bf16_a30": ChainSpec(
        "sampling_chain_b64_g5_v128256_bf16_a30", B=64, gamma=5, V=128256,
        dtype="bf16", greedy=False, temperature=0.7, sigma_q=2.0, a=0.7402,
        s=1.3448, alpha_target=0.3),
    "sampling_chain_b64_g5_v128256_bf16_a60": ChainSpec(
        "sampling_chain_b64_g5_v128256_bf16_a60", B=64, gamma=5, V=128256,
        dtype="bf16", greedy=False, temperature=0.7, sigma_q=2.0, a=0.9331,
        s=0.7192, alpha_target=0.6),
    "sampling_chain_b64_g5_v128256_bf16_a90": ChainSpec(
        "sampling_chain_b64_g5_v128256_bf16_a90", B=64, gamma=5, V=128256,
        dtype="bf16", greedy=False, temperature=0.7, sigma_q=2.0, a=0.996,
        s=0.1787, alpha_target=0.9),
    "tree_b16_n64_v50257_bf16": TreeSpec(
        "tree_b16_n64_v50257_bf16", B=16, V=50257, dtype="bf16", greedy=False,
        temperature=1.0, sigma_q=2.0, a=0.9, s=0.75, alpha_target=0.7),
    "cascade_b128_g8_g4_v128256_bf16": CascadeSpec(
        "cascade_b128_g8_g4_v128256_bf16", B=128, gamma1=8, gamma2=4,
        V=128256, dtype="bf16", greedy=False, temperature=1.0, sigma_q=2.0,
        a01=0.9, s01=0.465, a12=0.9, s12=1.024, alpha01_target=0.8,
        alpha12_target=0.6),
}


@dataclass(frozen=True)
class PipelineSpec:
    """k-model PipeSpec snapshot: windows[s-1] is stage s's window (windows[0]
    = drafted tokens).  Logits: M_0 ~ sigma_q N(0, 1); M_s = a[s-1] M_{s-1} +
    s[s-1] N(0, 1) row by row (the cascade's model, one more link per stage)."""
    name: str
    B: int
    windows: tuple
    V: int
    dtype: str
    greedy: bool
    temperature: float
    sigma_q: float
    a: tuple
    s: tuple
    final_bonus: bool = False
    pad: int = 0

    @property
    def k(self) -> int:
        return len(self.windows) + 1


# Four models (M_0 -> M_1 -> M_2 -> M_3): the cascade's first two links, and
# a third with the second link's scales.
PIPELINE_SPECS = {
    "pipeline4_b128_g8_g6_g4_v128256_bf16": PipelineSpec(
        "pipeline4_b128_g8_g6_g4_v128256_bf16", B=128, windows=(8, 6, 4), V=128256, dtype="bf16", greedy=False,
        temperature=1.0, sigma_q=2.0, a=(0.9, 0.9, 0.9), s=(0.465, 1.024, 1.024)),
}


@dataclass(frozen=True)
class PipelineAsyncSpec:
    """PipeSpec stages at independent buffer offsets: stage s verifies w_s =
    windows[s-1] tokens of O_{s-1} after the l_s tokens O_s already holds.
    Buffer lengths: l_{k-1} uniform in [0, max_base), l_{s-1} = l_s + w_s +
    a gap uniform in [0, extra] (a gap of 0: the window ends the buffer
    below).  Per stage and sequence: M_{s-1} rows Q ~ sigma_q N(0, 1) at the
    window's positions and the one after, M_s rows a[s-1] Q + s[s-1] N(0, 1)
    (the pipeline's model), the window tokens drawn from M_{s-1}'s softmax
    at the temperature (greedy: its argmax); the windows of different stages
    cover disjoint positions, so they are drawn independently."""
    name: str
    B: int
    windows: tuple
    V: int
    dtype: str = "bf16"
    greedy: bool = False
    temperature: float = 1.0
    sigma_q: float = 2.0
    a: tuple = (0.9, 0.9, 0.9)
    s: tuple = (0.465, 1.024, 1.024)
    final_bonus: bool = False
    extra: int = 2
    max_base: int = 64
    pad: int = 0

    @property
    def k(self) -> int:
        return len(self.windows) + 1


PIPELINE_ASYNC_SPECS = {
    "pipeline4_async_b128_g8_g6_g4_v128256_bf16": PipelineAsyncSpec(
        "pipeline4_async_b128_g8_g6_g4_v128256_bf16", B=128, windows=(8, 6, 4), V=128256),
}


@dataclass(frozen=True)
class CompactSpec:
    """Cache compaction after a tree verification: B sequences, each with one
    row of row_bytes per tree node (the tree of tree_topology) and a kept root
    path drawn by walking from the root, keeping a random child with
    probability `keep` at each level (at most max_depth kept nodes)."""
    name: str
    B: int
    row_bytes: int
    max_depth: int = 6
    keep: float = 0.7
    max_prefix: int = 64
    branching: tuple = (4, 3, 2, 2, 1, 1)
    n_nodes: int = 64
    pad: int = 0          # row stride = row_bytes + pad bytes


# Row size: the keys and values of one token in every layer of a 32-layer
# model with 8 key-value heads of dimension 128 in bfloat16
# (2 x 32 x 8 x 128 x 2 B = 131072 B).
COMPACT_SPECS = {
    "tree_kv_compact_b16_n64_d6_w131072": CompactSpec("tree_kv_compact_b16_n64_d6_w131072", B=16, row_bytes=131072),
}


@dataclass(frozen=True)
class ClaspSpec:
    """CLaSp layer selection: B sequences, an L-layer stack of width d whose
    layers are residual linear maps with bfloat16 weights W_l ~ N(0, scale^2
    / d), and M layers to skip.  The full model's hidden states h_0 .. h_L
    come from h_0 ~ N(0, 1) and h_{l+1} = h_l + W_l h_l + N(0, tau^2) in
    float64 (unrounded inputs plus per-layer noise: the full model is not
    exactly the stack the draft's layers compute), stored as float32."""
    name: str
    B: int
    L: int
    d: int
    M: int
    scale: float = 0.3
    tau: float = 0.1


# LLaMA-3-8B's depth and width (32 layers, d = 4096) with 12 of 32 layers
# skipped, the setting of the CLaSp page's DP versus brute-force comparison.
CLASP_SPECS = {
    "clasp_b16_l32_d4096_m12_bf16": ClaspSpec("clasp_b16_l32_d4096_m12_bf16", B=16, L=32, d=4096, M=12),
}


@dataclass(frozen=True)
class LmHeadSpec:
    """Chain verification from final hidden states and LM-head weights (the
    LM head folded into the verification).  Target head W_t [V, d_t] ~
    N(0, sigma_logit^2 / d_t) rounded to bfloat16, target hidden states
    h_t ~ N(0, 1) rounded to bfloat16, so target logits have standard
    deviation about sigma_logit.  The draft reads the first d_d hidden
    coordinates: W_d = bf16(W_t[:, :d_d] * sqrt(d_t / d_d)) (W_d = W_t when
    d_d = d_t: one shared head, as in self-speculative decoding) and
    h_d = bf16(h_t[:, :gamma, :d_d] + s N(0, 1)), so draft logits are the
    target's plus noise of scale about s * sigma_logit; s is chosen for the
    named mean acceptance.  Drafted tokens are drawn from the draft softmax
    with the Gumbel-max trick (its argmax in greedy mode)."""
    name: str
    B: int
    gamma: int
    V: int
    d_target: int
    d_draft: int
    greedy: bool
    temperature: float
    sigma_logit: float = 2.0
    s: float = 0.35
    alpha_target: float | None = None


# The 128256-vocabulary sampling chain's verification shape (B = 64,
# gamma = 5, T = 0.7) with the LM head that produces its logits: LLaMA-3-8B's
# width d = 4096, one head shared by target and draft.
LM_HEAD_SPECS = {
    "lm_head_chain_b64_g5_v128256_d4096_bf16": LmHeadSpec(
        "lm_head_chain_b64_g5_v128256_d4096_bf16", B=64, gamma=5, V=128256, d_target=4096, d_draft=4096,
        greedy=False, temperature=0.7, alpha_target=0.6),
}


def with_sizes(spec, **kw):
    """A copy of a spec with some fields replaced (e.g. a smaller B or V)."""
    return dataclasses.replace(spec, **kw)


# --------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------

def _rng(seed: int, salt: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(salt)])


def _pad(x: np.ndarray, pad: int) -> np.ndarray:
    if pad == 0:
        return x
    width = list(x.shape)
    width[-1] += pad
    out = np.zeros(width, dtype=x.dtype)
    out[..., : x.shape[-1]] = x
    return out


def make_chain(spec: ChainSpec, seed: int = 0) -> dict:
    """Chain workload: target [B, gamma+1, V+pad], draft [B, gamma, V+pad],
    tokens int32 [B, gamma], u float32 [B, gamma], v float32 [B],
    prefix_len int32 [B]."""
    rng = _rng(seed, 1)
    B, g, V = spec.B, spec.gamma, spec.V
    target = np.empty((B, g + 1, V), np.uint16 if spec.dtype == "bf16" else np.float32)
    draft = np.empty((B, g, V), target.dtype)
    tokens = np.empty((B, g), np.int32)
    for b in range(B):  # one sequence at a time keeps the float32 temporaries small
        q = rng.standard_normal((g + 1, V), dtype=np.float32) * np.float32(spec.sigma_q)
        p = np.float32(spec.a) * q + rng.standard_normal((g + 1, V), dtype=np.float32) * np.float32(spec.s)
        qs = _store(q[:g], spec.dtype)
        draft[b] = qs
        target[b] = _store(p, spec.dtype)
        qv = _values(qs, spec.dtype)
        if spec.greedy:
            tokens[b] = np.argmax(qv, axis=-1)
        else:
            tokens[b] = _gumbel_argmax(rng, qv / np.float32(spec.temperature))
    u = rng.random((B, g), dtype=np.float32)
    v = rng.random(B, dtype=np.float32)
    prefix = rng.integers(0, 4096, B, dtype=np.int32)
    return dict(kind="chain", spec=spec, target=_pad(target, spec.pad),
                draft=_pad(draft, spec.pad), tokens=tokens, u=u, v=v,
                prefix_len=prefix)


def tree_topology(branching=(4, 3, 2, 2, 1, 1), n_nodes=64) -> np.ndarray:
    """Parent array of the draft tree used by the tree workload.

    The full tree with the given per-depth branching is enumerated as paths of
    0-based sibling ranks; the n_nodes paths with the smallest key
    (sum of ranks, depth, path) are kept and numbered in key order, so that
    parent[i] < i and the kept set is closed under parents.  For the default
    arguments the kept nodes per depth are 1/4/9/11/13/13/13.
    """
    paths = [()]
    frontier = [()]
    for width in branching:
        frontier = [p + (r,) for p in frontier for r in range(width)]
        paths.extend(frontier)
    paths.sort(key=lambda p: (sum(p), len(p), p))
    kept = paths[:n_nodes]
    index = {p: i for i, p in enumerate(kept)}
    parent = np.array([-1] + [index[p[:-1]] for p in kept[1:]], dtype=np.int32)
    return parent


def make_tree(spec: TreeSpec, seed: int = 0) -> dict:
    """Tree workload: parent int32 [B, N], tokens int32 [B, N] (tokens[:, 0]
    unused), target / draft [B, N, V+pad], u float32 [B, N], v float32 [B],
    prefix_len int32 [B].  Each child's token is drawn from the draft softmax
    of its parent's row, independently of its siblings (with replacement)."""
    rng = _rng(seed, 2)
    B, V = spec.B, spec.V
    parent1 = tree_topology(spec.branching, spec.n_nodes)
    N = len(parent1)
    parent = np.tile(parent1, (B, 1))
    dt = np.uint16 if spec.dtype == "bf16" else np.float32
    target = np.empty((B, N, V), dt)
    draft = np.empty((B, N, V), dt)
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        q = rng.standard_normal((N, V), dtype=np.float32) * np.float32(spec.sigma_q)
        p = np.float32(spec.a) * q + rng.standard_normal((N, V), dtype=np.float32) * np.float32(spec.s)
        qs = _store(q, spec.dtype)
        draft[b] = qs
        target[b] = _store(p, spec.dtype)
        qv = _values(qs, spec.dtype) / np.float32(spec.temperature)
        if spec.greedy:
            tokens[b, 1:] = np.argmax(qv[parent1[1:]], axis=-1)
        else:
            tokens[b, 1:] = _gumbel_argmax(rng, qv[parent1[1:]])
    u = rng.random((B, N), dtype=np.float32)
    v = rng.random(B, dtype=np.float32)
    prefix = rng.integers(0, 4096, B, dtype=np.int32)
    depth = np.zeros(N, np.int64)
    for i in range(1, N):
        depth[i] = depth[parent1[i]] + 1
    return dict(kind="tree", spec=spec, parent=parent, tokens=tokens,
                target=_pad(target, spec.pad), draft=_pad(draft, spec.pad),
                u=u, v=v, prefix_len=prefix, max_depth=int(depth.max()))


def make_cascade(spec: CascadeSpec, seed: int = 0) -> dict:
    """Cascade workload: l0 [B, g1, V+pad] (M_0), l1 [B, g1+1, V+pad] (M_1),
    l2 [B, g2, V+pad] (M_2), tokens int32 [B, g1] drawn from M_0, u1 [B, g1],
    v1 [B], u2 [B, g2], v2 [B], base0 = base1 int32 [B]."""
    rng = _rng(seed, 3)
    B, g1, g2, V = spec.B, spec.gamma1, spec.gamma2, spec.V
    dt = np.uint16 if spec.dtype == "bf16" else np.float32
    l0 = np.empty((B, g1, V), dt)
    l1 = np.empty((B, g1 + 1, V), dt)
    l2 = np.empty((B, g2, V), dt)
    tokens = np.empty((B, g1), np.int32)
    for b in range(B):
        m0 = rng.standard_normal((g1 + 1, V), dtype=np.float32) * np.float32(spec.sigma_q)
        m1 = np.float32(spec.a01) * m0 + rng.standard_normal((g1 + 1, V), dtype=np.float32) * np.float32(spec.s01)
        m2 = np.float32(spec.a12) * m1[:g2] + rng.standard_normal((g2, V), dtype=np.float32) * np.float32(spec.s12)
        s0 = _store(m0[:g1], spec.dtype)
        l0[b] = s0
        l1[b] = _store(m1, spec.dtype)
        l2[b] = _store(m2, spec.dtype)
        v0 = _values(s0, spec.dtype)
        if spec.greedy:
            tokens[b] = np.argmax(v0, axis=-1)
        else:
            tokens[b] = _gumbel_argmax(rng, v0 / np.float32(spec.temperature))
    u1 = rng.random((B, g1), dtype=np.float32)
    v1 = rng.random(B, dtype=np.float32)
    u2 = rng.random((B, g2), dtype=np.float32)
    v2 = rng.random(B, dtype=np.float32)
    base = rng.integers(0, 4096, B, dtype=np.int32)
    return dict(kind="cascade", spec=spec, l0=_pad(l0, spec.pad),
                l1=_pad(l1, spec.pad), l2=_pad(l2, spec.pad), tokens=tokens,
                u1=u1, v1=v1, u2=u2, v2=v2, base0=base.copy(), base1=base.copy())


def make_compact(spec: CompactSpec, seed: int = 0) -> dict:
    """Compaction workload: tree_rows uint8 [B, N, W+pad], cache uint8
    [B, C, W+pad] with C = max_prefix + max_depth + 1 (random bytes),
    path_nodes int32 [B, max_depth+1] (root first, -1 padded), path_len int32
    [B], prefix_len int32 [B] in [0, max_prefix), parent int32 [N]."""
    rng = _rng(seed, 7)
    parent = tree_topology(spec.branching, spec.n_nodes)
    N, B, D = len(parent), spec.B, spec.max_depth
    children = [[] for _ in range(N)]
    for n in range(1, N):
        children[parent[n]].append(n)
    path_nodes = -np.ones((B, D + 1), np.int32)
    path_len = np.zeros(B, np.int32)
    for b in range(B):
        node, path = 0, [0]
        while len(path) <= D and children[node] and rng.random() < spec.keep:
            node = int(children[node][rng.integers(0, len(children[node]))])
            path.append(node)
        path_nodes[b, :len(path)] = path
        path_len[b] = len(path) - 1
    prefix_len = rng.integers(0, spec.max_prefix, B).astype(np.int32)
    C = spec.max_prefix + D + 1
    width = spec.row_bytes + spec.pad
    tree_rows = rng.integers(0, 256, (B, N, width), dtype=np.uint8)
    cache = rng.integers(0, 256, (B, C, width), dtype=np.uint8)
    return dict(kind="compact", spec=spec, tree_rows=tree_rows, cache=cache, path_nodes=path_nodes,
                path_len=path_len, prefix_len=prefix_len, parent=parent)


def make_clasp(spec: ClaspSpec, seed: int = 0) -> dict:
    """CLaSp workload: weights uint16 [L, d, d] (bfloat16 bits of W_l[out][in]),
    hidden float32 [B, L+1, d] (h_0 .. h_L of the full model)."""
    rng = _rng(seed, 9)
    B, L, d = spec.B, spec.L, spec.d
    weights = np.empty((L, d, d), np.uint16)
    sd = np.float32(spec.scale / np.sqrt(d))
    for l in range(L):
        weights[l] = bf16_from_float32(rng.standard_normal((d, d), dtype=np.float32) * sd)
    hidden = np.empty((B, L + 1, d), np.float32)
    x = rng.standard_normal((B, d))
    hidden[:, 0] = x
    for l in range(L):
        Wl = float32_from_bf16(weights[l]).astype(np.float64)
        x = x + x @ Wl.T + spec.tau * rng.standard_normal((B, d))
        hidden[:, l + 1] = x
    return dict(kind="clasp", spec=spec, weights=weights, hidden=hidden)


def clasp_weight_values(w: dict) -> np.ndarray:
    """The workload's weights as float32 values [L, d, d] (exact)."""
    return float32_from_bf16(w["weights"])


def pipeline_rows(spec: PipelineSpec, s: int) -> int:
    """Rows per sequence of model s."""
    g = spec.windows
    if s == 0:
        return g[0]
    if s == 1:
        return g[0] + 1
    return g[s - 1] + (1 if (spec.final_bonus and s == spec.k - 1) else 0)


def make_pipeline(spec: PipelineSpec, seed: int = 0) -> dict:
    """Pipeline workload: models = [M_0 .. M_{k-1}] logits [B, rows_s, V+pad],
    tokens int32 [B, windows[0]] drawn from M_0, us[s-1] [B, windows[s-1]],
    vs[s-1] [B], base int32 [k-1, B]."""
    rng = _rng(seed, 5)
    B, V, k = spec.B, spec.V, spec.k
    dt = np.uint16 if spec.dtype == "bf16" else np.float32
    rows = [pipeline_rows(spec, s) for s in range(k)]
    depth = max(rows)
    models = [np.empty((B, rows[s], V), dt) for s in range(k)]
    tokens = np.empty((B, spec.windows[0]), np.int32)
    for b in range(B):
        m = rng.standard_normal((depth, V), dtype=np.float32) * np.float32(spec.sigma_q)
        for s in range(k):
            if s > 0:
                m = np.float32(spec.a[s - 1]) * m + rng.standard_normal((depth, V), dtype=np.float32) * np.float32(
                    spec.s[s - 1])
            models[s][b] = _store(m[:rows[s]], spec.dtype)
        v0 = _values(models[0][b], spec.dtype)
        if spec.greedy:
            tokens[b] = np.argmax(v0, axis=-1)
        else:
            tokens[b] = _gumbel_argmax(rng, v0 / np.float32(spec.temperature))
    us = [rng.random((B, g), dtype=np.float32) for g in spec.windows]
    vs = [rng.random(B, dtype=np.float32) for _ in spec.windows]
    base = np.tile(rng.integers(0, 4096, B, dtype=np.int32), (k - 1, 1))
    return dict(kind="pipeline", spec=spec, models=[_pad(x, spec.pad) for x in models], tokens=tokens, us=us,
                vs=vs, base=base)


def make_pipeline_async(spec: PipelineAsyncSpec, seed: int = 0) -> dict:
    """Asynchronous snapshot workload: per stage targets [B, w_s + 1, V+pad]
    (M_s), drafts [B, w_s, V+pad] (M_{s-1}), tokens int32 [B, w_s], us
    float32 [B, w_s], vs float32 [B]; length int32 [k, B]."""
    rng = _rng(seed, 11)
    B, V, k = spec.B, spec.V, spec.k
    dt = np.uint16 if spec.dtype == "bf16" else np.float32
    length = np.zeros((k, B), np.int32)
    length[k - 1] = rng.integers(0, spec.max_base, B)
    for s in range(k - 1, 0, -1):
        length[s - 1] = length[s] + spec.windows[s - 1] + rng.integers(0, spec.extra + 1, B)
    targets, drafts, tokens = [], [], []
    for s in range(1, k):
        w = spec.windows[s - 1]
        tg = np.empty((B, w + 1, V), dt)
        dr = np.empty((B, w, V), dt)
        tk = np.empty((B, w), np.int32)
        for b in range(B):
            q = rng.standard_normal((w + 1, V), dtype=np.float32) * np.float32(spec.sigma_q)
            p = np.float32(spec.a[s - 1]) * q + rng.standard_normal((w + 1, V), dtype=np.float32) * np.float32(
                spec.s[s - 1])
            dr[b] = _store(q[:w], spec.dtype)
            tg[b] = _store(p, spec.dtype)
            qv = _values(dr[b], spec.dtype)
            tk[b] = np.argmax(qv, axis=-1) if spec.greedy else _gumbel_argmax(rng, qv / np.float32(spec.temperature))
        targets.append(_pad(tg, spec.pad))
        drafts.append(_pad(dr, spec.pad))
        tokens.append(tk)
    us = [rng.random((B, w), dtype=np.float32) for w in spec.windows]
    vs = [rng.random(B, dtype=np.float32) for _ in spec.windows]
    return dict(kind="pipeline_async", spec=spec, targets=targets, drafts=drafts, tokens=tokens, us=us, vs=vs,
                length=length)


def make_lm_head(spec: LmHeadSpec, seed: int = 0) -> dict:
    """LM-head workload (bfloat16 bit patterns as uint16): h_target [B,
    gamma+1, d_t], h_draft [B, gamma, d_d], w_target [V, d_t], w_draft [V,
    d_d], tokens int32 [B, gamma], u float32 [B, gamma], v float32 [B],
    prefix_len int32 [B]."""
    rng = _rng(seed, 7)
    B, g, V, dt, dd = spec.B, spec.gamma, spec.V, spec.d_target, spec.d_draft
    w_t = bf16_from_float32(rng.standard_normal((V, dt), dtype=np.float32) * np.float32(spec.sigma_logit / np.sqrt(dt)))
    h_t = bf16_from_float32(rng.standard_normal((B, g + 1, dt), dtype=np.float32))
    if dd == dt:
        w_d = w_t
    else:
        w_d = bf16_from_float32(float32_from_bf16(w_t[:, :dd]) * np.float32(np.sqrt(dt / dd)))
    noise = rng.standard_normal((B, g, dd), dtype=np.float32) * np.float32(spec.s)
    h_d = bf16_from_float32(float32_from_bf16(h_t[:, :g, :dd]) + noise)
    tokens = np.empty((B, g), np.int32)
    wd_f = float32_from_bf16(w_d)
    for b in range(B):  # the draft logits of one sequence at a time
        logits = float32_from_bf16(h_d[b]) @ wd_f.T
        if spec.greedy:
            tokens[b] = np.argmax(logits, axis=-1)
        else:
            tokens[b] = _gumbel_argmax(rng, logits / np.float32(spec.temperature))
    u = rng.random((B, g), dtype=np.float32)
    v = rng.random(B, dtype=np.float32)
    prefix = rng.integers(0, 4096, B, dtype=np.int32)
    return dict(kind="lm_head", spec=spec, h_target=h_t, h_draft=h_d, w_target=w_t, w_draft=w_d,
                tokens=tokens, u=u, v=v, prefix_len=prefix)


def make(spec, seed: int = 0) -> dict:
    if isinstance(spec, str):
        spec = {**SPECS, **COMPACT_SPECS, **PIPELINE_SPECS, **PIPELINE_ASYNC_SPECS, **CLASP_SPECS,
                **LM_HEAD_SPECS}[spec]
    if isinstance(spec, LmHeadSpec):
        return make_lm_head(spec, seed)
    if isinstance(spec, PipelineSpec):
        return make_pipeline(spec, seed)
    if isinstance(spec, PipelineAsyncSpec):
        return make_pipeline_async(spec, seed)
    if isinstance(spec, ClaspSpec):
        return make_clasp(spec, seed)
    if isinstance(spec, CompactSpec):
        return make_compact(spec, seed)
    if isinstance(spec, ChainSpec):
        return make_chain(spec, seed)
    if isinstance(spec, TreeSpec):
        return make_tree(spec, seed)
    if isinstance(spec, CascadeSpec):
        return make_cascade(spec, seed)
    raise TypeError(type(spec))


def logit_bytes(w: dict) -> int:
    """Bytes of logits handed to one verification call (rows x V x size)."""
    spec = w["spec"]
    es = 2 if spec.dtype == "bf16" else 4
    if w["kind"] == "chain":
        rows = spec.gamma + 1 + (0 if spec.greedy else spec.gamma)
    elif w["kind"] == "tree":
        rows = w["target"].shape[1] * (1 if spec.greedy else 2)
    elif w["kind"] == "pipeline":
        rows = sum(pipeline_rows(spec, s) for s in range(1 if spec.greedy else 0, spec.k))
    else:
        rows = spec.gamma1 + 1 + spec.gamma2 + (0 if spec.greedy else spec.gamma1)
    return spec.B * rows * spec.V * es
