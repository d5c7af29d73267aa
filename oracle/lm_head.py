"""Chain verification from the models' final hidden states (the LM head
folded into the verification), written out in float64 NumPy.

TEST INFRASTRUCTURE ONLY (see the package docstring): only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` call it.

Source: "Accelerating LLM Inference with Staged Speculative Decoding"
(arXiv 2308.04623), abstract: small-batch inference has low arithmetic
intensity, so the step is bound by memory traffic; the verification reads
the vocabulary-wide logits, which the LM head writes just before.  The rule
is the one of ``oracle.verify`` (PipeSpec review, Circularity Check).

Reading (R19 in the design notes): the target logits at the gamma + 1
positions are H_t W_t^T and the draft logits at the gamma positions
H_d W_d^T, with hidden states H [rows, d] and LM-head weights W [V, d] given
as bfloat16 values; the products are exact here (float64 of the bfloat16
values; float32 accumulation on the tensor cores is the kernel's business),
and the chain rule is applied to them as to stored logits.
"""

from __future__ import annotations

import numpy as np

from .verify import bf16_bits_to_float64, verify_chain_sequence


def head_logits(hidden, weights):
    """hidden float64 [rows, d], weights float64 [V, d] -> logits [rows, V]."""
    return np.asarray(hidden, np.float64) @ np.asarray(weights, np.float64).T


def verify_chain_from_hidden(h_target, h_draft, w_target, w_draft, tokens, u, v, prefix_len, temperature, greedy):
    """Batch: h_target [B, gamma+1, d], h_draft [B, gamma, d], w_target
    [V, d], w_draft [V, d] (float64 values of bfloat16 numbers), tokens int
    [B, gamma], u [B, gamma], v [B], prefix_len [B].  Returns accept_len,
    out_token, rollback_idx, error, margin_u, margin_v [B], and the chain
    oracle's diagnostics p_at_draft, q_at_draft [B, gamma], resid_mass,
    min_mass [B]."""
    B, gamma = tokens.shape
    res = {k: np.zeros(B, np.int64) for k in ("accept_len", "out_token", "rollback_idx", "error")}
    res.update(margin_u=np.zeros(B), margin_v=np.zeros(B), resid_mass=np.zeros(B), min_mass=np.zeros(B),
               p_at_draft=np.zeros((B, gamma)), q_at_draft=np.zeros((B, gamma)))
    for b in range(B):
        target = head_logits(h_target[b], w_target)
        draft = None if greedy else head_logits(h_draft[b], w_draft)
        r = verify_chain_sequence(target, draft, [int(t) for t in tokens[b]], None if greedy else u[b],
                                  None if greedy else float(v[b]), temperature, greedy)
        for k in ("accept_len", "out_token", "error", "margin_u", "margin_v", "resid_mass", "min_mass"):
            res[k][b] = r[k]
        res["p_at_draft"][b] = r["p_at_draft"]
        res["q_at_draft"][b] = r["q_at_draft"]
        res["rollback_idx"][b] = int(prefix_len[b]) + r["accept_len"]
    return res


def bf16_values(bits):
    """bfloat16 bit patterns (uint16) -> float64 values."""
    return bf16_bits_to_float64(np.asarray(bits, np.uint16))
