"""Reading R3 on the GPU: a residual with no mass after a rejection.

In exact arithmetic max(0, p - q) has mass 0 only when p == q, and then a
token is rejected only where p = q = 0 (reading R2).  The exact cases below
copy the target rows into the draft rows and mask the drafted token (-inf in
both), so the rejection, the zero mass, the fallback draw from p and error
bit 8 are all fixed by the inputs: both sides must agree on the whole error
word.  The rows span several statistics chunks and pass tiles.

The last case is the inexact neighbour: rows one bfloat16 step apart at a
low-probability drafted token.  Its float64 residual mass is positive but far
below the float32 rounding of the rows' weights, so the oracle reports it as
set aside and the GPU result is only checked for validity.
"""

import numpy as np
import pytest

from workloads import synth

from . import gpu_helpers as H

pytestmark = pytest.mark.gpu

S = synth.SPECS
W = synth.with_sizes
NEG_INF_BF16 = np.uint16(0xFF80)


def _mask_chain(w, b, pos):
    """Draft rows 0..pos of sequence b equal the target rows (every earlier
    position then has r = 1 and is kept) and the drafted token at pos is
    masked in both rows: rejected with zero residual mass."""
    w["draft"][b, :pos + 1] = w["target"][b, :pos + 1]
    d = int(w["tokens"][b, pos])
    w["target"][b, pos, d] = NEG_INF_BF16
    w["draft"][b, pos, d] = NEG_INF_BF16


def test_chain_zero_mass_exact(cuda_device):
    spec = W(S["sampling_chain_b32_g8_v32000_bf16"], B=8, gamma=5, V=40000, pad=3)
    w = synth.make(spec, seed=31)
    for b, pos in ((1, 0), (4, 2), (6, 4)):
        _mask_chain(w, b, pos)
    g, o = H.gpu_chain(w, cuda_device), H.oracle_chain(w)
    for b, pos in ((1, 0), (4, 2), (6, 4)):
        assert o["error"][b] == 8 and o["accept_len"][b] == pos and o["min_mass"][b] == 0.0
        assert g["seq_error"][b] == 8 and g["accept_len"][b] == pos
    flagged = H.compare_chain(g, o, False)
    assert not flagged[[1, 4, 6]].any()
    assert g["error_word"][0] & 8


def test_chain_zero_mass_exact_consulted_only(cuda_device):
    from oracle import consulted as Cn
    spec = W(S["sampling_chain_b32_g8_v32000_bf16"], B=6, gamma=4, V=20000)
    w = synth.make(spec, seed=32)
    _mask_chain(w, 2, 1)
    g = H.gpu_chain(w, cuda_device, consulted_only=True)
    o = Cn.verify_chain_consulted(w["target"], w["draft"], w["tokens"], w["u"], w["v"], w["prefix_len"],
                                  spec.temperature, spec.dtype, V=spec.V)
    assert o["error"][2] == 8 and g["seq_error"][2] == 8
    flagged = H.set_aside(o, False)
    H.compare_errors(g["seq_error"], o["error"], flagged, 5)
    keep = ~flagged
    for k in ("accept_len", "out_token", "rollback_idx"):
        assert np.array_equal(g[k][keep], o[k][keep]), k


def test_tree_zero_mass_exact(cuda_device):
    spec = W(S["tree_b16_n64_v50257_bf16"], B=4, V=33000)
    w = synth.make(spec, seed=33)
    # sequence 1: the root's rows equal, the first child's token masked
    first_child = int(np.flatnonzero(w["parent"][1] == 0)[0])
    w["draft"][1, 0] = w["target"][1, 0]
    t = int(w["tokens"][1, first_child])
    w["target"][1, 0, t] = NEG_INF_BF16
    w["draft"][1, 0, t] = NEG_INF_BF16
    g, o = H.gpu_tree(w, cuda_device), H.oracle_tree(w)
    assert o["error"][1] == 8 and o["path_len"][1] == 0
    assert g["seq_error"][1] == 8 and g["path_len"][1] == 0
    H.compare_tree(g, o, False)


def test_cascade_stage1_zero_mass_exact(cuda_device):
    spec = W(S["cascade_b128_g8_g4_v128256_bf16"], B=6, V=25000, pad=1)
    w = synth.make(spec, seed=34)
    # sequence 3: M_0 and M_1 agree on positions 0..2, token 2 masked in both
    w["l0"][3, :3] = w["l1"][3, :3]
    d = int(w["tokens"][3, 2])
    w["l0"][3, 2, d] = NEG_INF_BF16
    w["l1"][3, 2, d] = NEG_INF_BF16
    g, o = H.gpu_cascade(w, cuda_device), H.oracle_cascade(w)
    assert o["a1"][3] == 2 and o["error"][3] & 8
    assert g["a1"][3] == 2 and g["seq_error"][3] & 8
    H.compare_cascade(g, o, False)


def test_chain_rows_one_step_apart_are_set_aside(cuda_device):
    """Rows equal except that the draft logit of the drafted token is one
    bfloat16 step above the target's: r is just below 1 and u just below 1,
    so position 0 is rejected, and the residual is the normalisation
    difference of two rows that agree to about 1e-13: far below what the
    float32 weights resolve."""
    spec = W(S["sampling_chain_b32_g8_v32000_bf16"], B=6, gamma=3, V=40000)
    w = synth.make(spec, seed=35)
    b = 2
    w["draft"][b, 0] = w["target"][b, 0]
    vals = synth.float32_from_bf16(w["target"][b, 0])
    d = int(np.argmin(vals))  # a low-probability token
    w["tokens"][b, 0] = d
    w["draft"][b, 0, d] = w["target"][b, 0, d] - np.uint16(1)  # negative: one step larger in magnitude ...
    if synth.float32_from_bf16(w["draft"][b, 0, d:d + 1])[0] < vals[d]:
        w["draft"][b, 0, d] = w["target"][b, 0, d] + np.uint16(1)  # ... so go the other way
    assert synth.float32_from_bf16(w["draft"][b, 0, d:d + 1])[0] > vals[d]
    w["u"][b, 0] = np.float32(0.999999)
    g, o = H.gpu_chain(w, cuda_device), H.oracle_chain(w)
    assert o["accept_len"][b] == 0 and 0.0 < o["min_mass"][b] < H.Z_MIN
    flagged = H.compare_chain(g, o, False)
    assert flagged[b]
    # set aside, but still a valid result: the same rejection, a token in
    # range, no data-error bits and no wait that gave up
    assert g["accept_len"][b] == 0 and 0 <= g["out_token"][b] < spec.V
    assert g["seq_error"][b] & ~8 == 0
