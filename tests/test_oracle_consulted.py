"""The consulted-rows chain oracle against the ordinary chain oracle (no GPU).

Pins:
  * on finite inputs, decisions, token, rollback, residual mass and error bits
    equal the ordinary rule's (oracle.verify, pinned in tests/pins.py), and
    p(d_i), q(d_i) equal it at every consulted position and are NaN after;
  * a non-finite row is an error exactly when it is consulted (rows of the
    first rejection or before, the bonus row when everything is kept);
  * rows_read = 2 (a + 1) after a rejection at a, 2 gamma + 1 otherwise.
Planted mistakes (an error raised for unconsulted rows, a position's rows
counted once) must fail a pin.
"""

import numpy as np
import pytest

from oracle import consulted as Cn
from oracle import verify as V
from workloads import synth


def _case(seed, alpha_name="sampling_chain_b64_g5_v128256_bf16_a60", B=24, V_=900):
    spec = synth.with_sizes(synth.SPECS[alpha_name], B=B, V=V_)
    return spec, synth.make(spec, seed=seed)


def pin_equal_on_finite(fn):
    for name in ("sampling_chain_b64_g5_v128256_bf16_a05", "sampling_chain_b64_g5_v128256_bf16_a60",
                 "sampling_chain_b64_g5_v128256_bf16_a90"):
        spec, w = _case(3, name)
        o = V.verify_chain(w["target"], w["draft"], w["tokens"], w["u"], w["v"], w["prefix_len"], spec.temperature,
                           False, spec.dtype, V=spec.V)
        c = fn(w["target"], w["draft"], w["tokens"], w["u"], w["v"], w["prefix_len"], spec.temperature,
               spec.dtype, V=spec.V)
        for k in ("accept_len", "out_token", "rollback_idx", "error"):
            assert np.array_equal(c[k], o[k]), k
        assert np.allclose(c["resid_mass"], o["resid_mass"], rtol=0, atol=0)
        g = spec.gamma
        for b in range(spec.B):
            a = int(o["accept_len"][b])
            last = min(a, g - 1)
            assert np.array_equal(c["p_at_draft"][b, :last + 1], o["p_at_draft"][b, :last + 1])
            assert np.array_equal(c["q_at_draft"][b, :last + 1], o["q_at_draft"][b, :last + 1])
            assert np.isnan(c["p_at_draft"][b, last + 1:]).all() and np.isnan(c["q_at_draft"][b, last + 1:]).all()
            want = 2 * (a + 1) if a < g else 2 * g + 1
            assert c["rows_read"][b] == want


def pin_nonfinite_only_when_consulted(fn):
    spec, w = _case(5, B=12)
    o = V.verify_chain(w["target"], w["draft"], w["tokens"], w["u"], w["v"], w["prefix_len"], spec.temperature,
                       False, spec.dtype, V=spec.V)
    g = spec.gamma
    nan = synth.bf16_from_float32(np.array([np.nan], np.float32))[0]
    expect = np.zeros(spec.B, np.int64)
    for b in range(spec.B):
        a = int(o["accept_len"][b])
        if b % 3 == 0 and a + 1 < g:       # after the first rejection: never read
            w["draft"][b, a + 1, 7] = nan
        elif b % 3 == 1:                   # the rejected position itself (or the bonus row): read
            if a < g:
                w["target"][b, a, 3] = nan
            else:
                w["target"][b, g, 3] = nan
            expect[b] = V.ERR_NONFINITE
        elif a > 0:                        # a kept position: read
            w["draft"][b, 0, 1] = nan
            expect[b] = V.ERR_NONFINITE
    c = fn(w["target"], w["draft"], w["tokens"], w["u"], w["v"], w["prefix_len"], spec.temperature, spec.dtype,
           V=spec.V)
    assert np.array_equal(c["error"], expect), (c["error"], expect)


PINS = [pin_equal_on_finite, pin_nonfinite_only_when_consulted]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(Cn.verify_chain_consulted)


def _flag_everything(*args, **kw):
    r = Cn.verify_chain_consulted(*args, **kw)
    target, draft = args[0], args[1]
    dtype, V_ = args[7], kw.get("V")
    for b in range(target.shape[0]):
        rows = [V.row_to_float64(target[b, i, :V_], dtype) for i in range(target.shape[1])]
        rows += [V.row_to_float64(draft[b, i, :V_], dtype) for i in range(draft.shape[1])]
        if any(V.row_is_nonfinite(x) for x in rows):
            r["error"][b] = V.ERR_NONFINITE
    return r


def _rows_once(*args, **kw):
    r = Cn.verify_chain_consulted(*args, **kw)
    r["rows_read"] = r["rows_read"] // 2 + 1
    return r


@pytest.mark.parametrize("mutant", [_flag_everything, _rows_once], ids=lambda m: m.__name__)
def test_planted_mistake_is_caught(mutant):
    caught = False
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught = True
            break
    assert caught
