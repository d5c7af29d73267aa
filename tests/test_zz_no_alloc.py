"""spec_verify_chain_noalloc against spec_verify_chain on the GPU.

The no-allocation entry point keeps its scratch in a static device array
shared by every call on the device, so it is checked on two calls in a row
(the second sees whatever the first left behind) and must give exactly the
outputs of the workspace entry point on the same inputs.  This file sorts
last so that it also runs after every other GPU test in the same process;
it passes on its own in a fresh process as well.
"""

import numpy as np
import pytest
import torch

from workloads import synth
from .gpu_helpers import dev, dev_logits, logits_view

pytestmark = pytest.mark.gpu


def _inputs(spec, seed, device):
    w = synth.make_chain(spec, seed=seed)
    tgt = logits_view(dev_logits(w["target"], spec.dtype, device), spec.V)
    drf = logits_view(dev_logits(w["draft"], spec.dtype, device), spec.V)
    return (tgt, drf, dev(w["tokens"], device), dev(w["u"], device), dev(w["v"], device),
            dev(w["prefix_len"], device))


def _np(out):
    torch.cuda.synchronize()
    return {k: v.cpu().numpy().copy() for k, v in out.items()}


def _same(a, b):
    assert a.keys() == b.keys()
    for k in a:
        assert a[k].tobytes() == b[k].tobytes(), k


CASES = [
    synth.with_sizes(synth.SPECS["sampling_chain_b32_g8_v32000_bf16"], B=16),
    synth.with_sizes(synth.SPECS["sampling_chain_b64_g5_v128256_bf16_a60"], B=64),
    synth.with_sizes(synth.SPECS["greedy_chain_b4_g4_v1000_f32"], B=8, pad=3),
]


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_noalloc_matches_workspace_entry_on_consecutive_calls(cuda_device, spec):
    from draft_verification_gb300 import ChainPlan, ChainPlanNoAlloc
    kw = dict(greedy=spec.greedy, temperature=spec.temperature)
    for seed in (11, 12):  # two calls in a row, different inputs
        args = _inputs(spec, seed, cuda_device)
        want = _np(ChainPlan(*args, **kw).run())
        plan = ChainPlanNoAlloc(*args, **kw)
        first = _np(plan.run())
        second = _np(plan.run())
        _same(first, want)
        _same(second, want)
        assert want["error_word"][0] == 0


def test_noalloc_consulted_only_on_consecutive_calls(cuda_device):
    # consulted-only mode keeps its control words (chunk counters, first
    # rejections) in the shared scratch and must find them cleared on every
    # call, whatever the previous call left there: two calls in a row on each
    # of two input sets, against the workspace entry point in the same mode
    from draft_verification_gb300 import ChainPlan, ChainPlanNoAlloc
    spec = synth.with_sizes(synth.SPECS["sampling_chain_b64_g5_v128256_bf16_a30"], B=24)
    kw = dict(greedy=False, temperature=spec.temperature, consulted_only=True)
    for seed in (13, 14):
        args = _inputs(spec, seed, cuda_device)
        want = _np(ChainPlan(*args, **kw).run())
        plan = ChainPlanNoAlloc(*args, **kw)
        first = _np(plan.run())
        second = _np(plan.run())
        _same(first, want)
        _same(second, want)
        assert (want["accept_len"] < spec.gamma).any()  # some rows after a rejection were skipped


def test_noalloc_runs_allocate_no_device_memory(cuda_device):
    from draft_verification_gb300 import ChainPlanNoAlloc
    spec = synth.with_sizes(synth.SPECS["sampling_chain_b32_g8_v32000_bf16"], B=8)
    plan = ChainPlanNoAlloc(*_inputs(spec, 3, cuda_device), greedy=False,
                            temperature=spec.temperature)
    assert plan.workspace.numel() == 0
    plan.run()  # first call on the device: symbol lookup, module load
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info(cuda_device)[0]
    for _ in range(3):
        plan.run()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(cuda_device)[0] == free0


def test_noalloc_oversize_is_refused(cuda_device):
    from draft_verification_gb300 import _lib
    import ctypes as C
    a = _lib.ChainArgs()
    a.B, a.gamma, a.V, a.ld = 4096, 8, 131072, 131072
    a.dtype, a.mode, a.temperature = _lib.SPEC_BF16, _lib.SPEC_SAMPLE, 1.0
    code = _lib.lib().spec_verify_chain_noalloc(C.byref(a), None)
    assert code == _lib.SPEC_EWORKSPACE
    assert "workspace" in _lib.status_string(code)
