"""The torch binding's own argument checks (no GPU: each raises before any
device memory is touched)."""

import pytest
import torch

from draft_verification_gb300 import ClaspPlan, PipelineAsyncPlan


def test_clasp_plan_rejects_bad_inputs():
    h = torch.zeros(2, 5, 64)
    w = torch.zeros(4, 64, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        ClaspPlan(h.double(), w, 2)                     # hidden must be float32
    with pytest.raises(TypeError):
        ClaspPlan(h, w.float(), 2)                      # weights must be bfloat16
    with pytest.raises(TypeError):
        ClaspPlan(h, w[:3], 2)                          # one matrix per layer
    with pytest.raises(TypeError):
        ClaspPlan(h[:, :, :32], w, 2)                   # widths must agree
    with pytest.raises(TypeError):
        ClaspPlan(h.transpose(0, 1), w, 2)              # contiguous only
    with pytest.raises(ValueError):
        ClaspPlan(h, w, 5)                              # M > L
    with pytest.raises(ValueError):
        ClaspPlan(torch.zeros(2, 5, 60), torch.zeros(4, 60, 60, dtype=torch.bfloat16), 2)  # d % 8 != 0


def test_pipeline_async_plan_rejects_bad_inputs():
    B, Vv = 3, 50
    tg = [torch.zeros(B, 4, Vv, dtype=torch.bfloat16), torch.zeros(B, 3, Vv, dtype=torch.bfloat16)]
    dr = [torch.zeros(B, 3, Vv, dtype=torch.bfloat16), torch.zeros(B, 2, Vv, dtype=torch.bfloat16)]
    tok = [torch.zeros(B, 3, dtype=torch.int32), torch.zeros(B, 2, dtype=torch.int32)]
    length = torch.zeros(3, B, dtype=torch.int32)
    with pytest.raises(ValueError):
        PipelineAsyncPlan(tg, dr, tok[:1], length, greedy=True)          # one token window per stage
    with pytest.raises(ValueError):
        PipelineAsyncPlan(tg, dr, tok, torch.zeros(2, B, dtype=torch.int32), greedy=True)  # [k, B] lengths
    with pytest.raises(ValueError):
        PipelineAsyncPlan([tg[0], tg[1][:, :2]], dr, tok, length, greedy=True)  # w_s + 1 target rows
    with pytest.raises(ValueError):
        PipelineAsyncPlan([tg[0], tg[1].float()], dr, tok, length, greedy=True)  # one dtype
    with pytest.raises(TypeError):
        PipelineAsyncPlan(tg, dr, tok, length.long(), greedy=True)       # int32 lengths
