"""Torch-facing binding of the verification library (argument marshalling only).

PyTorch supplies device memory and the current stream; every step of the
verification runs in the CUDA kernels behind the C ABI (include/spec_verify.h).

Two ways to call:
  * ``verify_chain / verify_tree / verify_cascade``: one call, returns a dict
    of output tensors.  Device tensors stay on the device; CPU tensors are
    copied to ``device`` first and the results copied back (end-to-end use).
  * ``ChainPlan / TreePlan / CascadePlan``: bind the input and output buffers
    once, then ``plan.run()`` launches with no Python-side allocation (a
    prebuilt argument struct and one ctypes call).
"""

from __future__ import annotations

import ctypes as C

import torch

from . import _lib as L

_DTYPES = {torch.float32: L.SPEC_F32, torch.bfloat16: L.SPEC_BF16}


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _rows(t: torch.Tensor, rows: int, name: str) -> int:
    """Row stride (elements) of a [B, rows, V] logit view; checks the layout
    the C ABI assumes: row (b, i) starts at (b * rows + i) * ld."""
    if t.dim() != 3 or t.shape[1] != rows:
        raise ValueError(f"{name}: expected [B, {rows}, V], got {tuple(t.shape)}")
    if t.dtype not in _DTYPES:
        raise TypeError(f"{name}: logits must be float32 or bfloat16")
    if t.stride(2) != 1:
        raise ValueError(f"{name}: logits must have unit element stride")
    if rows == 1:  # one row per sequence: the row stride is the batch stride
        return t.stride(0) if t.shape[0] > 1 else t.shape[2]
    if t.shape[0] > 1 and t.stride(0) != rows * t.stride(1):
        raise ValueError(f"{name}: rows must be evenly strided")
    return t.stride(1)


def _i32(t, name):
    if t is None:
        return None
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous int32 tensor")
    return t


def _f32(t, name):
    if t is None:
        return None
    if t.dtype != torch.float32 or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous float32 tensor")
    return t


def _check(code: int, what: str):
    if code != L.SPEC_OK:
        raise RuntimeError(f"{what} failed: {L.status_string(code)} ({code})")


def _stream_handle(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


class _Plan:
    def run(self, stream=None):
        _check(self._call(C.byref(self.args), _stream_handle(stream)), type(self).__name__)
        return self.out


class ChainPlan(_Plan):
    """Chain verification bound to fixed buffers.  See spec_verify_chain."""

    def __init__(self, target, draft, tokens, u=None, v=None, prefix_len=None, *,
                 greedy=False, temperature=1.0, V=None, workspace=None, want_probs=True, consulted_only=False):
        B, R, width = target.shape
        gamma = R - 1
        V = width if V is None else V
        dev = target.device
        ld = _rows(target, gamma + 1, "target")
        if not greedy and gamma > 0:
            if draft is None or draft.dtype != target.dtype or _rows(draft, gamma, "draft") != ld:
                raise ValueError("draft: same dtype and row stride as target required")
        lib = L.lib()
        self.keep = [target, draft, tokens, u, v, prefix_len]
        self.out = dict(
            accept_len=torch.empty(B, dtype=torch.int32, device=dev),
            out_token=torch.empty(B, dtype=torch.int32, device=dev),
            rollback_idx=torch.empty(B, dtype=torch.int32, device=dev),
            seq_error=torch.empty(B, dtype=torch.int32, device=dev),
            error_word=torch.zeros(1, dtype=torch.int32, device=dev),
        )
        if want_probs:
            self.out["p_at_draft"] = torch.empty(B, gamma, dtype=torch.float32, device=dev)
            self.out["q_at_draft"] = torch.empty(B, gamma, dtype=torch.float32, device=dev)
            self.out["resid_mass"] = torch.empty(B, dtype=torch.float32, device=dev)
        need = lib.spec_chain_workspace_size(B, gamma, V)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        self.workspace = workspace
        a = L.ChainArgs()
        a.B, a.gamma, a.V, a.ld = B, gamma, V, ld
        a.dtype = _DTYPES[target.dtype]
        a.mode = L.SPEC_GREEDY if greedy else L.SPEC_SAMPLE
        a.temperature = float(temperature)
        a.target_logits = _ptr(target)
        a.draft_logits = _ptr(draft) if not greedy else None
        a.draft_tokens = _ptr(_i32(tokens, "tokens"))
        a.u = _ptr(_f32(u, "u")) if not greedy else None
        a.v = _ptr(_f32(v, "v")) if not greedy else None
        a.prefix_len = _ptr(_i32(prefix_len, "prefix_len"))
        o = self.out
        a.accept_len, a.out_token = _ptr(o["accept_len"]), _ptr(o["out_token"])
        a.rollback_idx, a.seq_error = _ptr(o["rollback_idx"]), _ptr(o["seq_error"])
        a.error_word = _ptr(o["error_word"])
        a.p_at_draft = _ptr(o.get("p_at_draft"))
        a.q_at_draft = _ptr(o.get("q_at_draft"))
        a.resid_mass = _ptr(o.get("resid_mass"))
        a.workspace, a.workspace_bytes = _ptr(workspace), workspace.numel()
        a.consulted_only = int(bool(consulted_only))
        self.args = a
        self._call = lib.spec_verify_chain


class ChainPlanNoAlloc(ChainPlan):
    """ChainPlan bound to spec_verify_chain_noalloc: the library's static
    scratch replaces the workspace tensor, so neither this plan nor its runs
    allocate scratch.  Runs that can overlap on the GPU race on that scratch;
    the first run on a device should come before any stream capture."""

    def __init__(self, target, *args, **kw):
        if kw.get("workspace") is not None:
            raise TypeError("ChainPlanNoAlloc takes no workspace")
        # a zero-element tensor holds no device memory; the entry point
        # ignores the workspace fields
        kw["workspace"] = torch.empty(0, dtype=torch.uint8, device=target.device)
        super().__init__(target, *args, **kw)
        self._call = L.lib().spec_verify_chain_noalloc


class LmHeadChainPlan(_Plan):
    """Chain verification from final hidden states and LM-head weights,
    bound to fixed buffers.  See spec_verify_chain_lm_head.

    h_target [B, gamma+1, d_t] and h_draft [B, gamma, d_d] bfloat16 hidden
    states, w_target [V, d_t] and w_draft [V, d_d] bfloat16 heads (the draft
    ones are not read in greedy mode and may be None).  The workspace holds
    the chunk partials and, in sampling mode, the float32 logits of every row
    (``target_logits()`` / ``draft_logits()`` view them after a run)."""

    def __init__(self, h_target, h_draft, w_target, w_draft, tokens, u=None, v=None, prefix_len=None, *,
                 greedy=False, temperature=1.0, workspace=None):
        B, R, d_t = h_target.shape
        gamma = R - 1
        V = w_target.shape[0]
        dev = h_target.device
        for name, t in (("h_target", h_target), ("w_target", w_target)):
            if t.dtype != torch.bfloat16 or not t.is_contiguous():
                raise ValueError(f"{name}: contiguous bfloat16 required")
        d_d = 0
        if not greedy and gamma > 0:
            for name, t in (("h_draft", h_draft), ("w_draft", w_draft)):
                if t is None or t.dtype != torch.bfloat16 or not t.is_contiguous():
                    raise ValueError(f"{name}: contiguous bfloat16 required")
            d_d = h_draft.shape[2]
            if tuple(h_draft.shape[:2]) != (B, gamma) or tuple(w_draft.shape) != (V, d_d):
                raise ValueError("h_draft [B, gamma, d_draft] and w_draft [V, d_draft] required")
        if w_target.shape[1] != d_t:
            raise ValueError("w_target [V, d_target] required")
        lib = L.lib()
        self.B, self.gamma, self.V = B, gamma, V
        self.keep = [h_target, h_draft, w_target, w_draft, tokens, u, v, prefix_len]
        self.out = dict(
            accept_len=torch.empty(B, dtype=torch.int32, device=dev),
            out_token=torch.empty(B, dtype=torch.int32, device=dev),
            rollback_idx=torch.empty(B, dtype=torch.int32, device=dev),
            seq_error=torch.empty(B, dtype=torch.int32, device=dev),
            error_word=torch.zeros(1, dtype=torch.int32, device=dev),
            p_at_draft=torch.empty(B, gamma, dtype=torch.float32, device=dev),
            q_at_draft=torch.empty(B, gamma, dtype=torch.float32, device=dev),
            resid_mass=torch.empty(B, dtype=torch.float32, device=dev),
        )
        mode = L.SPEC_GREEDY if greedy else L.SPEC_SAMPLE
        need = lib.spec_lm_head_chain_workspace_size(B, gamma, V, mode)
        if workspace is None:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        self.workspace = workspace
        self.greedy = greedy
        a = L.LmHeadChainArgs()
        a.B, a.gamma, a.V, a.d_target, a.d_draft = B, gamma, V, d_t, d_d
        a.mode = mode
        a.temperature = float(temperature)
        a.h_target, a.w_target = _ptr(h_target), _ptr(w_target)
        a.h_draft = _ptr(h_draft) if d_d else None
        a.w_draft = _ptr(w_draft) if d_d else None
        a.draft_tokens = _ptr(_i32(tokens, "tokens"))
        a.u = _ptr(_f32(u, "u")) if not greedy else None
        a.v = _ptr(_f32(v, "v")) if not greedy else None
        a.prefix_len = _ptr(_i32(prefix_len, "prefix_len"))
        o = self.out
        a.accept_len, a.out_token = _ptr(o["accept_len"]), _ptr(o["out_token"])
        a.rollback_idx, a.seq_error = _ptr(o["rollback_idx"]), _ptr(o["seq_error"])
        a.error_word = _ptr(o["error_word"])
        a.p_at_draft, a.q_at_draft = _ptr(o["p_at_draft"]), _ptr(o["q_at_draft"])
        a.resid_mass = _ptr(o["resid_mass"])
        a.workspace, a.workspace_bytes = _ptr(workspace), workspace.numel()
        self.args = a
        self._call = lib.spec_verify_chain_lm_head

    def _logits(self, first_row, rows):
        # the workspace layout of spec_lm_head_chain_workspace_size: the
        # partials (two columns per 256-entry vocabulary tile, at most 256),
        # then the target rows, then the draft rows (each part
        # rounded up to 256 bytes), row stride V rounded up to 8
        if self.greedy:
            raise ValueError("greedy calls store no logits")
        ldl = (self.V + 7) // 8 * 8
        chunks = min(2 * ((self.V + 255) // 256), 256)
        part = -(-self.B * (2 * self.gamma + 1) * chunks * 8 // 256) * 256
        tbytes = -(-self.B * (self.gamma + 1) * ldl * 4 // 256) * 256
        off = part + (0 if first_row == 0 else tbytes)
        f = self.workspace[off: off + rows * ldl * 4].view(torch.float32)
        return f.view(rows, ldl)[:, :self.V]

    def target_logits(self):
        return self._logits(0, self.B * (self.gamma + 1)).view(self.B, self.gamma + 1, self.V)

    def draft_logits(self):
        return self._logits(1, self.B * self.gamma).view(self.B, self.gamma, self.V)


class TreePlan(_Plan):
    """Tree verification bound to fixed buffers.  See spec_verify_tree."""

    def __init__(self, parent, tokens, target, draft, u=None, v=None, prefix_len=None, *,
                 max_depth, greedy=False, temperature=1.0, V=None, workspace=None, consulted_only=False):
        B, N, width = target.shape
        V = width if V is None else V
        dev = target.device
        ld = _rows(target, N, "target")
        if not greedy:
            if draft is None or draft.dtype != target.dtype or _rows(draft, N, "draft") != ld:
                raise ValueError("draft: same dtype and row stride as target required")
        lib = L.lib()
        self.keep = [parent, tokens, target, draft, u, v, prefix_len]
        self.out = dict(
            path_len=torch.empty(B, dtype=torch.int32, device=dev),
            path_nodes=torch.empty(B, max_depth + 1, dtype=torch.int32, device=dev),
            out_token=torch.empty(B, dtype=torch.int32, device=dev),
            rollback_idx=torch.empty(B, dtype=torch.int32, device=dev),
            seq_error=torch.empty(B, dtype=torch.int32, device=dev),
            error_word=torch.zeros(1, dtype=torch.int32, device=dev),
        )
        need = lib.spec_tree_workspace_size(B, N, V)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        self.workspace = workspace
        a = L.TreeArgs()
        a.B, a.N, a.max_depth, a.V, a.ld = B, N, int(max_depth), V, ld
        a.dtype = _DTYPES[target.dtype]
        a.mode = L.SPEC_GREEDY if greedy else L.SPEC_SAMPLE
        a.temperature = float(temperature)
        a.parent = _ptr(_i32(parent, "parent"))
        a.node_tokens = _ptr(_i32(tokens, "tokens"))
        a.target_logits = _ptr(target)
        a.draft_logits = _ptr(draft) if not greedy else None
        a.u = _ptr(_f32(u, "u")) if not greedy else None
        a.v = _ptr(_f32(v, "v")) if not greedy else None
        a.prefix_len = _ptr(_i32(prefix_len, "prefix_len"))
        o = self.out
        a.path_len, a.path_nodes = _ptr(o["path_len"]), _ptr(o["path_nodes"])
        a.out_token, a.rollback_idx = _ptr(o["out_token"]), _ptr(o["rollback_idx"])
        a.seq_error, a.error_word = _ptr(o["seq_error"]), _ptr(o["error_word"])
        a.workspace, a.workspace_bytes = _ptr(workspace), workspace.numel()
        a.consulted_only = int(bool(consulted_only))
        self.args = a
        self._call = lib.spec_verify_tree


class CascadePlan(_Plan):
    """PipeSpec cascade snapshot bound to fixed buffers.  See spec_verify_cascade."""

    def __init__(self, l0, l1, l2, tokens, u1=None, v1=None, u2=None, v2=None, base0=None,
                 base1=None, *, greedy=False, temperature=1.0, V=None, workspace=None):
        B, g1p1, width = l1.shape
        g1 = g1p1 - 1
        g2 = l2.shape[1]
        V = width if V is None else V
        dev = l1.device
        ld = _rows(l1, g1 + 1, "l1")
        if _rows(l2, g2, "l2") != ld or l2.dtype != l1.dtype:
            raise ValueError("l2: same dtype and row stride as l1 required")
        if not greedy and (l0 is None or l0.dtype != l1.dtype or _rows(l0, g1, "l0") != ld):
            raise ValueError("l0: same dtype and row stride as l1 required")
        lib = L.lib()
        self.keep = [l0, l1, l2, tokens, u1, v1, u2, v2, base0, base1]
        names = ("a1", "t1", "a2", "w2", "t2", "t2_valid", "r0", "r1", "committed", "seq_error")
        self.out = {k: torch.empty(B, dtype=torch.int32, device=dev) for k in names}
        self.out["error_word"] = torch.zeros(1, dtype=torch.int32, device=dev)
        need = lib.spec_cascade_workspace_size(B, g1, g2, V)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        self.workspace = workspace
        a = L.CascadeArgs()
        a.B, a.gamma1, a.gamma2, a.V, a.ld = B, g1, g2, V, ld
        a.dtype = _DTYPES[l1.dtype]
        a.mode = L.SPEC_GREEDY if greedy else L.SPEC_SAMPLE
        a.temperature = float(temperature)
        a.l0 = _ptr(l0) if not greedy else None
        a.l1, a.l2 = _ptr(l1), _ptr(l2)
        a.draft_tokens = _ptr(_i32(tokens, "tokens"))
        if not greedy:
            a.u1, a.v1 = _ptr(_f32(u1, "u1")), _ptr(_f32(v1, "v1"))
            a.u2, a.v2 = _ptr(_f32(u2, "u2")), _ptr(_f32(v2, "v2"))
        a.base0, a.base1 = _ptr(_i32(base0, "base0")), _ptr(_i32(base1, "base1"))
        for k in names:
            setattr(a, k, _ptr(self.out[k]))
        a.error_word = _ptr(self.out["error_word"])
        a.workspace, a.workspace_bytes = _ptr(workspace), workspace.numel()
        self.args = a
        self._call = lib.spec_verify_cascade


class PipelinePlan(_Plan):
    """k-model PipeSpec snapshot bound to fixed buffers.  See spec_verify_pipeline.

    models: list of k logit views [B, rows_s, V] with one row stride (models[0]
    may be None in greedy mode); windows: stage windows (windows[0] = drafted
    tokens); us / vs: per-stage uniforms (sampling); base: int32 [k-1, B] or
    None."""

    def __init__(self, models, tokens, windows, us=None, vs=None, base=None, *, greedy=False, temperature=1.0,
                 final_bonus=False, V=None, workspace=None):
        k = len(models)
        windows = [int(g) for g in windows]
        if len(windows) != k - 1:
            raise ValueError("windows: one per stage (k - 1)")
        ref = models[1]
        B = ref.shape[0]
        V = ref.shape[2] if V is None else V
        dev = ref.device
        rows = [windows[0], windows[0] + 1] + [windows[s - 1] + (1 if (final_bonus and s == k - 1) else 0)
                                               for s in range(2, k)]
        ld = None
        for s, m in enumerate(models):
            if m is None:
                if not greedy or s != 0:
                    raise ValueError(f"models[{s}] is required")
                continue
            if m.dtype != ref.dtype:
                raise ValueError("every model: the same dtype")
            this = _rows(m, rows[s], f"models[{s}]")
            if ld is not None and this != ld:
                raise ValueError("every model: the same row stride")
            ld = this
        lib = L.lib()
        self.keep = [models, tokens, us, vs, base]
        i32 = lambda *shape: torch.empty(*shape, dtype=torch.int32, device=dev)
        self.out = dict(a=i32(B, k - 1), w=i32(B, k - 1), t=i32(B, k - 1), t_valid=i32(B, k - 1), r=i32(B, k - 1),
                        committed=i32(B), seq_error=i32(B),
                        error_word=torch.zeros(1, dtype=torch.int32, device=dev))
        win = (C.c_int * (L.SPEC_MAX_MODELS - 1))(*windows)
        need = lib.spec_pipeline_workspace_size(B, k, win, int(final_bonus), V)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        self.workspace = workspace
        a = L.PipelineArgs()
        a.B, a.k, a.final_bonus, a.V, a.ld = B, k, int(bool(final_bonus)), V, ld
        a.window = win
        a.dtype = _DTYPES[ref.dtype]
        a.mode = L.SPEC_GREEDY if greedy else L.SPEC_SAMPLE
        a.temperature = float(temperature)
        for s, m in enumerate(models):
            a.logits[s] = None if m is None else m.data_ptr()
        a.draft_tokens = _i32(tokens, "tokens").data_ptr()
        if not greedy:
            for s in range(k - 1):
                a.u[s] = _f32(us[s], f"us[{s}]").data_ptr()
                a.v[s] = _f32(vs[s], f"vs[{s}]").data_ptr()
        a.base = None if base is None else _i32(base, "base").data_ptr()
        o = self.out
        a.a, a.w, a.t, a.t_valid, a.r = (o[n].data_ptr() for n in ("a", "w", "t", "t_valid", "r"))
        a.committed, a.seq_error, a.error_word = (o[n].data_ptr() for n in ("committed", "seq_error", "error_word"))
        a.workspace, a.workspace_bytes = workspace.data_ptr(), workspace.numel()
        self.args = a
        self._call = lib.spec_verify_pipeline


class PipelineAsyncPlan(_Plan):
    """PipeSpec stages at independent buffer offsets, bound to fixed buffers.
    See spec_verify_pipeline_async.

    targets: per stage s = 1 .. k-1 the logit view [B, w_s + 1, V] of M_s;
    drafts: per stage [B, w_s, V] of M_{s-1} (None in greedy mode); tokens:
    per stage int32 [B, w_s] (the window); us / vs: per stage uniforms
    (sampling); length: int32 [k, B] buffer lengths before the snapshot.
    ``run()`` returns a, t, t_valid, r [B, k-1], committed, seq_error and
    error_word."""

    def __init__(self, targets, drafts, tokens, length, us=None, vs=None, *, greedy=False, temperature=1.0,
                 final_bonus=False, V=None, workspace=None):
        S = len(targets)
        k = S + 1
        if not 1 <= S <= L.SPEC_MAX_MODELS - 1 or len(tokens) != S:
            raise ValueError("targets and tokens: one per stage, 1 .. 7 stages")
        windows = [int(t.shape[1]) for t in tokens]
        ref = targets[0]
        B = ref.shape[0]
        V = ref.shape[2] if V is None else V
        dev = ref.device
        ld = None

        def stride(m, rows, name):
            nonlocal ld
            if m.dtype != ref.dtype:
                raise ValueError("every logit view: the same dtype")
            this = _rows(m, rows, name)
            if ld is not None and this != ld:
                raise ValueError("every logit view: the same row stride")
            ld = this

        for s in range(S):
            stride(targets[s], windows[s] + 1, f"targets[{s}]")
            if not greedy:
                stride(drafts[s], windows[s], f"drafts[{s}]")
        length = _i32(length, "length")
        if tuple(length.shape) != (k, B):
            raise ValueError(f"length: expected [{k}, {B}]")
        lib = L.lib()
        self.keep = [targets, drafts, tokens, length, us, vs]
        i32 = lambda *shape: torch.empty(*shape, dtype=torch.int32, device=dev)
        self.out = dict(a=i32(B, S), t=i32(B, S), t_valid=i32(B, S), r=i32(B, S), committed=i32(B),
                        seq_error=i32(B), error_word=torch.zeros(1, dtype=torch.int32, device=dev))
        win = (C.c_int * (L.SPEC_MAX_MODELS - 1))(*windows)
        need = lib.spec_pipeline_async_workspace_size(B, k, win, V)
        if need == 0:
            raise ValueError(f"asynchronous snapshot sizes out of range: B={B} k={k} windows={windows} V={V}")
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        self.workspace = workspace
        a = L.PipelineAsyncArgs()
        a.B, a.k, a.final_bonus, a.V, a.ld = B, k, int(bool(final_bonus)), V, ld
        a.window = win
        a.dtype = _DTYPES[ref.dtype]
        a.mode = L.SPEC_GREEDY if greedy else L.SPEC_SAMPLE
        a.temperature = float(temperature)
        for s in range(S):
            a.target[s] = targets[s].data_ptr()
            a.tokens[s] = _i32(tokens[s], f"tokens[{s}]").data_ptr()
            if not greedy:
                a.draft[s] = drafts[s].data_ptr()
                a.u[s] = _f32(us[s], f"us[{s}]").data_ptr()
                a.v[s] = _f32(vs[s], f"vs[{s}]").data_ptr()
        a.length = length.data_ptr()
        o = self.out
        a.a, a.t, a.t_valid, a.r = (o[n].data_ptr() for n in ("a", "t", "t_valid", "r"))
        a.committed, a.seq_error, a.error_word = (o[n].data_ptr() for n in ("committed", "seq_error", "error_word"))
        a.workspace, a.workspace_bytes = workspace.data_ptr(), workspace.numel()
        self.args = a
        self._call = lib.spec_verify_pipeline_async


def _to_device(xs, device):
    moved = []
    for x in xs:
        if isinstance(x, torch.Tensor) and x.device.type == "cpu":
            x = x.to(device, non_blocking=True)
        moved.append(x)
    return moved


def _finish(out, host):
    if not host:
        return out
    return {k: v.to("cpu", non_blocking=True) for k, v in out.items()}


def verify_chain(target, draft, tokens, u=None, v=None, prefix_len=None, *, greedy=False,
                 temperature=1.0, V=None, device="cuda", stream=None, consulted_only=False):
    """Verify B draft chains; returns accept_len, out_token, rollback_idx,
    p_at_draft, q_at_draft, resid_mass, seq_error, error_word."""
    host = target.device.type == "cpu"
    if host:
        target, draft, tokens, u, v, prefix_len = _to_device(
            [target, draft, tokens, u, v, prefix_len], device)
    plan = ChainPlan(target, draft, tokens, u, v, prefix_len, greedy=greedy,
                     temperature=temperature, V=V, consulted_only=consulted_only)
    return _finish(plan.run(stream), host)


def verify_tree(parent, tokens, target, draft, u=None, v=None, prefix_len=None, *, max_depth,
                greedy=False, temperature=1.0, V=None, device="cuda", stream=None, consulted_only=False):
    """Walk B draft trees; returns path_len, path_nodes, out_token,
    rollback_idx, seq_error, error_word."""
    host = target.device.type == "cpu"
    if host:
        parent, tokens, target, draft, u, v, prefix_len = _to_device(
            [parent, tokens, target, draft, u, v, prefix_len], device)
    plan = TreePlan(parent, tokens, target, draft, u, v, prefix_len, max_depth=max_depth,
                    greedy=greedy, temperature=temperature, V=V, consulted_only=consulted_only)
    return _finish(plan.run(stream), host)


def verify_cascade(l0, l1, l2, tokens, u1=None, v1=None, u2=None, v2=None, base0=None,
                   base1=None, *, greedy=False, temperature=1.0, V=None, device="cuda",
                   stream=None):
    """One PipeSpec cascade snapshot; returns a1, t1, a2, w2, t2, t2_valid,
    r0, r1, committed, seq_error, error_word."""
    host = l1.device.type == "cpu"
    if host:
        l0, l1, l2, tokens, u1, v1, u2, v2, base0, base1 = _to_device(
            [l0, l1, l2, tokens, u1, v1, u2, v2, base0, base1], device)
    plan = CascadePlan(l0, l1, l2, tokens, u1, v1, u2, v2, base0, base1, greedy=greedy,
                       temperature=temperature, V=V)
    return _finish(plan.run(stream), host)


def _byte_rows(t: torch.Tensor, name: str):
    """(rows per sequence, row bytes, row stride in bytes) of a uint8 tensor
    [B, R, W] whose last dimension is contiguous."""
    if t.dtype != torch.uint8 or t.dim() != 3 or t.stride(2) != 1 or t.stride(0) != t.shape[1] * t.stride(1):
        raise TypeError(f"{name}: expected a uint8 tensor [B, rows, W] with contiguous rows "
                        "(row stride >= W, sequences back to back)")
    return t.shape[1], t.shape[2], t.stride(1)


def compact_tree_path(tree_rows, cache, path_nodes, path_len, prefix_len=None, stream=None):
    """Move each sequence's kept tree path into its contiguous cache, in place.

    tree_rows uint8 [B, N, W] (one row per tree node), cache uint8 [B, C, W]
    (written in place), path_nodes int32 [B, max_depth+1] and path_len int32
    [B] as returned by verify_tree, prefix_len int32 [B] or None.  Returns the
    per-sequence error bits (int32 [B]: 0, or ERR_PARENT for a malformed path).
    See spec_compact_tree_path.
    """
    lib = L.lib()
    B = tree_rows.shape[0]
    N, W, tree_ld = _byte_rows(tree_rows, "tree_rows")
    Cr, W2, cache_ld = _byte_rows(cache, "cache")
    if W2 != W or cache.shape[0] != B:
        raise ValueError("tree_rows and cache: same batch and row size required")
    path_nodes = _i32(path_nodes, "path_nodes")
    seq_error = torch.empty(B, dtype=torch.int32, device=cache.device)
    a = L.CompactArgs()
    a.B, a.N, a.max_depth, a.cache_rows = B, N, path_nodes.shape[1] - 1, Cr
    a.row_bytes, a.tree_ld, a.cache_ld = W, tree_ld, cache_ld
    a.tree_rows, a.cache = _ptr(tree_rows), _ptr(cache)
    a.path_nodes, a.path_len = _ptr(path_nodes), _ptr(_i32(path_len, "path_len"))
    a.prefix_len = _ptr(_i32(prefix_len, "prefix_len"))
    a.seq_error, a.error_word = _ptr(seq_error), None
    _check(lib.spec_compact_tree_path(C.byref(a), _stream_handle(stream)), "compact_tree_path")
    return seq_error


def verify_pipeline(models, tokens, windows, us=None, vs=None, base=None, *, greedy=False, temperature=1.0,
                    final_bonus=False, V=None, device="cuda", stream=None):
    """One k-model PipeSpec snapshot; returns a, w, t, t_valid, r [B, k-1],
    committed, seq_error, error_word (host tensors in, host tensors out)."""
    host = tokens.device.type == "cpu"
    if host:
        models = _to_device(list(models), device)
        tokens, base = _to_device([tokens, base], device)
        us = None if us is None else _to_device(list(us), device)
        vs = None if vs is None else _to_device(list(vs), device)
    plan = PipelinePlan(models, tokens, windows, us, vs, base, greedy=greedy, temperature=temperature,
                        final_bonus=final_bonus, V=V)
    return _finish(plan.run(stream), host)


class ClaspPlan(_Plan):
    """CLaSp layer selection bound to fixed buffers.  See spec_clasp_layer_select.

    hidden float32 [B, L+1, d] (h_0 .. h_L), weights bfloat16 [L, d, d]
    (W_l[out][in]), M layers to skip.  ``run()`` returns skip_mask int32
    [B, L], score float32 [B] and, with ``choices=True``, choice uint8
    [B, L, M+1] (1 skip, 0 keep, 255 not evaluated).
    """

    def __init__(self, hidden, weights, M, *, choices=False, workspace=None):
        lib = L.lib()
        if hidden.dtype != torch.float32 or not hidden.is_contiguous() or hidden.dim() != 3:
            raise TypeError("hidden: expected a contiguous float32 tensor [B, L+1, d]")
        B, L1, d = hidden.shape
        if weights.dtype != torch.bfloat16 or not weights.is_contiguous() or tuple(weights.shape) != (L1 - 1, d, d):
            raise TypeError(f"weights: expected a contiguous bfloat16 tensor [{L1 - 1}, {d}, {d}]")
        dev = hidden.device
        need = int(lib.spec_clasp_workspace_size(B, L1 - 1, d, int(M)))
        if need == 0:
            raise ValueError(f"CLaSp sizes out of range: B={B} L={L1 - 1} d={d} M={M}")
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        self.workspace = workspace
        self.out = {"skip_mask": torch.empty((B, L1 - 1), dtype=torch.int32, device=dev),
                    "score": torch.empty(B, dtype=torch.float32, device=dev)}
        if choices:
            self.out["choice"] = torch.empty((B, L1 - 1, int(M) + 1), dtype=torch.uint8, device=dev)
        self._keep = (hidden, weights)
        a = L.ClaspArgs()
        a.B, a.L, a.d, a.M = B, L1 - 1, d, int(M)
        a.hidden, a.weights = _ptr(hidden), _ptr(weights)
        a.skip_mask, a.score = _ptr(self.out["skip_mask"]), _ptr(self.out["score"])
        a.choice = _ptr(self.out.get("choice"))
        a.workspace, a.workspace_bytes = _ptr(workspace), workspace.numel()
        self.args = a
        self._call = lib.spec_clasp_layer_select


def clasp_layer_select(hidden, weights, M, *, choices=False, device="cuda", stream=None):
    """One CLaSp layer selection (host tensors in, host tensors out; device
    tensors stay on the device).  See ClaspPlan."""
    host = hidden.device.type == "cpu"
    if host:
        hidden, weights = _to_device([hidden, weights], device)
    plan = ClaspPlan(hidden, weights, M, choices=choices)
    return _finish(plan.run(stream), host)


def verify_pipeline_async(targets, drafts, tokens, length, us=None, vs=None, *, greedy=False, temperature=1.0,
                          final_bonus=False, V=None, device="cuda", stream=None):
    """One asynchronous PipeSpec snapshot (host tensors in, host tensors out;
    device tensors stay on the device).  See PipelineAsyncPlan."""
    host = length.device.type == "cpu"
    if host:
        targets = _to_device(list(targets), device)
        drafts = None if drafts is None else _to_device(list(drafts), device)
        tokens = _to_device(list(tokens), device)
        (length,) = _to_device([length], device)
        us = None if us is None else _to_device(list(us), device)
        vs = None if vs is None else _to_device(list(vs), device)
    plan = PipelineAsyncPlan(targets, drafts, tokens, length, us, vs, greedy=greedy, temperature=temperature,
                             final_bonus=final_bonus, V=V)
    return _finish(plan.run(stream), host)


def workspace_bytes(kind: str, *sizes) -> int:
    fn = {"chain": "spec_chain_workspace_size", "tree": "spec_tree_workspace_size",
          "cascade": "spec_cascade_workspace_size", "clasp": "spec_clasp_workspace_size",
          "lm_head": "spec_lm_head_chain_workspace_size"}[kind]
    return int(getattr(L.lib(), fn)(*sizes))
