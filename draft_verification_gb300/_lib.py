"""ctypes view of the C ABI declared in include/spec_verify.h.

Argument marshalling only: the structures below mirror the C structs field
for field, and ``lib()`` loads the in-tree libspecverify.so.  There is no
fallback: if the library is missing or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes as C
import os

from .build import lib_path

SPEC_OK, SPEC_EINVAL, SPEC_EDTYPE, SPEC_EALIGN, SPEC_EWORKSPACE, SPEC_ECUDA = 0, -1, -2, -3, -4, -5
SPEC_F32, SPEC_BF16 = 0, 1
SPEC_GREEDY, SPEC_SAMPLE = 0, 1
SPEC_NOALLOC_SCRATCH_BYTES = 8 << 20
ERR_TOKEN, ERR_PARENT, ERR_NONFINITE, ERR_ZERO_MASS, ERR_INTERNAL, ERR_WINDOW = 1, 2, 4, 8, 16, 32

_vp = C.c_void_p


class ChainArgs(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("gamma", C.c_int), ("V", C.c_int), ("ld", C.c_longlong),
        ("dtype", C.c_int), ("mode", C.c_int), ("temperature", C.c_float),
        ("target_logits", _vp), ("draft_logits", _vp), ("draft_tokens", _vp),
        ("u", _vp), ("v", _vp), ("prefix_len", _vp),
        ("accept_len", _vp), ("out_token", _vp), ("rollback_idx", _vp),
        ("p_at_draft", _vp), ("q_at_draft", _vp), ("resid_mass", _vp),
        ("seq_error", _vp), ("error_word", _vp),
        ("workspace", _vp), ("workspace_bytes", C.c_size_t),
        ("consulted_only", C.c_int)
    ]


class TreeArgs(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("N", C.c_int), ("max_depth", C.c_int), ("V", C.c_int),
        ("ld", C.c_longlong), ("dtype", C.c_int), ("mode", C.c_int),
        ("temperature", C.c_float),
        ("parent", _vp), ("node_tokens", _vp), ("target_logits", _vp),
        ("draft_logits", _vp), ("u", _vp), ("v", _vp), ("prefix_len", _vp),
        ("path_len", _vp), ("path_nodes", _vp), ("out_token", _vp),
        ("rollback_idx", _vp), ("seq_error", _vp), ("error_word", _vp),
        ("workspace", _vp), ("workspace_bytes", C.c_size_t),
        ("consulted_only", C.c_int)
    ]


class CascadeArgs(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("gamma1", C.c_int), ("gamma2", C.c_int), ("V", C.c_int),
        ("ld", C.c_longlong), ("dtype", C.c_int), ("mode", C.c_int),
        ("temperature", C.c_float),
        ("l0", _vp), ("l1", _vp), ("l2", _vp), ("draft_tokens", _vp),
        ("u1", _vp), ("v1", _vp), ("u2", _vp), ("v2", _vp),
        ("base0", _vp), ("base1", _vp),
        ("a1", _vp), ("t1", _vp), ("a2", _vp), ("w2", _vp), ("t2", _vp),
        ("t2_valid", _vp), ("r0", _vp), ("r1", _vp), ("committed", _vp),
        ("seq_error", _vp), ("error_word", _vp),
        ("workspace", _vp), ("workspace_bytes", C.c_size_t)
    ]


SPEC_MAX_MODELS = 8


class PipelineArgs(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("k", C.c_int), ("window", C.c_int * (SPEC_MAX_MODELS - 1)), ("final_bonus", C.c_int),
        ("V", C.c_int), ("ld", C.c_longlong), ("dtype", C.c_int), ("mode", C.c_int),
        ("temperature", C.c_float),
        ("logits", _vp * SPEC_MAX_MODELS), ("draft_tokens", _vp),
        ("u", _vp * (SPEC_MAX_MODELS - 1)), ("v", _vp * (SPEC_MAX_MODELS - 1)), ("base", _vp),
        ("a", _vp), ("w", _vp), ("t", _vp), ("t_valid", _vp), ("r", _vp), ("committed", _vp),
        ("seq_error", _vp), ("error_word", _vp),
        ("workspace", _vp), ("workspace_bytes", C.c_size_t)
    ]


class PipelineAsyncArgs(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("k", C.c_int), ("window", C.c_int * (SPEC_MAX_MODELS - 1)), ("final_bonus", C.c_int),
        ("V", C.c_int), ("ld", C.c_longlong), ("dtype", C.c_int), ("mode", C.c_int),
        ("temperature", C.c_float),
        ("target", _vp * (SPEC_MAX_MODELS - 1)), ("draft", _vp * (SPEC_MAX_MODELS - 1)),
        ("tokens", _vp * (SPEC_MAX_MODELS - 1)), ("u", _vp * (SPEC_MAX_MODELS - 1)),
        ("v", _vp * (SPEC_MAX_MODELS - 1)), ("length", _vp),
        ("a", _vp), ("t", _vp), ("t_valid", _vp), ("r", _vp), ("committed", _vp),
        ("seq_error", _vp), ("error_word", _vp),
        ("workspace", _vp), ("workspace_bytes", C.c_size_t)
    ]


class LmHeadChainArgs(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("gamma", C.c_int), ("V", C.c_int), ("d_target", C.c_int), ("d_draft", C.c_int),
        ("mode", C.c_int), ("temperature", C.c_float),
        ("h_target", _vp), ("h_draft", _vp), ("w_target", _vp), ("w_draft", _vp),
        ("draft_tokens", _vp), ("u", _vp), ("v", _vp), ("prefix_len", _vp),
        ("accept_len", _vp), ("out_token", _vp), ("rollback_idx", _vp),
        ("p_at_draft", _vp), ("q_at_draft", _vp), ("resid_mass", _vp),
        ("seq_error", _vp), ("error_word", _vp),
        ("workspace", _vp), ("workspace_bytes", C.c_size_t)
    ]


class CompactArgs(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("N", C.c_int), ("max_depth", C.c_int), ("cache_rows", C.c_int),
        ("row_bytes", C.c_longlong), ("tree_ld", C.c_longlong), ("cache_ld", C.c_longlong),
        ("tree_rows", _vp), ("cache", _vp), ("path_nodes", _vp), ("path_len", _vp),
        ("prefix_len", _vp), ("seq_error", _vp), ("error_word", _vp)
    ]


class ClaspArgs(C.Structure):
    _fields_ = [
        ("B", C.c_int), ("L", C.c_int), ("d", C.c_int), ("M", C.c_int),
        ("hidden", _vp), ("weights", _vp), ("skip_mask", _vp), ("score", _vp), ("choice", _vp),
        ("workspace", _vp), ("workspace_bytes", C.c_size_t)
    ]


# every symbol include/spec_verify.h declares, with its ctypes signature
SIGNATURES = {
    "spec_chain_workspace_size": (C.c_size_t, [C.c_int, C.c_int, C.c_int]),
    "spec_verify_chain": (C.c_int, [C.POINTER(ChainArgs), _vp]),
    "spec_verify_chain_noalloc": (C.c_int, [C.POINTER(ChainArgs), _vp]),
    "spec_tree_workspace_size": (C.c_size_t, [C.c_int, C.c_int, C.c_int]),
    "spec_verify_tree": (C.c_int, [C.POINTER(TreeArgs), _vp]),
    "spec_cascade_workspace_size": (C.c_size_t, [C.c_int, C.c_int, C.c_int, C.c_int]),
    "spec_verify_cascade": (C.c_int, [C.POINTER(CascadeArgs), _vp]),
    "spec_pipeline_workspace_size": (C.c_size_t, [C.c_int, C.c_int, C.POINTER(C.c_int), C.c_int, C.c_int]),
    "spec_verify_pipeline": (C.c_int, [C.POINTER(PipelineArgs), _vp]),
    "spec_compact_tree_path": (C.c_int, [C.POINTER(CompactArgs), _vp]),
    "spec_pipeline_async_workspace_size": (C.c_size_t, [C.c_int, C.c_int, C.POINTER(C.c_int), C.c_int]),
    "spec_verify_pipeline_async": (C.c_int, [C.POINTER(PipelineAsyncArgs), _vp]),
    "spec_clasp_workspace_size": (C.c_size_t, [C.c_int, C.c_int, C.c_int, C.c_int]),
    "spec_clasp_layer_select": (C.c_int, [C.POINTER(ClaspArgs), _vp]),
    "spec_status_string": (C.c_char_p, [C.c_int]),
    "spec_test_inject_copy_timeout": (C.c_int, [C.c_int]),
    "spec_test_inject_head_copy_timeout": (C.c_int, [C.c_int]),
    "spec_lm_head_chain_workspace_size": (C.c_size_t, [C.c_int, C.c_int, C.c_int, C.c_int]),
    "spec_verify_chain_lm_head": (C.c_int, [C.POINTER(LmHeadChainArgs), _vp]),
}

_LIB = None


def lib() -> C.CDLL:
    """Load libspecverify.so (built by draft_verification_gb300.build)."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m draft_verification_gb300.build` "
                "(there is no CPU fallback)")
        handle = C.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def status_string(code: int) -> str:
    return lib().spec_status_string(code).decode()
