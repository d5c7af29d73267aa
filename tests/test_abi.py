"""The C ABI without a GPU: the library builds and loads, exports every
symbol include/spec_verify.h declares, the ctypes structures match the C
layout, and argument errors are reported before anything is launched."""

import ctypes as C
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    from draft_verification_gb300 import _lib, build
    if shutil.which("nvcc") is None and not os.path.exists(build.lib_path()):
        pytest.skip("neither nvcc nor a built library is available")
    build.build()
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(spec_\w+)\s*\(", text, re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) == 19, names
    for n in names:
        assert hasattr(lib, n), n
    from draft_verification_gb300 import _lib
    assert sorted(_lib.SIGNATURES) == names


def test_struct_layout_matches_header(tmp_path):
    from draft_verification_gb300 import _lib
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    if shutil.which("gcc") is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("gcc or CUDA headers missing")
    structs = {"spec_chain_args": _lib.ChainArgs, "spec_tree_args": _lib.TreeArgs,
               "spec_cascade_args": _lib.CascadeArgs, "spec_compact_args": _lib.CompactArgs,
               "spec_pipeline_args": _lib.PipelineArgs, "spec_clasp_args": _lib.ClaspArgs,
               "spec_pipeline_async_args": _lib.PipelineAsyncArgs, "spec_lm_head_chain_args": _lib.LmHeadChainArgs}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "spec_verify.h"', "int main(void){"]
    for cname, py in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0;}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {}
    for line in out:
        if line:
            s, f, v = line.split()
            got[(s, f)] = int(v)
    for cname, py in structs.items():
        assert got[(cname, "size")] == C.sizeof(py), cname
        for f, _ in py._fields_:
            assert got[(cname, f)] == getattr(py, f).offset, (cname, f)


def test_status_strings(lib):
    from draft_verification_gb300 import _lib
    assert _lib.status_string(0) == "ok"
    assert "workspace" in _lib.status_string(-4)


def test_workspace_sizes(lib):
    # the chunk partials of the statistics kernel: 8 B per (sequence, row,
    # 8192-element chunk: the float32 chunk), rounded up to 256 B
    def size(B, rows, V):
        return (B * rows * -(-V // 8192) * 8 + 255) // 256 * 256

    assert lib.spec_chain_workspace_size(64, 5, 128256) == size(64, 11, 128256) == 90112
    assert lib.spec_tree_workspace_size(16, 64, 50257) == size(16, 128, 50257)
    assert lib.spec_cascade_workspace_size(128, 8, 4, 128256) == size(128, 21, 128256)
    assert lib.spec_chain_workspace_size(0, 5, 10) == 0


def _chain(**kw):
    from draft_verification_gb300 import _lib
    a = _lib.ChainArgs()
    a.B, a.gamma, a.V, a.ld = 2, 3, 100, 100
    a.dtype, a.mode, a.temperature = _lib.SPEC_BF16, _lib.SPEC_SAMPLE, 1.0
    fake = 0x10000  # never dereferenced: validation fails first, or no launch happens
    for f in ("target_logits", "draft_logits", "draft_tokens", "u", "v", "accept_len",
              "out_token", "workspace"):
        setattr(a, f, fake)
    a.workspace_bytes = 1 << 20
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,code", [
    ("B", 0, -1), ("V", 0, -1), ("ld", 50, -1), ("gamma", 33, -1), ("gamma", -1, -1),
    ("temperature", 0.0, -1), ("temperature", float("inf"), -1), ("dtype", 7, -2),
    ("mode", 5, -2), ("target_logits", 0x10002, -3), ("draft_logits", 0x10008, -3),
    ("workspace_bytes", 8, -4), ("workspace", None, -4), ("accept_len", None, -1),
    ("u", None, -1),
])
def test_chain_argument_errors_are_reported_before_launch(lib, field, value, code):
    a = _chain(**{field: value})
    assert lib.spec_verify_chain(C.byref(a), None) == code


def test_consulted_only_is_sampling_only(lib):
    from draft_verification_gb300 import _lib
    # refused before anything touches the device (no control-word clear)
    a = _chain(mode=_lib.SPEC_GREEDY, consulted_only=1)
    assert lib.spec_verify_chain(C.byref(a), None) == -1
    a = _chain(gamma=0, consulted_only=1)
    assert lib.spec_verify_chain(C.byref(a), None) == -1


def test_tree_and_cascade_argument_errors(lib):
    from draft_verification_gb300 import _lib
    t = _lib.TreeArgs()
    t.B, t.N, t.max_depth, t.V, t.ld = 1, 1025, 3, 10, 10
    t.dtype, t.mode, t.temperature = 1, 1, 1.0
    assert lib.spec_verify_tree(C.byref(t), None) == -1
    t.N, t.max_depth = 8, 8  # max_depth > N - 1
    assert lib.spec_verify_tree(C.byref(t), None) == -1
    c = _lib.CascadeArgs()
    c.B, c.gamma1, c.gamma2, c.V, c.ld = 1, 4, 6, 10, 10  # gamma2 > gamma1 + 1
    c.dtype, c.mode, c.temperature = 1, 1, 1.0
    assert lib.spec_verify_cascade(C.byref(c), None) == -1
    assert lib.spec_verify_chain(None, None) == -1


def test_noalloc_chain_rejects_before_touching_the_device(lib):
    from draft_verification_gb300 import _lib
    assert lib.spec_verify_chain_noalloc(None, None) == -1
    assert lib.spec_verify_chain_noalloc(C.byref(_chain(B=0)), None) == -1
    assert lib.spec_verify_chain_noalloc(C.byref(_chain(gamma=33)), None) == -1
    # the static scratch is 8 MiB; a batch whose scratch exceeds it is refused
    assert _lib.SPEC_NOALLOC_SCRATCH_BYTES == 8 << 20
    big = _chain(B=4096, gamma=8, V=131072, ld=131072)
    assert lib.spec_chain_workspace_size(4096, 8, 131072) > _lib.SPEC_NOALLOC_SCRATCH_BYTES
    assert lib.spec_verify_chain_noalloc(C.byref(big), None) == -4
    assert lib.spec_chain_workspace_size(1024, 8, 131072) <= _lib.SPEC_NOALLOC_SCRATCH_BYTES


def test_each_kind_accepts_exactly_its_workspace_size(lib):
    # a workspace of exactly the reported size passes validation (the call
    # then fails at the launch: there is no GPU here), one byte less does not
    import torch
    if torch.cuda.is_available():
        pytest.skip("would launch on placeholder pointers")
    from draft_verification_gb300 import _lib
    fake = 0x10000
    a = _chain()
    a.workspace_bytes = lib.spec_chain_workspace_size(a.B, a.gamma, a.V)
    assert lib.spec_verify_chain(C.byref(a), None) == _lib.SPEC_ECUDA
    a.workspace_bytes -= 1
    assert lib.spec_verify_chain(C.byref(a), None) == -4

    t = _lib.TreeArgs()
    t.B, t.N, t.max_depth, t.V, t.ld = 2, 6, 3, 100, 100
    t.dtype, t.mode, t.temperature = _lib.SPEC_BF16, _lib.SPEC_SAMPLE, 1.0
    for f in ("parent", "node_tokens", "target_logits", "draft_logits", "u", "v", "path_len",
              "path_nodes", "out_token", "workspace"):
        setattr(t, f, fake)
    t.workspace_bytes = lib.spec_tree_workspace_size(t.B, t.N, t.V)
    assert lib.spec_verify_tree(C.byref(t), None) == _lib.SPEC_ECUDA
    t.workspace_bytes -= 1
    assert lib.spec_verify_tree(C.byref(t), None) == -4

    c = _lib.CascadeArgs()
    c.B, c.gamma1, c.gamma2, c.V, c.ld = 2, 4, 3, 100, 100
    c.dtype, c.mode, c.temperature = _lib.SPEC_BF16, _lib.SPEC_SAMPLE, 1.0
    for f in ("l0", "l1", "l2", "draft_tokens", "u1", "v1", "u2", "v2", "a1", "t1", "a2", "w2",
              "t2", "t2_valid", "r0", "r1", "committed", "workspace"):
        setattr(c, f, fake)
    c.workspace_bytes = lib.spec_cascade_workspace_size(c.B, c.gamma1, c.gamma2, c.V)
    assert lib.spec_verify_cascade(C.byref(c), None) == _lib.SPEC_ECUDA
    c.workspace_bytes -= 1
    assert lib.spec_verify_cascade(C.byref(c), None) == -4


def _compact(**kw):
    from draft_verification_gb300 import _lib
    a = _lib.CompactArgs()
    a.B, a.N, a.max_depth, a.cache_rows = 2, 8, 3, 16
    a.row_bytes, a.tree_ld, a.cache_ld = 64, 64, 64
    fake = 0x10000  # never dereferenced: every case fails validation
    for f in ("tree_rows", "cache", "path_nodes", "path_len"):
        setattr(a, f, fake)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value", [
    ("B", 0), ("B", 65536), ("N", 0), ("max_depth", -1), ("max_depth", 65535), ("cache_rows", 0),
    ("row_bytes", 0), ("tree_ld", 63), ("cache_ld", 32), ("tree_rows", None), ("cache", None),
    ("path_nodes", None), ("path_len", None),
])
def test_compact_argument_errors_are_reported_before_launch(lib, field, value):
    assert lib.spec_compact_tree_path(C.byref(_compact(**{field: value})), None) == -1
    assert lib.spec_compact_tree_path(None, None) == -1


def test_pipeline_argument_errors_and_workspace(lib):
    from draft_verification_gb300 import _lib
    win = (C.c_int * 7)(8, 6, 4)
    # rows M_0..M_3 = 8 + 9 + 6 + 4 (+1 with the final bonus)
    assert lib.spec_pipeline_workspace_size(128, 4, win, 0, 128256) == 256 * ((128 * 27 * 16 * 8 + 255) // 256)
    assert lib.spec_pipeline_workspace_size(128, 4, win, 1, 128256) == 256 * ((128 * 28 * 16 * 8 + 255) // 256)
    assert lib.spec_pipeline_workspace_size(128, 9, win, 0, 100) == 0
    bad = (C.c_int * 7)(8, 0, 4)
    assert lib.spec_pipeline_workspace_size(128, 4, bad, 0, 100) == 0

    def args(**kw):
        a = _lib.PipelineArgs()
        a.B, a.k, a.V, a.ld = 2, 4, 100, 100
        a.window = (C.c_int * 7)(3, 2, 2)
        a.dtype, a.mode, a.temperature = _lib.SPEC_BF16, _lib.SPEC_SAMPLE, 1.0
        fake = 0x10000
        for i in range(4):
            a.logits[i] = fake
        for i in range(3):
            a.u[i] = fake
            a.v[i] = fake
        for f in ("draft_tokens", "a", "w", "t", "t_valid", "r", "committed", "workspace"):
            setattr(a, f, fake)
        a.workspace_bytes = 1 << 20
        for key, v in kw.items():
            setattr(a, key, v)
        return a

    for kw, code in [(dict(k=1), -1), (dict(k=9), -1), (dict(B=0), -1), (dict(window=(C.c_int * 7)(3, 33, 2)), -1),
                     (dict(temperature=0.0), -1), (dict(dtype=5), -2), (dict(committed=None), -1),
                     (dict(workspace_bytes=8), -4)]:
        assert lib.spec_verify_pipeline(C.byref(args(**kw)), None) == code, kw
    a = args()
    a.logits[2] = None
    assert lib.spec_verify_pipeline(C.byref(a), None) == -1
    a = args()
    a.logits[1] = 0x10002
    assert lib.spec_verify_pipeline(C.byref(a), None) == -3
    a = args()
    a.u[2] = None
    assert lib.spec_verify_pipeline(C.byref(a), None) == -1
    assert lib.spec_verify_pipeline(None, None) == -1


def _clasp(**kw):
    from draft_verification_gb300 import _lib
    a = _lib.ClaspArgs()
    a.B, a.L, a.d, a.M = 2, 4, 64, 2
    fake = 0x10000  # 256-byte aligned, never dereferenced
    for f in ("hidden", "weights", "skip_mask", "score", "workspace"):
        setattr(a, f, fake)
    a.workspace_bytes = 1 << 30
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_clasp_workspace_size(lib):
    B, L, d, M = 16, 32, 4096, 12
    cells = (M + 1) * B * d

    def r(x):
        return 256 * ((x + 255) // 256)
    want = 2 * r(4 * cells) + r(2 * 2 * cells) + r(2 * 4 * cells) + r(L * (M + 1) * B) + (32 << 20)
    assert lib.spec_clasp_workspace_size(B, L, d, M) == want
    for bad in [(0, 4, 64, 2), (65536, 4, 64, 2), (2, 0, 64, 2), (2, 4097, 64, 2), (2, 4, 60, 2), (2, 4, 0, 2),
                (2, 4, 65544, 2), (2, 4, 64, -1), (2, 4, 64, 5)]:
        assert lib.spec_clasp_workspace_size(*bad) == 0, bad
    assert lib.spec_clasp_workspace_size(2, 4, 64, 4) > 0  # M = L: skip every layer
    assert lib.spec_clasp_workspace_size(2, 4, 64, 0) > 0  # M = 0: keep every layer


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), -1), (dict(L=0), -1), (dict(d=12), -1), (dict(M=5), -1), (dict(M=-1), -1),
    (dict(hidden=None), -1), (dict(weights=None), -1), (dict(skip_mask=None), -1), (dict(score=None), -1),
    (dict(hidden=0x10004), -3), (dict(weights=0x10008), -3),
    (dict(workspace=None), -4), (dict(workspace_bytes=1024), -4), (dict(workspace=0x10010), -4),
])
def test_clasp_argument_errors_are_reported_before_launch(lib, kw, code):
    assert lib.spec_clasp_layer_select(C.byref(_clasp(**kw)), None) == code
    assert lib.spec_clasp_layer_select(None, None) == -1


def test_clasp_accepts_exactly_its_workspace_size(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("would launch on placeholder pointers")
    from draft_verification_gb300 import _lib
    a = _clasp()
    a.workspace_bytes = lib.spec_clasp_workspace_size(a.B, a.L, a.d, a.M)
    assert lib.spec_clasp_layer_select(C.byref(a), None) == _lib.SPEC_ECUDA  # no GPU here
    a.workspace_bytes -= 1
    assert lib.spec_clasp_layer_select(C.byref(a), None) == -4


def _async(**kw):
    from draft_verification_gb300 import _lib
    a = _lib.PipelineAsyncArgs()
    a.B, a.k, a.V, a.ld = 2, 4, 100, 100
    a.window = (C.c_int * 7)(3, 2, 2)
    a.dtype, a.mode, a.temperature = _lib.SPEC_BF16, _lib.SPEC_SAMPLE, 1.0
    fake = 0x10000  # never dereferenced: every case fails validation
    for i in range(3):
        for arr in (a.target, a.draft, a.tokens, a.u, a.v):
            arr[i] = fake
    for f in ("length", "a", "t", "t_valid", "r", "committed", "workspace"):
        setattr(a, f, fake)
    a.workspace_bytes = 1 << 20
    for key, v in kw.items():
        setattr(a, key, v)
    return a


def test_pipeline_async_workspace_and_argument_errors(lib):
    from draft_verification_gb300 import _lib
    win = (C.c_int * 7)(8, 6, 4)
    chain = lib.spec_chain_workspace_size(128, 8, 128256)  # the largest stage's chain workspace
    scratch = 256 * ((3 * 3 * 128 * 4 + 255) // 256)
    assert lib.spec_pipeline_async_workspace_size(128, 4, win, 128256) == 256 * ((chain + 255) // 256) + scratch
    assert lib.spec_pipeline_async_workspace_size(128, 9, win, 100) == 0
    assert lib.spec_pipeline_async_workspace_size(128, 1, win, 100) == 0
    assert lib.spec_pipeline_async_workspace_size(0, 4, win, 100) == 0
    assert lib.spec_pipeline_async_workspace_size(128, 4, (C.c_int * 7)(8, 0, 4), 100) == 0
    assert lib.spec_pipeline_async_workspace_size(128, 4, (C.c_int * 7)(8, 33, 4), 100) == 0
    for kw, code in [(dict(k=1), -1), (dict(k=9), -1), (dict(B=0), -1), (dict(window=(C.c_int * 7)(3, 33, 2)), -1),
                     (dict(dtype=5), -2), (dict(mode=3), -2), (dict(committed=None), -1), (dict(length=None), -1),
                     (dict(workspace_bytes=8), -4), (dict(workspace=0x10008), -4)]:
        assert lib.spec_verify_pipeline_async(C.byref(_async(**kw)), None) == code, kw
    # checks every stage's chain call would make, made before any launch
    for kw, code in [(dict(V=2097153, ld=2097153), -1), (dict(ld=99), -1), (dict(temperature=0.0), -1),
                     (dict(temperature=float("inf")), -1)]:
        assert lib.spec_verify_pipeline_async(C.byref(_async(**kw)), None) == code, kw
    for field in ("target", "draft"):
        a = _async()
        getattr(a, field)[2] = 0x10008  # the last stage's rows misaligned
        assert lib.spec_verify_pipeline_async(C.byref(a), None) == -3, field
    for field in ("target", "tokens", "draft", "u", "v"):
        a = _async()
        getattr(a, field)[2] = None
        assert lib.spec_verify_pipeline_async(C.byref(a), None) == -1, field
    # greedy mode needs no draft rows or uniforms
    a = _async(mode=_lib.SPEC_GREEDY)
    for i in range(3):
        a.draft[i] = a.u[i] = a.v[i] = None
    a.workspace_bytes = 8
    assert lib.spec_verify_pipeline_async(C.byref(a), None) == -4
    assert lib.spec_verify_pipeline_async(None, None) == -1


def test_lm_head_argument_errors_and_workspace(lib):
    from draft_verification_gb300 import _lib
    sampling = lib.spec_lm_head_chain_workspace_size(64, 5, 128256, _lib.SPEC_SAMPLE)
    greedy = lib.spec_lm_head_chain_workspace_size(64, 5, 128256, _lib.SPEC_GREEDY)
    ldl = 128256
    part = 64 * 11 * 256 * 8
    assert sampling == part + 64 * 6 * ldl * 4 + 64 * 5 * ldl * 4  # every part already 256-aligned
    assert greedy == -(-64 * 6 * 256 * 8 // 256) * 256
    assert lib.spec_lm_head_chain_workspace_size(0, 5, 100, _lib.SPEC_SAMPLE) == 0
    assert lib.spec_lm_head_chain_workspace_size(4, 33, 100, _lib.SPEC_SAMPLE) == 0
    # the layout the binding's logits views assume: two partial columns per
    # 256-entry vocabulary tile (at most 256), then the target and draft rows
    # with a row stride of V rounded up to 8, each part rounded up to 256 B
    for B, g, V in ((6, 4, 9000), (5, 3, 5000), (3, 4, 1000), (2, 0, 100), (7, 2, 257), (64, 5, 128256)):
        up = lambda n: -(-n // 256) * 256
        chunks = min(2 * ((V + 255) // 256), 256)
        ldl = (V + 7) // 8 * 8
        part = up(B * (2 * g + 1) * chunks * 8)
        assert lib.spec_lm_head_chain_workspace_size(B, g, V, _lib.SPEC_SAMPLE) == \
            part + up(B * (g + 1) * ldl * 4) + up(B * g * ldl * 4), (B, g, V)
        assert lib.spec_lm_head_chain_workspace_size(B, g, V, _lib.SPEC_GREEDY) == up(B * (g + 1) * chunks * 8)

    def args(**kw):
        a = _lib.LmHeadChainArgs()
        a.B, a.gamma, a.V, a.d_target, a.d_draft = 2, 3, 1000, 64, 64
        a.mode, a.temperature = _lib.SPEC_SAMPLE, 1.0
        for name in ("h_target", "h_draft", "w_target", "w_draft", "draft_tokens", "u", "v", "accept_len",
                     "out_token", "workspace"):
            setattr(a, name, 4096)
        a.workspace_bytes = 1 << 30
        for k, v in kw.items():
            setattr(a, k, v)
        return a

    cases = [(dict(d_target=60), _lib.SPEC_EINVAL), (dict(d_draft=0), _lib.SPEC_EINVAL),
             (dict(V=0), _lib.SPEC_EINVAL), (dict(gamma=33), _lib.SPEC_EINVAL),
             (dict(temperature=0.0), _lib.SPEC_EINVAL), (dict(w_target=None), _lib.SPEC_EINVAL),
             (dict(h_draft=None), _lib.SPEC_EINVAL), (dict(mode=7), _lib.SPEC_EDTYPE),
             (dict(h_target=4097), _lib.SPEC_EALIGN), (dict(w_draft=4104), _lib.SPEC_EALIGN),
             (dict(workspace_bytes=16), _lib.SPEC_EWORKSPACE), (dict(workspace=4096 + 128), _lib.SPEC_EWORKSPACE)]
    for kw, code in cases:
        assert lib.spec_verify_chain_lm_head(C.byref(args(**kw)), None) == code, kw
