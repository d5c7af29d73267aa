"""The alignment-checking debug build (build(debug_checks=True)) compiles for
sm_103a, links, and exports the same C ABI; its kernels replace every
misaligned 16-byte load, bulk copy, L2 prefetch or tensor-map copy by an
error report (no GPU needed for this check)."""

import ctypes as C
import os
import shutil

import pytest


def test_debug_checks_build_exports_the_abi():
    from draft_verification_gb300 import _lib, build
    if shutil.which("nvcc") is None:
        pytest.skip("nvcc is not available")
    path = build.build(debug_checks=True)
    assert path == build.lib_path(True) and path != build.lib_path(False)
    assert os.path.exists(path)
    handle = C.CDLL(path)
    for name in _lib.SIGNATURES:
        assert hasattr(handle, name), name
