"""The C-ABI library loads on a CPU-only host and exports every symbol the
header declares; argument validation runs on the host before any launch."""
import ctypes
import os
import re

import pytest

from long_context_compressed_18_b300 import build, lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z][a-z0-9_]*)\s*\(", src, re.M)
    return sorted(set(names))


def test_header_declares_binding_exports():
    assert set(_declared()) == set(lib.EXPORTS)


def test_library_exports_every_declared_symbol():
    build.build()
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in _declared():
        assert hasattr(so, name), name


def test_host_side_validation_without_gpu():
    L = lib.load()
    # workspace queries are pure host arithmetic
    assert L.csa_topk_select_workspace_size(1, 4, 1000, 64) == 0
    assert L.csa_topk_select_workspace_size(32, 1, 262144, 1024) > 0
    assert L.csa_index_scores_workspace_size(1, 100, 128, lib.E2M1) > 0
    assert L.csa_index_scores_workspace_size(1, 100, 128, lib.E4M3) == 0
    # argument errors are reported before anything touches the device
    st = L.csa_compress(1, 16, 0, None, 1, None, None, None, None, None, None, None)
    assert st == 1 and "m=0" in L.csa_last_error().decode()
    st = L.csa_index_scores(1, 4, 0, 4, 8, 64, 128, None, lib.BF16, None, None, lib.E4M3, None,
                            None, None, 0, None)
    assert st == 2
    st = L.csa_index_scores(1, 4, 0, 4, 8, 32, 128, None, lib.BF16, None, None, lib.BF16, None,
                            None, None, 0, None)
    assert st == 2 and "H_I=64" in L.csa_last_error().decode()
    st = L.csa_topk_select(1, 1, 0, 1, 10, 0, None, None, None, 0, None)
    assert st == 2
    st = L.hca_attn(1, 1, 0, 4, 8, 12, 128, 0.1, None, None, None, lib.BF16, None, None, None)
    assert st == 2
    # the softmax scale must be positive and finite
    for bad in (0.0, -0.5, float("inf"), float("nan")):
        st = L.hca_attn(1, 1, 0, 4, 8, 64, 128, bad, None, None, None, lib.BF16, None, None, None)
        assert st == 1 and "scale" in L.csa_last_error().decode()
    # misaligned pointer
    st = L.swa_attn(1, 1, 0, 8, 4, 8, 64, 0.1, 8, 16, 16, lib.F32, 16, None, None)
    assert st == 3
