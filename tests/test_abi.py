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
                            None, 0, None, lib.F32, None, 0, None)
    assert st == 2
    st = L.csa_index_scores(1, 4, 0, 4, 8, 32, 128, None, lib.BF16, None, None, lib.BF16, None,
                            None, 0, None, lib.F32, None, 0, None)
    assert st == 2 and "H_I=64" in L.csa_last_error().decode()
    st = L.csa_topk_select(1, 1, 0, 1, 10, 0, None, lib.F32, None, None, 0, None)
    assert st == 2
    st = L.hca_attn(1, 1, 0, 4, 8, 12, 1, 128, 0.1, None, None, None, lib.BF16, None, None, None)
    assert st == 2
    # the softmax scale must be positive and finite
    for bad in (0.0, -0.5, float("inf"), float("nan")):
        st = L.hca_attn(1, 1, 0, 4, 8, 64, 1, 128, bad, None, None, None, lib.BF16, None, None, None)
        assert st == 1 and "scale" in L.csa_last_error().decode()
    # misaligned pointer
    st = L.swa_attn(1, 1, 0, 8, 4, 8, 1, 64, 0.1, 8, 16, 16, lib.F32, 16, None, None)
    assert st == 3


def test_empty_inputs_and_limits_without_gpu():
    """Empty calls succeed without touching the device; the documented limits
    are enforced on the host (fake, aligned device addresses are never used)."""
    import ctypes as C
    L = lib.load()
    P, I = C.c_void_p, C.c_int
    bf, e2 = (I * 1)(lib.BF16), (I * 1)(lib.E2M1)
    addr = (P * 1)(256)
    # compression: fewer tokens than one block, or no sequences, is an empty call
    assert L.csa_compress(1, 3, 4, None, 1, (P * 1)(None), bf, (I * 1)(128), (P * 1)(None), bf, None, None) == 0
    assert L.csa_compress(0, 64, 4, None, 1, (P * 1)(None), bf, (I * 1)(128), (P * 1)(None), bf, None, None) == 0
    # widths: a power of two in [8, 256], at least 32 for E2M1 outputs
    for d in (4, 24, 512):
        st = L.csa_compress(1, 16, 4, 256, 1, addr, bf, (I * 1)(d), addr, bf, None, None)
        assert st == 2 and "power of two" in L.csa_last_error().decode()
    st = L.csa_compress(1, 16, 4, 256, 1, addr, bf, (I * 1)(16), addr, e2, addr, None)
    assert st == 2 and "E2M1" in L.csa_last_error().decode()
    # top-k: k <= 4096, rows <= 524,288 entries, long rows need the workspace
    assert L.csa_topk_select(1, 1, 0, 4, 1000, 4097, 256, lib.F32, 256, None, 0, None) == 2
    assert L.csa_topk_select(1, 1, 0, 4, 524289, 16, 256, lib.F32, 256, None, 0, None) == 2
    need = L.csa_topk_select_workspace_size(2, 1, 262144, 1024)
    st = L.csa_topk_select(2, 1, 4 * 262144 - 1, 4, 262144, 1024, 256, lib.F32, 256, None, 0, None)
    assert st == 4 and str(need) in L.csa_last_error().decode()
    st = L.csa_topk_select(2, 1, 4 * 262144 - 1, 4, 262144, 1024, 256, lib.F32, 256, 256, need - 16, None)
    assert st == 4
    assert L.csa_topk_select(0, 1, 0, 4, 1000, 16, None, lib.F32, None, None, 0, None) == 0


def test_topk_row_count_is_checked_in_64_bits():
    """B * n_q beyond INT_MAX (or beyond the grid once a long row is split into
    chunks) is rejected on the host instead of wrapping around; the workspace
    query computes in 64 bits."""
    L = lib.load()
    B, n_q = 70000, 40000                        # 2.8e9 rows
    assert L.csa_topk_select(B, n_q, 0, 4, 1000, 16, 256, lib.F32, 256, None, 0, None) == 2
    assert "grid limit" in L.csa_last_error().decode()
    assert L.csa_topk_select_noalloc(B, n_q, 0, 4, 1000, 16, 256, 256, None) == 2
    # 2^27 long rows of 16 chunks each exceed INT_MAX CTAs
    assert L.csa_topk_select(1 << 14, 1 << 13, 4 * 524288 - 1, 4, 524288, 16, 256, lib.F32, 256, None, 0, None) == 2
    need = L.csa_topk_select_workspace_size(65536, 65536, 262144, 1024)
    assert need >= 65536 * 65536 * 8 * 4096      # no 32-bit wraparound
