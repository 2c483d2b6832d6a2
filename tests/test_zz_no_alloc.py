"""The allocation-free top-k entry point.

csa_topk_select_noalloc serves callers that cannot allocate device memory
(a plugin inside a runtime that owns all device memory, or a latency-critical
path that must not call cudaMalloc).  It must select exactly what
csa_topk_select selects with a caller workspace, call after call, although
every call reuses the same built-in scratch array.  This file is collected
last so that a run stopping at the first failure has run every other test."""
import numpy as np
import pytest
import torch

from long_context_compressed_18_b300 import inputs, lib

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _reference(B, n_q, q_pos0, m, Nc, k, scores):
    out = torch.empty(B * n_q, k, dtype=torch.int32, device=DEV)
    nbytes = lib.csa_topk_select_workspace_size(B, n_q, Nc, k)
    ws = lib.empty_workspace(nbytes)
    lib.csa_topk_select(B, n_q, q_pos0, m, Nc, k, scores, out, ws, nbytes)
    return out


def _noalloc(B, n_q, q_pos0, m, Nc, k, scores):
    out = torch.full((B * n_q, k), -7, dtype=torch.int32, device=DEV)
    lib.csa_topk_select_noalloc(B, n_q, q_pos0, m, Nc, k, scores, out)
    return out


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    cases = [
        # two-phase selection over 1M-context rows: the scratch is used
        dict(B=32, n_q=1, q_pos0=(1 << 20) - 1, m=4, Nc=262144, k=1024, seed=901, ties=0),
        # a second call with other rows and heavy ties, reusing the same scratch
        dict(B=5, n_q=1, q_pos0=(1 << 20) - 1, m=4, Nc=262144, k=1024, seed=902, ties=40),
        # a single-pass shape (no scratch needed) after the two above
        dict(B=2, n_q=9, q_pos0=4000, m=4, Nc=5000, k=64, seed=903, ties=0),
    ]
    assert lib.csa_topk_select_workspace_size(32, 1, 262144, 1024) <= lib.NOALLOC_SCRATCH_BYTES
    for c in cases:
        sc = inputs.random_scores(c["B"] * c["n_q"], c["Nc"], seed=c["seed"], tie_levels=c["ties"]).to(DEV)
        args = (c["B"], c["n_q"], c["q_pos0"], c["m"], c["Nc"], c["k"], sc)
        want = _reference(*args)
        got = _noalloc(*args)
        torch.cuda.synchronize()
        lib.csa_device_status()
        assert torch.equal(got, want), c       # integer output: bit-exact


def test_noalloc_rejects_selection_larger_than_scratch():
    # 63 rows of 262,144 entries fit the 4 MiB array; 64 do not
    assert lib.csa_topk_select_workspace_size(63, 1, 262144, 1024) <= lib.NOALLOC_SCRATCH_BYTES
    assert lib.csa_topk_select_workspace_size(64, 1, 262144, 1024) > lib.NOALLOC_SCRATCH_BYTES
    sc = torch.zeros(64, 262144, dtype=torch.float32, device=DEV)
    out = torch.empty(64, 1024, dtype=torch.int32, device=DEV)
    with pytest.raises(lib.CsaError) as e:
        lib.csa_topk_select_noalloc(64, 1, (1 << 20) - 1, 4, 262144, 1024, sc, out)
    assert e.value.status == 4 and "4 MiB" in str(e.value)
