"""Shared helpers of the GPU parity tests: device tensors, tolerance checks."""
import numpy as np
import torch

import oracle
from long_context_compressed_18_b300 import lib

DEV = "cuda"


def to_dev(t):
    return None if t is None else t.to(DEV).contiguous()


def host(t):
    return None if t is None else t.detach().cpu()


def assert_close(got, want, atol, rtol=0.0, what=""):
    """Element-wise |got - want| <= atol + rtol * |want| (float64), with a
    report of the worst element."""
    g = np.asarray(got, np.float64)
    w = np.asarray(want, np.float64)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    err = np.abs(g - w)
    bound = atol + rtol * np.abs(w)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} elements off; worst at {i}: "
                             f"got {g[i]}, want {w[i]}, |err| {err[i]:.3g} > {bound[i]:.3g}")
    return float(err.max()) if err.size else 0.0


def topk_near_tie_check(gpu_sel, ora_sel, scores64, lens, k, rel=1e-3):
    """Top-k sets must be identical except at near-ties: every element of the
    symmetric difference has an oracle score within rel * |s_k| of the oracle's
    k-th score s_k.  Returns the number of rows with a near-tie swap."""
    swaps = 0
    for r in range(gpu_sel.shape[0]):
        L = int(lens[r])
        c = min(k, L)
        g = gpu_sel[r]
        o = ora_sel[r]
        assert np.all(g[c:] == -1) and np.all(o[c:] == -1), r
        gs, os_ = set(g[:c].tolist()), set(o[:c].tolist())
        assert len(gs) == c and all(0 <= j < L for j in gs), r
        assert list(g[:c]) == sorted(g[:c]), r
        diff = gs ^ os_
        if not diff:
            continue
        row = scores64[r, :L]
        sk = np.sort(row)[::-1][c - 1]
        for j in diff:
            assert abs(row[j] - sk) <= rel * abs(sk), (r, j, row[j], sk)
        swaps += 1
    return swaps


def sync_status():
    torch.cuda.synchronize()
    lib.csa_device_status()
