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


def check_attn_stagewise(got_o, got_l, want_o, want_l, mag, what=""):
    """Attention with BF16 I/O against the oracle run on identical inputs (the
    same K/V values and the same selection).  Gates:
      * max-abs 2e-2 (the spec's BF16 tolerance);
      * per element, the error the arithmetic allows: the probabilities enter
        the P.V product rounded to bf16 (relative 2^-9 each, at most
        2^-9 * sum_j p_j |v_j| / l = 2^-9 * mag, mag being the same attention
        over |V|) and the output is rounded to bf16 (2^-9 |o|); twice both;
      * the normalised error max|got - want| / max|want| <= 1e-2, which still
        bites where outputs are far below the absolute tolerance;
      * lse within 5e-5 + 5e-6 relative, -inf exactly where the set is empty.
    Returns the normalised error."""
    g = np.asarray(got_o, np.float64).reshape(want_o.shape)
    w = np.asarray(want_o, np.float64)
    assert_close(g, w, atol=2e-2, what=f"{what} (spec max-abs)")
    err = np.abs(g - w)
    bound = 2.0 ** -8 * (np.abs(np.asarray(mag).reshape(w.shape)) + np.abs(w)) + 1e-6
    assert np.all(err <= bound), f"{what}: worst excess over the per-element bound {np.max(err - bound):.3g}"
    top = float(np.max(np.abs(w))) if w.size else 0.0
    norm = float(err.max() / top) if top > 0 else 0.0
    assert norm <= 1e-2, f"{what}: normalised error {norm:.3g}"
    if got_l is not None:
        check_lse(got_l, want_l, what)
    return norm


def check_lse(got_l, want_l, what=""):
    """lse within 5e-5 + 5e-6 relative; -inf exactly where the key set is empty."""
    gl = np.asarray(got_l, np.float64).reshape(want_l.shape)
    fin = np.isfinite(want_l)
    assert np.array_equal(np.isfinite(gl), fin) and np.all(gl[~fin] < 0), what
    assert_close(gl[fin], want_l[fin], atol=5e-5, rtol=5e-6, what=f"{what} lse")


def check_e2m1_keys(packed, sc_codes, x64):
    """FP4 indexer keys from the compression epilogue against the oracle's
    fp64 compressed values x64 [R, d]: each block scale lies within one E4M3
    step of amax/6 (raised to the smallest positive E4M3), and each dequantised
    element e * sc within half an E2M1 step (times sc) of x, or within
    |x| - 6 sc where x / sc saturates.  Bit equality is not required: the GPU
    quantises its fp32 compressed value, which may sit on the other side of a
    rounding boundary from the fp64 one."""
    vals = oracle.e2m1_decode_packed(packed).astype(np.float64)
    sc = oracle.e4m3_decode(sc_codes).astype(np.float64)
    R, d = x64.shape
    nb = d // 32
    xb = x64.reshape(R, nb, 32)
    amax = np.abs(xb).max(-1)
    target = np.maximum(amax / 6.0, 2.0 ** -9)
    assert np.all(np.abs(sc - target) <= 2.0 ** -3 * target + 2.0 ** -10), "block scale off by more than one E4M3 step"
    a = np.abs(xb) / sc[..., None]
    half_step = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0)) * sc[..., None]
    sat = np.maximum(np.abs(xb) - 6.0 * sc[..., None], 0.0)
    bound = np.maximum(half_step, sat) * (1 + 1e-6) + 1e-6 * np.abs(xb) + 1e-9
    err = np.abs(vals.reshape(R, nb, 32) * sc[..., None] - xb)
    assert np.all(err <= bound), f"E2M1 element off: worst excess {np.max(err - bound):.3g}"
