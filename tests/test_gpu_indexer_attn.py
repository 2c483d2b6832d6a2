"""GPU parity: indexer scores (fp32 CUDA cores; BF16 / E4M3 / E2M1 on tcgen05)
and attention (sparse / closed-block / window), against the oracle on
identical inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
from long_context_compressed_18_b300 import configs, inputs, lib
from helpers import DEV, assert_close, host, sync_status

pytestmark = pytest.mark.gpu


def _index_inputs(B, n_q, Nc, HI, dI, q_dt, k_dt, seed):
    g = torch.Generator().manual_seed(seed)
    qf = torch.randn(B, n_q, HI, dI, generator=g)
    kf = torch.randn(B, Nc, dI, generator=g)
    if q_dt == "f32":
        q, qs, qc = qf, None, lib.F32
    elif q_dt == "bf16":
        q, qs, qc = qf.to(torch.bfloat16), None, lib.BF16
    else:
        (q, qs), qc = inputs.quantise_e4m3_lastdim(qf), lib.E4M3
    if k_dt == "f32":
        k, ks, kc = kf, None, lib.F32
    elif k_dt == "bf16":
        k, ks, kc = kf.to(torch.bfloat16), None, lib.BF16
    elif k_dt == "e4m3":
        (k, ks), kc = inputs.quantise_e4m3_lastdim(kf), lib.E4M3
    else:
        (k, ks), kc = inputs.random_e2m1_keys(B, Nc, dI, seed + 1), lib.E2M1
    return q, qs, qc, k, ks, kc


def _oracle_values(q, qs, q_dt, k, ks, k_dt):
    qv = oracle.e4m3_decode(q) if q_dt == "e4m3" else host(q).float().numpy()
    if k_dt == "e2m1":
        x8, S, _ = oracle.fp4_to_e4m3(k, ks)
        kv, kscale = oracle.e4m3_decode(x8), S
    elif k_dt == "e4m3":
        kv, kscale = oracle.e4m3_decode(k), host(ks).numpy()
    else:
        kv, kscale = host(k).float().numpy(), None
    return qv, (None if qs is None else host(qs).numpy()), kv, kscale


INDEX_CASES = [
    dict(B=2, n_q=40, q_pos0=100, m=4, Nc=80, HI=4, dI=32, q_dt="f32", k_dt="f32"),
    dict(B=2, n_q=13, q_pos0=3000, m=4, Nc=1000, HI=64, dI=128, q_dt="bf16", k_dt="bf16"),
    dict(B=1, n_q=530, q_pos0=0, m=1, Nc=530, HI=64, dI=128, q_dt="bf16", k_dt="bf16"),
    dict(B=3, n_q=1, q_pos0=4 * 6000 - 1, m=4, Nc=6000, HI=64, dI=128, q_dt="e4m3", k_dt="e4m3"),
    dict(B=1, n_q=65, q_pos0=1000, m=4, Nc=400, HI=64, dI=128, q_dt="e4m3", k_dt="e4m3"),
    dict(B=2, n_q=9, q_pos0=2000, m=4, Nc=700, HI=64, dI=128, q_dt="e4m3", k_dt="e2m1"),
    dict(B=3, n_q=1, q_pos0=4 * 6001 - 1, m=4, Nc=6001, HI=64, dI=128, q_dt="e4m3", k_dt="e2m1"),   # widened in-kernel
    dict(B=2, n_q=3, q_pos0=4 * 2000 - 3, m=4, Nc=2000, HI=64, dI=128, q_dt="e4m3", k_dt="e2m1"),
    dict(B=2, n_q=1, q_pos0=4 * 3000 - 1, m=4, Nc=3000, HI=64, dI=128, q_dt="bf16", k_dt="bf16"),
]


@pytest.mark.parametrize("case", INDEX_CASES, ids=lambda c: f"{c['q_dt']}-{c['k_dt']}-B{c['B']}-nq{c['n_q']}-Nc{c['Nc']}")
def test_index_scores(case):
    c = dict(case)
    B, n_q, q_pos0, m, Nc, HI, dI = (c[x] for x in ("B", "n_q", "q_pos0", "m", "Nc", "HI", "dI"))
    q, qs, qc, k, ks, kc = _index_inputs(B, n_q, Nc, HI, dI, c["q_dt"], c["k_dt"], seed=Nc + n_q)
    scores = torch.full((B, n_q, Nc), float("nan"), dtype=torch.float32, device=DEV)
    wsb = lib.csa_index_scores_workspace_size(B, Nc, dI, kc)
    ws = lib.empty_workspace(wsb)
    lib.csa_index_scores(B, n_q, q_pos0, m, Nc, HI, dI, q.to(DEV), qc, None if qs is None else qs.to(DEV),
                         k.to(DEV), kc, None if ks is None else ks.to(DEV), scores, ws, wsb)
    sync_status()
    qv, qsv, kv, ksv = _oracle_values(q, qs, c["q_dt"], k, ks, c["k_dt"])
    s64, _ = oracle.index_scores(qv, qsv, kv, ksv, q_pos0, m)
    mag, _ = oracle.index_scores(np.abs(qv), None if qsv is None else np.abs(qsv), np.abs(kv),
                                 None if ksv is None else np.abs(ksv), q_pos0, m)
    got = host(scores).numpy().reshape(B * n_q, Nc)
    vis = np.isfinite(s64)
    assert np.all(np.isfinite(got[vis])), "visible score not written"
    rel = 2e-6 if c["q_dt"] == "f32" else 1e-5
    err = np.abs(got[vis] - s64[vis])
    bound = rel * mag[vis] + 1e-6
    worst = np.argmax(err - bound)
    assert np.all(err <= bound), (err[worst], bound[worst], got[vis][worst], s64[vis][worst])


def _attn_inputs(B, n_q, H, d, N_kv, dt, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    q = (torch.randn(B, n_q, H, d, generator=g) * scale).to(tdt)
    K = (torch.randn(B, N_kv, d, generator=g) * scale).to(tdt)
    V = torch.randn(B, N_kv, d, generator=g).to(tdt)
    return q, K, V


def _check_attn(out, lse, want_o, want_l, dt, mag=None):
    """BF16 I/O: besides the max-abs 2e-2 gate, each element is held to the
    error the arithmetic allows -- the probabilities P enter the P.V product
    rounded to bf16 (relative 2^-9 each, so at most 2^-9 * sum_j p_j |v_j| / l
    = 2^-9 * mag, mag being the same attention over |V|), and the output is
    rounded to bf16 (2^-9 |o|); the bound takes twice both."""
    got = host(out).float().numpy().reshape(want_o.shape)
    if dt == "bf16":
        assert_close(got, want_o, atol=2e-2, what="attn out (spec)")
        m = np.abs(want_o) if mag is None else mag.reshape(want_o.shape)
        err = np.abs(got - want_o)
        bound = 2.0 ** -8 * (m + np.abs(want_o)) + 1e-6
        assert np.all(err <= bound), f"attn out: worst excess {np.max(err - bound):.3g}"
    else:
        assert_close(got, want_o, atol=2e-5, rtol=2e-5, what="attn out")
    gl = host(lse).numpy().reshape(want_l.shape)
    fin = np.isfinite(want_l)
    assert np.array_equal(np.isfinite(gl), fin) and np.all(gl[~fin] < 0)
    assert_close(gl[fin], want_l[fin], atol=5e-5, rtol=5e-6, what="lse")


SPARSE_CASES = [
    dict(B=2, n_q=50, q_pos0=1000, m=4, N_c=400, k=128, H=64, d=128, dt="bf16"),
    dict(B=3, n_q=1, q_pos0=4 * 5000 - 1, m=4, N_c=5000, k=1024, H=64, d=128, dt="bf16"),   # split + combine
    # 128 heads (every MMA row used); 2 splits of 256 positions, the second
    # ragged; the sets hold 225 visible entries, then -1 padding
    dict(B=2, n_q=3, q_pos0=900, m=4, N_c=226, k=300, H=128, d=128, dt="bf16"),
    # eight 128-entry tiles per CTA (no split at n_q > 16): the gather ring wraps
    dict(B=1, n_q=20, q_pos0=4 * 3000 - 20, m=4, N_c=3000, k=1024, H=64, d=128, dt="bf16"),
    # ragged last tile (k = 200) with early queries that see few or no entries
    dict(B=1, n_q=40, q_pos0=0, m=4, N_c=100, k=200, H=64, d=128, dt="bf16"),
    # more query tokens than SMs, full sets of eight tiles; then from the start
    # of the context, so tokens with no, one or a few tiles follow one another
    dict(B=2, n_q=400, q_pos0=4 * 3000 - 400, m=4, N_c=3000, k=1024, H=64, d=128, dt="bf16"),
    dict(B=1, n_q=700, q_pos0=0, m=4, N_c=700, k=512, H=64, d=128, dt="bf16"),
    dict(B=1, n_q=100, q_pos0=0, m=4, N_c=256, k=64, H=8, d=64, dt="f32"),                  # short sets, -1 pads
    dict(B=2, n_q=2, q_pos0=300, m=1, N_c=301, k=200, H=32, d=64, dt="f32"),
]


@pytest.mark.parametrize("case", SPARSE_CASES, ids=lambda c: f"{c['dt']}-H{c['H']}-d{c['d']}-B{c['B']}-nq{c['n_q']}-k{c['k']}")
def test_sparse_attn(case):
    c = dict(case)
    s = configs.shape(kind="csa", B=c["B"], n=c["N_c"] * c["m"], m=c["m"], n_q=c["n_q"], q_pos0=c["q_pos0"],
                      H=c["H"], d=c["d"], k=c["k"])
    idx = inputs.random_index_sets(s, seed=c["N_c"])
    q, K, V = _attn_inputs(c["B"], c["n_q"], c["H"], c["d"], c["N_c"], c["dt"], seed=c["k"],
                           scale=c["d"] ** -0.25)
    tau = 1.0 / math.sqrt(c["d"])
    out = torch.empty_like(q, device=DEV)
    lse = torch.empty(c["B"], c["n_q"], c["H"], dtype=torch.float32, device=DEV)
    wsb = lib.csa_sparse_attn_workspace_size(c["B"], c["n_q"], c["H"], c["d"], c["k"])
    ws = lib.empty_workspace(wsb)
    dtc = lib.F32 if c["dt"] == "f32" else lib.BF16
    lib.csa_sparse_attn(c["B"], c["n_q"], c["H"], c["d"], c["N_c"], c["k"], tau, q.to(DEV), K.to(DEV), V.to(DEV),
                        dtc, idx.to(DEV), out, lse, ws, wsb)
    sync_status()
    wo, wl = oracle.attention(q, K, V, tau, oracle.SPARSE, idx=idx)
    mag, _ = oracle.attention(q, K, V.float().abs(), tau, oracle.SPARSE, idx=idx)
    _check_attn(out, lse, wo.reshape(q.shape), wl.reshape(lse.shape), c["dt"], mag)


DENSE_CASES = [
    dict(mode="hca", B=1, n_q=300, q_pos0=0, m=4, N=80, H=64, d=128, dt="bf16", window=0),
    dict(mode="hca", B=2, n_q=40, q_pos0=128 * 60 - 20, m=128, N=64, H=64, d=128, dt="bf16", window=0),
    dict(mode="hca", B=1, n_q=64, q_pos0=0, m=1, N=64, H=8, d=64, dt="f32", window=0),
    dict(mode="swa", B=1, n_q=600, q_pos0=0, m=1, N=600, H=64, d=128, dt="bf16", window=128),
    dict(mode="swa", B=2, n_q=301, q_pos0=0, m=1, N=301, H=64, d=128, dt="bf16", window=100),   # odd tail
    dict(mode="hca", B=2, n_q=33, q_pos0=4000, m=4, N=1010, H=128, d=128, dt="bf16", window=0),
    dict(mode="swa", B=1, n_q=20, q_pos0=500, m=1, N=520, H=128, d=128, dt="bf16", window=300),
    dict(mode="swa", B=2, n_q=70, q_pos0=0, m=1, N=70, H=16, d=64, dt="f32", window=1000),
]


@pytest.mark.parametrize("case", DENSE_CASES, ids=lambda c: f"{c['mode']}-{c['dt']}-m{c['m']}-nq{c['n_q']}-W{c['window']}")
def test_dense_attn(case):
    c = dict(case)
    q, K, V = _attn_inputs(c["B"], c["n_q"], c["H"], c["d"], c["N"], c["dt"], seed=c["n_q"], scale=c["d"] ** -0.25)
    tau = 1.0 / math.sqrt(c["d"])
    out = torch.empty_like(q, device=DEV)
    lse = torch.empty(c["B"], c["n_q"], c["H"], dtype=torch.float32, device=DEV)
    dtc = lib.F32 if c["dt"] == "f32" else lib.BF16
    if c["mode"] == "hca":
        lib.hca_attn(c["B"], c["n_q"], c["q_pos0"], c["m"], c["N"], c["H"], c["d"], tau, q.to(DEV), K.to(DEV),
                     V.to(DEV), dtc, out, lse)
        kw = dict(mode=oracle.CLOSED_BLOCKS, q_pos0=c["q_pos0"], m=c["m"])
    else:
        lib.swa_attn(c["B"], c["n_q"], c["q_pos0"], c["N"], c["window"], c["H"], c["d"], tau, q.to(DEV), K.to(DEV),
                     V.to(DEV), dtc, out, lse)
        kw = dict(mode=oracle.WINDOW, q_pos0=c["q_pos0"], window=c["window"])
    wo, wl = oracle.attention(q, K, V, tau, **kw)
    mag, _ = oracle.attention(q, K, V.float().abs(), tau, **kw)
    sync_status()
    _check_attn(out, lse, wo.reshape(q.shape), wl.reshape(lse.shape), c["dt"], mag)
