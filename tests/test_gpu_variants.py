"""GPU parity of the variant readings against the oracle's switches:
per-channel compression weights, the weighted / ReLU Lightning Indexer, and
GQA / MHA KV heads in the three attention calls."""
import math

import numpy as np
import pytest
import torch

import oracle
from long_context_compressed_18_b300 import inputs, lib
from helpers import DEV, assert_close, check_lse, host, sync_status, topk_near_tie_check

pytestmark = pytest.mark.gpu


# ---- per-channel compression weights ---------------------------------------

def _alloc(B, Nc, d, kind):
    if kind == lib.E4M3:
        return torch.empty(B, Nc, d, dtype=torch.uint8, device=DEV), torch.empty(B, Nc, device=DEV)
    if kind == lib.E2M1:
        return (torch.empty(B, Nc, d // 2, dtype=torch.uint8, device=DEV),
                torch.empty(B, Nc, d // 32, dtype=torch.uint8, device=DEV))
    return torch.empty(B, Nc, d, dtype=torch.float32 if kind == lib.F32 else torch.bfloat16, device=DEV), None


@pytest.mark.parametrize("m", [4, 128])
def test_per_channel_compression(m):
    g = torch.Generator().manual_seed(40 + m)
    B, Nc = 2, 301 if m == 4 else 13
    n = Nc * m + 3                                  # a ragged partial block at the end
    spec = [(torch.bfloat16, 128, lib.F32), (torch.float32, 64, lib.BF16), (torch.bfloat16, 128, lib.E4M3),
            (torch.bfloat16, 128, lib.E2M1)]
    xs = [torch.randn(B, n, d, generator=g).to(dt) for dt, d, _ in spec]
    lgs = [torch.randn(B, n, d, generator=g) * 2 for _, d, _ in spec]
    outs = [_alloc(B, Nc, d, k) for _, d, k in spec]
    lib.csa_compress_per_channel(B, n, m, [lg.to(DEV) for lg in lgs], [x.to(DEV) for x in xs],
                                 [lib.F32 if dt == torch.float32 else lib.BF16 for dt, _, _ in spec],
                                 [d for _, d, _ in spec], [o for o, _ in outs], [k for _, _, k in spec],
                                 [sc for _, sc in outs])
    sync_status()
    for (dt, d, kind), x, lg, (o, sc) in zip(spec, xs, lgs, outs):
        want = oracle.compress_per_channel(lg, x, m)
        if kind == lib.F32:
            assert_close(host(o).numpy(), want, atol=2e-6, rtol=2e-6, what=f"f32 m={m}")
        elif kind == lib.BF16:
            assert_close(host(o).float().numpy(), want, atol=1e-6, rtol=2.0 ** -8 + 1e-5, what=f"bf16 m={m}")
        elif kind == lib.E4M3:
            # per-row scale to 1e-6; dequantised values within one E4M3 step
            wc, ws = oracle.quant_e4m3_rows(want.astype(np.float32))
            assert_close(host(sc).numpy(), ws, atol=0, rtol=1e-6, what="e4m3 scales")
            dec = oracle.e4m3_decode(host(o).numpy()).astype(np.float64) * host(sc).numpy()[..., None]
            ref = oracle.e4m3_decode(wc).astype(np.float64) * ws[..., None]
            assert np.all(np.abs(dec - ref) <= (np.abs(ref) * 2.0 ** -3 + ws[..., None] * 2.0 ** -9) * 1.0001)
        else:
            from helpers import check_e2m1_keys
            check_e2m1_keys(host(o).numpy().reshape(-1, d // 2), host(sc).numpy().reshape(-1, d // 32),
                            want.reshape(-1, d))


# ---- weighted / ReLU indexer ---------------------------------------------------

def _idx(B, n_q, Nc, kind, seed):
    g = torch.Generator().manual_seed(seed)
    HI, dI = (64, 128) if kind != "f32" else (8, 32)
    qf, kf = torch.randn(B, n_q, HI, dI, generator=g), torch.randn(B, Nc, dI, generator=g)
    w = torch.randn(B, n_q, HI, generator=g)        # signed head weights
    if kind == "f32":
        return qf, lib.F32, None, kf, lib.F32, None, w, HI, dI
    if kind == "bf16":
        return qf.to(torch.bfloat16), lib.BF16, None, kf.to(torch.bfloat16), lib.BF16, None, w, HI, dI
    (q, qs), (k, ks) = inputs.quantise_e4m3_lastdim(qf), inputs.quantise_e4m3_lastdim(kf)
    return q, lib.E4M3, qs, k, lib.E4M3, ks, w, HI, dI


def _vals(t, code):
    return oracle.e4m3_decode(t) if code == lib.E4M3 else host(t).float().numpy()


@pytest.mark.parametrize("case", [
    dict(B=2, n_q=13, Nc=1000, kind="bf16"),
    dict(B=3, n_q=1, Nc=6000, kind="e4m3"),
    dict(B=1, n_q=9, Nc=700, kind="e4m3"),
    dict(B=2, n_q=20, Nc=90, kind="f32"),
])
@pytest.mark.parametrize("relu", [False, True])
def test_weighted_relu_index_scores(case, relu):
    B, n_q, Nc = case["B"], case["n_q"], case["Nc"]
    q_pos0 = 4 * Nc - n_q
    q, qc, qs, k, kc, ks, w, HI, dI = _idx(B, n_q, Nc, case["kind"], seed=Nc + n_q + relu)
    out = torch.full((B, n_q, Nc), float("nan"), device=DEV)
    lib.csa_index_scores(B, n_q, q_pos0, 4, Nc, HI, dI, q.to(DEV), qc, None if qs is None else qs.to(DEV),
                         k.to(DEV), kc, None if ks is None else ks.to(DEV), out, head_weight=w.to(DEV), relu=relu)
    sync_status()
    qv, kv = _vals(q, qc), _vals(k, kc)
    qsv = None if qs is None else host(qs).numpy()
    ksv = None if ks is None else host(ks).numpy()
    want, _ = oracle.index_scores(qv, qsv, kv, ksv, q_pos0, 4, head_w=w.numpy(), relu=relu)
    mag, _ = oracle.index_scores(np.abs(qv), None if qsv is None else np.abs(qsv), np.abs(kv),
                                 None if ksv is None else np.abs(ksv), q_pos0, 4, head_w=np.abs(w.numpy()))
    got = host(out).numpy().reshape(B * n_q, Nc)
    vis = np.isfinite(want)
    err = np.abs(got[vis] - want[vis])
    assert np.all(err <= (2e-6 if case["kind"] == "f32" else 1e-5) * mag[vis] + 1e-6), err.max()


def test_weighted_relu_index_topk_decode():
    """The fused decode route with head weights and ReLU: selection against
    the oracle's (near-ties only)."""
    B, Nc, k = 2, 60000, 1024
    q, qc, qs, kk, kc, ks, w, HI, dI = _idx(B, 1, Nc, "e4m3", seed=77)
    topk = torch.empty(B, 1, k, dtype=torch.int32, device=DEV)
    wb = lib.csa_index_topk_workspace_size(B, 1, Nc, HI, dI, k, kc)
    ws = lib.empty_workspace(wb)
    lib.csa_index_topk(B, 1, 4 * Nc - 1, 4, Nc, HI, dI, k, q.to(DEV), qc, qs.to(DEV), kk.to(DEV), kc, ks.to(DEV),
                       topk, ws, wb, head_weight=w.to(DEV), relu=True)
    sync_status()
    s64, _, sel = oracle.csa_index_topk(q, qs, "e4m3", kk, ks, "e4m3", 4 * Nc - 1, 4, k, head_w=w, relu=True)
    topk_near_tie_check(host(topk).numpy().reshape(B, k), sel, s64, [Nc] * B, k)


# ---- GQA / MHA KV heads ----------------------------------------------------------

KV_CASES = [
    dict(mode="sparse", B=2, n_q=5, H=8, H_kv=8, d=64, N=300, dt="f32"),       # MHA
    dict(mode="sparse", B=1, n_q=3, H=64, H_kv=4, d=128, N=3000, dt="bf16"),   # GQA, decode-like split
    dict(mode="hca", B=2, n_q=40, H=16, H_kv=2, d=64, N=50, dt="bf16"),
    dict(mode="swa", B=1, n_q=70, H=32, H_kv=8, d=128, N=70, dt="f32"),
    dict(mode="hca", B=1, n_q=20, H=4, H_kv=2, d=64, N=30, dt="f32"),          # two heads a KV head
]


@pytest.mark.parametrize("c", KV_CASES, ids=lambda c: f"{c['mode']}-H{c['H']}-kv{c['H_kv']}-{c['dt']}")
def test_kv_heads_attention(c):
    g = torch.Generator().manual_seed(c["N"] + c["H"])
    tdt = torch.float32 if c["dt"] == "f32" else torch.bfloat16
    dtc = lib.F32 if c["dt"] == "f32" else lib.BF16
    B, n_q, H, H_kv, d, N = c["B"], c["n_q"], c["H"], c["H_kv"], c["d"], c["N"]
    sc = d ** -0.25
    q = (torch.randn(B, n_q, H, d, generator=g) * sc).to(tdt)
    K = (torch.randn(B, N, H_kv, d, generator=g) * sc).to(tdt)
    V = torch.randn(B, N, H_kv, d, generator=g).to(tdt)
    tau = 1 / math.sqrt(d)
    out = torch.empty(B, n_q, H, d, dtype=tdt, device=DEV)
    lse = torch.empty(B, n_q, H, device=DEV)
    if c["mode"] == "sparse":
        k = 1024
        idx = torch.full((B, n_q, k), -1, dtype=torch.int32)
        for b in range(B):
            for i in range(n_q):
                cnt = min(k, N - i)
                idx[b, i, :cnt] = torch.randperm(N, generator=g)[:cnt].sort().values.to(torch.int32)
        wsb = lib.csa_sparse_attn_workspace_size(B, n_q, H, d, k)
        ws = lib.empty_workspace(wsb)
        lib.csa_sparse_attn(B, n_q, H, d, N, k, tau, q.to(DEV), K.to(DEV), V.to(DEV), dtc, idx.to(DEV), out, lse,
                            ws, wsb, H_kv=H_kv)
        kw = dict(mode=oracle.SPARSE, idx=idx)
    elif c["mode"] == "hca":
        q_pos0 = 4 * N - n_q
        lib.hca_attn(B, n_q, q_pos0, 4, N, H, d, tau, q.to(DEV), K.to(DEV), V.to(DEV), dtc, out, lse, H_kv=H_kv)
        kw = dict(mode=oracle.CLOSED_BLOCKS, q_pos0=q_pos0, m=4)
    else:
        lib.swa_attn(B, n_q, 0, N, 16, H, d, tau, q.to(DEV), K.to(DEV), V.to(DEV), dtc, out, lse, H_kv=H_kv)
        kw = dict(mode=oracle.WINDOW, q_pos0=0, window=16)
    sync_status()
    want_o, want_l = oracle.attention(q, K, V, tau, **kw)
    got = host(out).float().numpy().reshape(want_o.shape)
    if c["dt"] == "f32":
        assert_close(got, want_o, atol=2e-5, rtol=2e-5, what="gqa attention")
    else:   # fp32 arithmetic, the output rounded to bf16 once
        assert_close(got, want_o, atol=1e-6, rtol=2.0 ** -8 + 1e-5, what="gqa attention")
    check_lse(host(lse).numpy().reshape(want_l.shape), want_l, "gqa")
