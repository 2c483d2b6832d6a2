"""Parity of the named workloads at their full sizes, in the launch
configuration the benchmark times.

Two modes (the oracle is the plain CPU implementation; nothing of it comes
from the GPU except where a stage-wise gate says so):

* stage-wise -- the gates.  Each GPU stage is compared with the oracle stage
  fed the identical input bytes, including the GPU's own outputs of the stage
  before: the oracle scores and selects on the GPU's compressed (and, for FP4,
  quantised) indexer keys, and attends over the GPU's compressed K_c / V_c with
  the GPU's own selection.  Top-k sets must be identical except at near-ties
  (|s - s_k| <= 1e-3 |s_k|, counted), with no other exception; attention is
  held to the per-element bound of the arithmetic and the normalised error
  max|d| / max|ref| <= 1e-2.
* end to end -- reported, and gated only where the spec's tolerances apply
  unchanged: the oracle runs from the raw inputs (its own compression,
  quantisation, scores, selection, attention).  Compressed K / V must agree to
  within one bf16 rounding; top-k overlap is reported as recall; attention on
  rows whose sets agree must meet max-abs 2e-2 (BF16 indexer) or 6e-2
  (FP8 / FP4 indexer)."""
import math

import numpy as np
import pytest
import torch

import oracle
from long_context_compressed_18_b300 import configs, inputs, pipeline
from helpers import (DEV, assert_close, check_attn_stagewise, check_e2m1_keys, check_lse, host, sync_status,
                     topk_near_tie_check)

pytestmark = pytest.mark.gpu

# csa_index_topk scores the queries in chunks whose fp32 score buffer stays
# within 256 MB: chunk rows = 2^28 / (4 * B * N_c), a multiple of 4.
def _index_chunk_rows(s):
    return max(4, ((1 << 28) // (4 * s.B * max(s.N_c, 1))) & ~3)


def _np(t):
    return host(t).float().numpy()


def _take(t, rows, *shape, dtype=None):
    """Rows of t viewed as [-1, *shape], gathered where t lives, then copied
    to the host (floats widened to fp32), so that a few sampled rows of a
    multi-GB tensor are all that crosses to the host."""
    r = t.reshape(-1, *shape)[torch.as_tensor(np.asarray(rows), device=t.device)]
    r = r.cpu()
    return r.numpy() if not r.is_floating_point() else r.float().numpy()


def _sample_rows(n_q, count, seed, chunk=None, per_chunk=0):
    """Sorted flat rows: the first, middle and last row, `count` random rows,
    and with `chunk` given, `per_chunk` random rows inside every query chunk
    of that size plus the rows on both sides of each chunk boundary."""
    rng = np.random.default_rng(seed)
    picks = {0, n_q - 1, n_q // 2}
    picks.update(rng.choice(n_q, size=min(n_q, count), replace=False).tolist())
    if chunk:
        for c0 in range(0, n_q, chunk):
            c1 = min(n_q, c0 + chunk)
            picks.update(rng.integers(c0, c1, size=per_chunk).tolist())
            picks.update({c0, c1 - 1})
    return np.array(sorted(picks), np.int64)


def _rnd(dtype):
    if dtype == "f32":
        return lambda a: np.asarray(a, np.float64).astype(np.float32)
    return lambda a: torch.from_numpy(np.asarray(a, np.float64).astype(np.float32)).to(torch.bfloat16).float().numpy()


def _stagewise_csa(s, xc, g, rows):
    """Stage-wise gates of one CSA layer on the sampled rows.  Returns
    (near-tie rows, normalised attention error)."""
    lens = oracle.visible(s.q_pos0 + rows % s.n_q, s.m, s.N_c)
    # indexer + top-k on the GPU's compressed (quantised) indexer keys
    s64, _, sel = oracle.csa_index_topk(xc["idx_q"], xc["idx_q_scale"], s.idx_q_dtype, host(g["idx_k_c"]),
                                        host(g["idx_k_c_scale"]), s.idx_k_dtype, s.q_pos0, s.m, s.k, rows=rows)
    gsel = _take(g["topk"], rows, s.k)
    ties = topk_near_tie_check(gsel, sel, s64, lens, s.k)
    # attention over the GPU's K_c / V_c with the GPU's own selection
    q_rows = _take(xc["q"], rows, s.H, s.d)[None]
    kc, vc = host(g["k_c"]), host(g["v_c"])
    tau = 1.0 / math.sqrt(s.d)
    want_o, want_l = oracle.attention(q_rows, kc, vc, tau, oracle.SPARSE, idx=gsel[None])
    mag, _ = oracle.attention(q_rows, kc, np.abs(_np(vc)), tau, oracle.SPARSE, idx=gsel[None])
    got_o = _take(g["out"], rows, s.H, s.d)
    got_l = _take(g["lse"], rows, s.H)
    if s.dtype == "f32":
        assert_close(got_o, want_o, atol=2e-5, rtol=2e-5, what="csa attention (fp32)")
        check_lse(got_l, want_l, what="csa (fp32)")
        norm = 0.0
    else:
        norm = check_attn_stagewise(got_o, got_l, want_o, want_l, mag, what="csa attention")
    return ties, norm


def _end_to_end_csa(s, xc, g, rows, atol):
    """The oracle from raw inputs on the sampled rows: gates compressed K / V
    (one bf16 rounding), reports top-k recall, gates attention with the
    spec's max-abs tolerance on rows whose sets agree.  Returns recall."""
    kc = oracle.compress(xc["logits"], xc["k"], s.m)
    vc = oracle.compress(xc["logits"], xc["v"], s.m)
    ic = oracle.compress(xc["logits"], xc["idx_k"], s.m)
    tol = dict(atol=1e-5, rtol=1e-5) if s.dtype == "f32" else dict(atol=1e-6, rtol=2.0 ** -8 + 1e-5)
    assert_close(_np(g["k_c"]), kc, what="K_c", **tol)
    assert_close(_np(g["v_c"]), vc, what="V_c", **tol)
    ic32 = ic.astype(np.float32)
    if s.idx_k_dtype == "e2m1":
        check_e2m1_keys(host(g["idx_k_c"]).numpy().reshape(-1, s.d_I // 2),
                        host(g["idx_k_c_scale"]).numpy().reshape(-1, s.d_I // 32), ic.reshape(-1, s.d_I))
        ik, iks = oracle.quant_e2m1_blocks(ic32)
    elif s.idx_k_dtype == "e4m3":
        ik, iks = oracle.quant_e4m3_rows(ic32)
    else:
        assert_close(_np(g["idx_k_c"]), ic, what="indexer K_c", **tol)
        ik, iks = _rnd(s.idx_k_dtype)(ic), None
    _, _, sel = oracle.csa_index_topk(xc["idx_q"], xc["idx_q_scale"], s.idx_q_dtype, ik, iks, s.idx_k_dtype,
                                      s.q_pos0, s.m, s.k, rows=rows)
    gsel = _take(g["topk"], rows, s.k)
    lens = oracle.visible(s.q_pos0 + rows % s.n_q, s.m, s.N_c)
    hit = sum(len(set(gsel[r][gsel[r] >= 0].tolist()) & set(sel[r][sel[r] >= 0].tolist())) for r in range(len(rows)))
    recall = hit / max(1, int(np.minimum(lens, s.k).sum()))
    same = np.array([np.array_equal(gsel[r], sel[r]) for r in range(len(rows))])
    if same.any():
        rnd = _rnd(s.dtype)
        q_rows = _take(xc["q"], rows[same], s.H, s.d)[None]
        out, _ = oracle.attention(q_rows, rnd(kc), rnd(vc), 1.0 / math.sqrt(s.d), oracle.SPARSE,
                                  idx=sel[same][None])
        assert_close(_take(g["out"], rows[same], s.H, s.d), out, atol=atol, what="csa attention (e2e)")
    return recall


def _run_csa_layer(s, rows_count, seed, per_chunk=0):
    x = inputs.make_inputs(s, device=DEV)
    g = pipeline.csa_layer(x, s, pipeline.Workspace())
    sync_status()
    xc = {k: (None if v is None else v.cpu()) for k, v in x.items()}
    chunk = _index_chunk_rows(s) if per_chunk else None
    rows = _sample_rows(s.B * s.n_q, rows_count, seed, chunk=chunk, per_chunk=per_chunk)
    ties, norm = _stagewise_csa(s, xc, g, rows)
    atol = 6e-2 if s.idx_k_dtype in ("e4m3", "e2m1") else 2e-2
    recall = _end_to_end_csa(s, xc, g, rows, atol)
    print(f"{s.name}: {len(rows)} rows, near-tie rows {ties}, attention normalised error {norm:.2e}, "
          f"end-to-end top-k recall {recall:.4f}")
    return ties, recall


def test_tiny_csa_f32_full():
    s = configs.TINY_CSA_F32
    x = inputs.make_inputs(s)
    g = pipeline.csa_layer({k: (None if v is None else v.to(DEV)) for k, v in x.items()}, s, pipeline.Workspace())
    sync_status()
    rows = np.arange(s.n_q)
    ties, _ = _stagewise_csa(s, x, g, rows)          # every row
    recall = _end_to_end_csa(s, x, g, rows, atol=2e-2)
    assert recall >= 0.99, recall


def test_csa_prefill_bf16_full_size():
    s = configs.CSA_PREFILL_BF16
    _, recall = _run_csa_layer(s, 48, seed=2, per_chunk=4)
    assert recall >= 0.95, recall


@pytest.mark.parametrize("layer", [2, 4])
def test_hybrid_stack_csa_layer_stagewise(layer):
    """A CSA layer of the hybrid stack at n = 131,072 (FP4 indexer keys from
    the compression epilogue, widened to E4M3 for the tcgen05 indexer): the
    oracle widens and scores the GPU's own E2M1 keys and block scales; sampled
    rows cover every csa_index_topk query chunk and both sides of its
    boundaries."""
    s = configs.STACK_LAYERS[layer]
    assert s.kind == "csa" and s.idx_k_dtype == "e2m1"
    _, recall = _run_csa_layer(s, 16, seed=10 + layer, per_chunk=1)
    assert recall >= 0.9, recall


def test_csa_decode_1m_full_size():
    """Every one of the 32 sequences: top-k against the oracle's selection on
    the same E4M3 cache (near-ties only), attention and lse against the oracle
    on the GPU's own selection."""
    s = configs.CSA_DECODE_1M
    x = inputs.make_inputs(s, device=DEV)
    g = pipeline.csa_decode(x, s, pipeline.Workspace())
    sync_status()
    gsel_all = host(g["topk"]).numpy().reshape(s.B, s.k)
    tau = 1.0 / math.sqrt(s.d)
    ties = 0
    for b in range(s.B):
        iq, iqs = x["idx_q"][b:b + 1].cpu(), x["idx_q_scale"][b:b + 1].cpu()
        ik, iks = x["idx_k_c"][b:b + 1].cpu(), x["idx_k_c_scale"][b:b + 1].cpu()
        s64, _, sel = oracle.csa_index_topk(iq, iqs, "e4m3", ik, iks, "e4m3", s.q_pos0, s.m, s.k)
        gsel = gsel_all[b:b + 1]
        ties += topk_near_tie_check(gsel, sel, s64, [s.N_c], s.k)
        q, kc, vc = x["q"][b:b + 1].cpu(), x["k_c"][b:b + 1].cpu(), x["v_c"][b:b + 1].cpu()
        want_o, want_l = oracle.attention(q, kc, vc, tau, oracle.SPARSE, idx=gsel[None])
        mag, _ = oracle.attention(q, kc, vc.float().abs(), tau, oracle.SPARSE, idx=gsel[None])
        check_attn_stagewise(_np(g["out"][b]).reshape(1, s.H, s.d), host(g["lse"][b]).numpy().reshape(1, s.H),
                             want_o, want_l, mag, what=f"decode b={b}")
    print(f"decode: 32 sequences, near-tie rows {ties}")


def test_hca_prefill_1m_full_size():
    s = configs.HCA_PREFILL_1M
    x = inputs.make_inputs(s, device=DEV)
    g = pipeline.hca_layer(x, s)
    sync_status()
    xc = {k: (None if v is None else v.cpu()) for k, v in x.items()}
    kc = oracle.compress(xc["logits"], xc["k"], s.m)
    vc = oracle.compress(xc["logits"], xc["v"], s.m)
    assert_close(_np(g["k_c"]), kc, atol=1e-6, rtol=2.0 ** -8 + 1e-5, what="K_c")
    assert_close(_np(g["v_c"]), vc, atol=1e-6, rtol=2.0 ** -8 + 1e-5, what="V_c")
    rows = _sample_rows(s.n_q, 12, seed=4)
    # stage-wise: attention over the GPU's own K_c / V_c
    q_rows = _take(xc["q"], rows, s.H, s.d)
    gk, gv = host(g["k_c"]), host(g["v_c"])
    tau = 1.0 / math.sqrt(s.d)
    want, wl, mag = [], [], []
    for i, r in enumerate(rows):
        o, l_ = oracle.attention(q_rows[i:i + 1][None], gk, gv, tau, oracle.CLOSED_BLOCKS, q_pos0=s.q_pos0 + int(r), m=s.m)
        mg, _ = oracle.attention(q_rows[i:i + 1][None], gk, np.abs(_np(gv)), tau, oracle.CLOSED_BLOCKS,
                                 q_pos0=s.q_pos0 + int(r), m=s.m)
        want.append(o), wl.append(l_), mag.append(mg)
    check_attn_stagewise(_take(g["out"], rows, s.H, s.d), _take(g["lse"], rows, s.H),
                         np.concatenate(want), np.concatenate(wl), np.concatenate(mag), what="hca attention")


def test_hybrid_stack_full_size():
    """All six layers of the stack end to end at n = 131,072 on sampled rows:
    SWA and HCA stage-wise (HCA over the GPU's own compressed K / V); the CSA
    layers' stage-wise gates are in test_hybrid_stack_csa_layer_stagewise."""
    ws = pipeline.Workspace()
    for li, s in enumerate(configs.STACK_LAYERS):
        if s.kind == "csa":
            continue
        x = inputs.make_inputs(s, device=DEV)
        g = pipeline.run_layer(x, s, ws)
        sync_status()
        rows = _sample_rows(s.n_q, 6, seed=10 + li)
        xc = {k: (None if v is None else v.cpu()) for k, v in x.items()}
        q_rows = _take(xc["q"], rows, s.H, s.d)
        tau = 1.0 / math.sqrt(s.d)
        if s.kind == "hca":
            kc = oracle.compress(xc["logits"], xc["k"], s.m)
            assert_close(_np(g["k_c"]), kc, atol=1e-6, rtol=2.0 ** -8 + 1e-5, what=f"layer {li} K_c")
            K, V = host(g["k_c"]), host(g["v_c"])
            kw = lambda r: dict(mode=oracle.CLOSED_BLOCKS, q_pos0=int(r), m=s.m)
        else:
            K, V = xc["k"], xc["v"]
            kw = lambda r: dict(mode=oracle.WINDOW, q_pos0=int(r), window=s.window)
        res = [oracle.attention(q_rows[i:i + 1][None], K, V, tau, **kw(r)) for i, r in enumerate(rows)]
        mag = [oracle.attention(q_rows[i:i + 1][None], K, np.abs(_np(V)), tau, **kw(r))[0] for i, r in enumerate(rows)]
        check_attn_stagewise(_take(g["out"], rows, s.H, s.d), _take(g["lse"], rows, s.H),
                             np.concatenate([o for o, _ in res]), np.concatenate([l_ for _, l_ in res]),
                             np.concatenate(mag), what=f"layer {li} {s.kind}")
        del x, g, xc
        torch.cuda.empty_cache()


def test_decode_batch_invariance_and_determinism():
    """A sequence's decode output is bitwise identical alone or at any batch
    position, and across repeated runs ("DeepSeek V4 技术解读" §6.2)."""
    s = configs.shape(name="inv", kind="csa_decode", B=4, n=4 * 20000, m=4, n_q=1, q_pos0=4 * 20000 - 1,
                      H=64, d=128, H_I=64, d_I=128, k=1024, idx_q_dtype="e4m3", idx_k_dtype="e4m3")
    x = inputs.make_inputs(s, device=DEV)
    ws = pipeline.Workspace()
    g1 = pipeline.csa_decode(x, s, ws)
    g2 = pipeline.csa_decode(x, s, ws)
    s1 = configs.shape(**{**s.__dict__, "B": 1})
    x1 = inputs.make_inputs(s1, device=DEV, batches=[2])
    ga = pipeline.csa_decode(x1, s1, ws)
    sync_status()
    assert torch.equal(g1["topk"], g2["topk"]) and torch.equal(g1["out"], g2["out"])
    assert torch.equal(ga["topk"][0], g1["topk"][2])
    assert torch.equal(ga["out"][0], g1["out"][2]) and torch.equal(ga["lse"][0], g1["lse"][2])
