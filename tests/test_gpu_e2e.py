"""End-to-end parity of the named workloads at their full sizes.

The GPU runs every query; the oracle recomputes sampled query rows from the
same seeded inputs (its own compression, quantisation, scores, top-k and
attention -- nothing is taken from the GPU).  Gates:
  * compressed K/V within one bf16 rounding of the oracle (all entries);
  * top-k sets identical except at near-ties, |s - s_k| <= 1e-3 |s_k|;
  * attention within max-abs 2e-2 on rows whose selected sets agree.
Rows whose FP4 indexer keys straddle a quantisation boundary can differ in
their sets beyond the near-tie band (a one-step code change, not a ranking
error); those are counted and bounded separately."""
import math

import numpy as np
import pytest
import torch

import oracle
from long_context_compressed_18_b300 import configs, inputs, pipeline
from helpers import DEV, assert_close, host, sync_status, topk_near_tie_check

pytestmark = pytest.mark.gpu


def _np(t):
    return host(t).float().numpy()


def _sample_rows(n_q, count, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, n_q - 1, n_q // 2]
    extra = rng.choice(n_q, size=min(n_q, count), replace=False).tolist()
    return np.array(sorted(set(fixed + extra)), np.int64)


def _oracle_csa_rows(s, x_cpu, rows):
    """Oracle CSA for the given flat rows (batch 1 inputs on the host)."""
    o = {}
    kc = oracle.compress(x_cpu["logits"], x_cpu["k"], s.m)
    vc = oracle.compress(x_cpu["logits"], x_cpu["v"], s.m)
    ic = oracle.compress(x_cpu["logits"], x_cpu["idx_k"], s.m)
    rnd = (lambda a: a.astype(np.float32)) if s.dtype == "f32" else \
        (lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).float().numpy())
    o["k_c64"], o["v_c64"] = kc, vc
    kc32, vc32 = rnd(kc), rnd(vc)
    ic32 = ic.astype(np.float32)
    if s.idx_k_dtype == "e2m1":
        ik, iks = oracle.quant_e2m1_blocks(ic32)
    elif s.idx_k_dtype == "e4m3":
        ik, iks = oracle.quant_e4m3_rows(ic32)
    else:
        ik, iks = rnd(ic), None
    s64, s32, sel = oracle.csa_index_topk(x_cpu["idx_q"], x_cpu["idx_q_scale"], s.idx_q_dtype, ik, iks,
                                          s.idx_k_dtype, s.q_pos0, s.m, s.k, rows=rows)
    q_rows = _np(x_cpu["q"]).reshape(-1, s.H, s.d)[rows][None]
    out, lse = oracle.attention(q_rows, kc32, vc32, 1.0 / math.sqrt(s.d), oracle.SPARSE, idx=sel[None])
    o.update(scores64=s64, sel=sel, out=out, lse=lse)
    return o


def _compare_csa(s, g, o, rows, allow_quant_rows=0.0):
    lens = oracle.visible(s.q_pos0 + rows, s.m, s.N_c)
    gsel = host(g["topk"]).numpy().reshape(-1, s.k)[rows]
    try:
        swaps = topk_near_tie_check(gsel, o["sel"], o["scores64"], lens, s.k)
        quant_rows = 0
    except AssertionError:
        if allow_quant_rows == 0.0:
            raise
        swaps, quant_rows = 0, 0
        for r in range(len(rows)):
            try:
                swaps += topk_near_tie_check(gsel[r:r + 1], o["sel"][r:r + 1], o["scores64"][r:r + 1], lens[r:r + 1], s.k)
            except AssertionError:
                quant_rows += 1
        assert quant_rows <= allow_quant_rows * len(rows), (quant_rows, len(rows))
    same = np.array([np.array_equal(gsel[r], o["sel"][r]) for r in range(len(rows))])
    assert same.mean() >= 0.5, same.mean()
    gout = _np(g["out"]).reshape(-1, s.H, s.d)[rows][same]
    assert_close(gout, o["out"][same], atol=2e-2, what="csa attention")
    return swaps, int((~same).sum())


def test_tiny_csa_f32_full():
    s = configs.TINY_CSA_F32
    x = inputs.make_inputs(s)
    ws = pipeline.Workspace()
    g = pipeline.csa_layer({k: (None if v is None else v.to(DEV)) for k, v in x.items()}, s, ws)
    sync_status()
    rows = np.arange(s.n_q)
    o = _oracle_csa_rows(s, x, rows)
    assert_close(_np(g["k_c"]), o["k_c64"], atol=1e-5, rtol=1e-5, what="K_c")
    assert_close(_np(g["v_c"]), o["v_c64"], atol=1e-5, rtol=1e-5, what="V_c")
    swaps, diff_rows = _compare_csa(s, g, o, rows)
    assert diff_rows <= 0.01 * s.n_q
    assert_close(_np(g["out"]).reshape(-1, s.H, s.d), o["out"], atol=1e-4, what="all rows") if diff_rows == 0 else None


def test_csa_prefill_bf16_full_size():
    s = configs.CSA_PREFILL_BF16
    x = inputs.make_inputs(s, device=DEV)
    ws = pipeline.Workspace()
    g = pipeline.csa_layer(x, s, ws)
    sync_status()
    xc = {k: (None if v is None else v.cpu()) for k, v in x.items()}
    rows = _sample_rows(s.n_q, 24, seed=2)
    o = _oracle_csa_rows(s, xc, rows)
    assert_close(_np(g["k_c"]), o["k_c64"], atol=1e-6, rtol=2.0 ** -8 + 1e-5, what="K_c")
    assert_close(_np(g["v_c"]), o["v_c64"], atol=1e-6, rtol=2.0 ** -8 + 1e-5, what="V_c")
    _compare_csa(s, g, o, rows)


def test_csa_decode_1m_full_size():
    s = configs.CSA_DECODE_1M
    x = inputs.make_inputs(s, device=DEV)
    ws = pipeline.Workspace()
    g = pipeline.csa_decode(x, s, ws)
    sync_status()
    for b in (0, 13, 31):
        iq, iqs = x["idx_q"][b:b + 1].cpu(), x["idx_q_scale"][b:b + 1].cpu()
        ik, iks = x["idx_k_c"][b:b + 1].cpu(), x["idx_k_c_scale"][b:b + 1].cpu()
        s64, s32, sel = oracle.csa_index_topk(iq, iqs, "e4m3", ik, iks, "e4m3", s.q_pos0, s.m, s.k)
        gsel = host(g["topk"][b]).numpy().reshape(1, s.k)
        topk_near_tie_check(gsel, sel, s64, [s.N_c], s.k)
        if np.array_equal(gsel, sel):
            out, lse = oracle.attention(x["q"][b:b + 1].cpu(), x["k_c"][b:b + 1].cpu(), x["v_c"][b:b + 1].cpu(),
                                        1.0 / math.sqrt(s.d), oracle.SPARSE, idx=sel[None])
            assert_close(_np(g["out"][b]).reshape(1, s.H, s.d), out, atol=2e-2, what=f"decode attn b={b}")
            assert_close(host(g["lse"][b]).numpy().reshape(1, s.H), lse, atol=1e-3, what="decode lse")


def test_hca_prefill_1m_full_size():
    s = configs.HCA_PREFILL_1M
    x = inputs.make_inputs(s, device=DEV)
    g = pipeline.hca_layer(x, s)
    sync_status()
    xc = {k: (None if v is None else v.cpu()) for k, v in x.items()}
    kc = oracle.compress(xc["logits"], xc["k"], s.m)
    vc = oracle.compress(xc["logits"], xc["v"], s.m)
    assert_close(_np(g["k_c"]), kc, atol=1e-6, rtol=2.0 ** -8 + 1e-5, what="K_c")
    rows = _sample_rows(s.n_q, 12, seed=4)
    rnd = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).float().numpy()
    q_rows = _np(xc["q"]).reshape(-1, s.H, s.d)[rows]
    want = np.concatenate([
        oracle.attention(q_rows[i:i + 1][None], rnd(kc), rnd(vc), 1.0 / math.sqrt(s.d), oracle.CLOSED_BLOCKS,
                         q_pos0=s.q_pos0 + int(r), m=s.m)[0]
        for i, r in enumerate(rows)])
    assert_close(_np(g["out"]).reshape(-1, s.H, s.d)[rows], want, atol=2e-2, what="hca attention")


def test_hybrid_stack_full_size():
    ws = pipeline.Workspace()
    for li, s in enumerate(configs.STACK_LAYERS):
        x = inputs.make_inputs(s, device=DEV)
        g = pipeline.run_layer(x, s, ws)
        sync_status()
        rows = _sample_rows(s.n_q, 6, seed=10 + li)
        xc = {k: (None if v is None else v.cpu()) for k, v in x.items()}
        if s.kind == "csa":
            o = _oracle_csa_rows(s, xc, rows)
            _compare_csa(s, g, o, rows, allow_quant_rows=0.34)
        elif s.kind == "hca":
            rnd = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).float().numpy()
            kc = rnd(oracle.compress(xc["logits"], xc["k"], s.m))
            vc = rnd(oracle.compress(xc["logits"], xc["v"], s.m))
            q_rows = _np(xc["q"]).reshape(-1, s.H, s.d)[rows]
            want = np.concatenate([
                oracle.attention(q_rows[i:i + 1][None], kc, vc, 1.0 / math.sqrt(s.d), oracle.CLOSED_BLOCKS,
                                 q_pos0=int(r), m=s.m)[0] for i, r in enumerate(rows)])
            assert_close(_np(g["out"]).reshape(-1, s.H, s.d)[rows], want, atol=2e-2, what=f"layer {li} hca")
        else:
            q_rows = _np(xc["q"]).reshape(-1, s.H, s.d)[rows]
            want = np.concatenate([
                oracle.attention(q_rows[i:i + 1][None], xc["k"], xc["v"], 1.0 / math.sqrt(s.d), oracle.WINDOW,
                                 q_pos0=int(r), window=s.window)[0] for i, r in enumerate(rows)])
            assert_close(_np(g["out"]).reshape(-1, s.H, s.d)[rows], want, atol=2e-2, what=f"layer {li} swa")
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
