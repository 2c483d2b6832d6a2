"""Pins for the oracle's path steps: compression, indexer scores, top-k and
attention.  Each check is a closed form, an invariant, brute force on a tiny
input, or a special case that reduces to a library routine (numpy dot,
torch's scaled_dot_product_attention)."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from long_context_compressed_18_b300 import configs

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ---- compression ------------------------------------------------------------

def test_compress_equal_logits_is_block_mean():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((2, 40, 6)).astype(np.float32)
    lg = np.full((2, 40), 0.37, np.float32)
    out = oracle.compress(lg, x, 4)
    assert out.shape == (2, 10, 6)
    want = x.astype(np.float64).reshape(2, 10, 4, 6).mean(2)
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-14)


def test_compress_dominant_logit_selects_token():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((1, 32, 5)).astype(np.float32)
    lg = np.zeros((1, 32), np.float32)
    pick = [2, 4, 11, 13, 17, 22, 24, 31]          # one per block of 4
    lg[0, pick] = 1e4
    out = oracle.compress(lg, x, 4)
    np.testing.assert_array_equal(out[0], x[0, pick].astype(np.float64))
    # a very negative logit drops its token from the block
    lg2 = np.zeros((1, 8), np.float32)
    lg2[0, 0] = -1e4
    out2 = oracle.compress(lg2, x[:, :8], 4)
    np.testing.assert_allclose(out2[0, 0], x[0, 1:4].astype(np.float64).mean(0), atol=1e-14)


def test_compress_m1_identity_and_closed_blocks_only():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((1, 9, 3)).astype(np.float32)
    lg = rng.standard_normal((1, 9)).astype(np.float32)
    np.testing.assert_array_equal(oracle.compress(lg, x, 1), x.astype(np.float64))
    out = oracle.compress(lg, x, 4)                # trailing partial block dropped
    assert out.shape == (1, 2, 3)


def test_compress_two_token_closed_form():
    # m = 2: w0 = 1 / (1 + e^(l1 - l0)) -- the logistic function
    x = np.array([[[1.0, 0.0], [0.0, 1.0]]], np.float32)
    lg = np.array([[0.5, -1.25]], np.float32)
    out = oracle.compress(lg, x, 2)
    w0 = 1.0 / (1.0 + math.exp(-1.25 - 0.5))
    np.testing.assert_allclose(out[0, 0], [w0, 1 - w0], rtol=1e-15)


# ---- indexer scores ---------------------------------------------------------

def test_index_score_single_head_is_dot_product():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 5, 1, 16)).astype(np.float32)
    k = rng.standard_normal((1, 7, 16)).astype(np.float32)
    s64, _ = oracle.index_scores(q, None, k, None, q_pos0=100, m=1)
    want = np.einsum("td,jd->tj", q[0, :, 0].astype(np.float64), k[0].astype(np.float64))
    np.testing.assert_allclose(s64, want, rtol=1e-13, atol=1e-13)


def test_index_score_sums_scaled_heads():
    rng = np.random.default_rng(4)
    B, nq, H, d, N = 2, 3, 5, 8, 6
    q = rng.standard_normal((B, nq, H, d)).astype(np.float32)
    k = rng.standard_normal((B, N, d)).astype(np.float32)
    qs = rng.uniform(0.5, 2, (B, nq, H)).astype(np.float32)
    ks = rng.uniform(0.5, 2, (B, N)).astype(np.float32)
    s64, s32 = oracle.index_scores(q, qs, k, ks, q_pos0=1000, m=4)
    qsum = (q.astype(np.float64) * qs[..., None]).sum(2)          # [B, nq, d]
    want = np.einsum("bqd,bjd->bqj", qsum, k.astype(np.float64)) * ks[:, None, :]
    np.testing.assert_allclose(s64.reshape(B, nq, N), want, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(s32, s64.astype(np.float32))


def test_index_visibility_closed_blocks():
    q = np.ones((1, 12, 1, 2), np.float32)
    k = np.ones((1, 3, 2), np.float32)
    s64, _ = oracle.index_scores(q, None, k, None, q_pos0=0, m=4)
    for t in range(12):
        nv = (t + 1) // 4
        assert np.all(np.isfinite(s64[t, :nv])) and np.all(np.isnan(s64[t, nv:])), t
    # entry j first becomes visible at t = 4j + 3
    assert np.isnan(s64[2, 0]) and np.isfinite(s64[3, 0])


# ---- top-k ------------------------------------------------------------------

def _brute_topk(s, k):
    L = len(s)
    key = lambda j: (-(0.0 if s[j] == 0 else s[j]), j)
    c = min(k, L)
    found = []
    for sub in itertools.combinations(range(L), c):
        inside = set(sub)
        if all(key(a) < key(b) for a in inside for b in range(L) if b not in inside):
            found.append(sub)
    assert len(found) == 1
    return list(found[0]) + [-1] * (k - c)


def test_topk_brute_force_tiny():
    rng = np.random.default_rng(5)
    for trial in range(200):
        L = int(rng.integers(0, 9))
        k = int(rng.integers(1, 6))
        vals = rng.integers(-3, 4, L).astype(np.float32) * 0.5   # many ties
        if L > 2 and trial % 3 == 0:
            vals[1] = -0.0
            vals[2] = 0.0
        s = np.zeros((1, 10), np.float32)
        s[0, :L] = vals
        got = oracle.topk(s, [L], k)[0].tolist()
        assert got == _brute_topk(vals.tolist(), k), (vals, k, got)


def test_topk_short_rows_take_everything():
    s = np.random.default_rng(6).standard_normal((3, 50)).astype(np.float32)
    got = oracle.topk(s, [0, 7, 50], 16)
    assert got[0].tolist() == [-1] * 16
    assert got[1].tolist() == list(range(7)) + [-1] * 9
    assert len(set(got[2].tolist())) == 16 and sorted(got[2].tolist()) == got[2].tolist()


# ---- attention --------------------------------------------------------------

def _sdpa_causal(q, K, V, tau, window=None):
    """torch SDPA in fp64 with one KV head broadcast to all heads."""
    B, n, H, d = q.shape
    qt = torch.from_numpy(q.astype(np.float64)).permute(0, 2, 1, 3)
    Kt = torch.from_numpy(K.astype(np.float64))[:, None].expand(B, H, n, d)
    Vt = torch.from_numpy(V.astype(np.float64))[:, None].expand(B, H, n, d)
    i = torch.arange(n)[:, None]
    j = torch.arange(n)[None, :]
    mask = j <= i
    if window is not None:
        mask &= j > i - window
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, attn_mask=mask, scale=tau)
    return o.permute(0, 2, 1, 3).numpy()


def _qkv(B=2, n=24, H=3, d=8, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, n, H, d)).astype(np.float32)
    K = rng.standard_normal((B, n, d)).astype(np.float32)
    V = rng.standard_normal((B, n, d)).astype(np.float32)
    return q, K, V


def test_closed_block_attention_m1_is_causal_sdpa():
    q, K, V = _qkv()
    tau = 1 / math.sqrt(8)
    out, lse = oracle.attention(q, K, V, tau, oracle.CLOSED_BLOCKS, q_pos0=0, m=1)
    want = _sdpa_causal(q, K, V, tau)
    np.testing.assert_allclose(out.reshape(want.shape), want, rtol=1e-12, atol=1e-12)


def test_sparse_attention_full_selection_is_causal_sdpa():
    q, K, V = _qkv(seed=1)
    B, n = q.shape[:2]
    idx = np.full((B, n, n), -1, np.int32)
    for t in range(n):
        idx[:, t, :t + 1] = np.arange(t + 1)
    tau = 0.3
    out, _ = oracle.attention(q, K, V, tau, oracle.SPARSE, idx=idx)
    want = _sdpa_causal(q, K, V, tau)
    np.testing.assert_allclose(out.reshape(want.shape), want, rtol=1e-12, atol=1e-12)


def test_window_attention_matches_masked_sdpa():
    q, K, V = _qkv(seed=2)
    tau = 0.35
    for W in (1, 5, 24, 100):
        out, _ = oracle.attention(q, K, V, tau, oracle.WINDOW, q_pos0=0, window=W)
        want = _sdpa_causal(q, K, V, tau, window=W)
        np.testing.assert_allclose(out.reshape(want.shape), want, rtol=1e-12, atol=1e-12)
    out1, lse1 = oracle.attention(q, K, V, tau, oracle.WINDOW, q_pos0=0, window=1)
    np.testing.assert_array_equal(out1.reshape(q.shape), np.broadcast_to(V[:, :, None, :], q.shape))


def test_lse_and_empty_set():
    q, K, V = _qkv(B=1, n=8, H=2, d=4, seed=3)
    idx = np.full((1, 8, 2), -1, np.int32)
    idx[0, :, 0] = 5
    out, lse = oracle.attention(q, K, V, 0.5, oracle.SPARSE, idx=idx)
    np.testing.assert_array_equal(out.reshape(1, 8, 2, 4), np.broadcast_to(V[0, 5], (1, 8, 2, 4)))
    want = 0.5 * np.einsum("thd,d->th", q[0].astype(np.float64), K[0, 5].astype(np.float64))
    np.testing.assert_allclose(lse, want.reshape(8, 2), rtol=1e-14)
    out0, lse0 = oracle.attention(q, K, V, 0.5, oracle.CLOSED_BLOCKS, q_pos0=0, m=4)
    assert np.all(out0[:3] == 0) and np.all(np.isneginf(lse0[:3]))   # t < m-1: nothing visible


def test_full_topk_csa_equals_dense_closed_block_attention():
    """k >= N_c: CSA selects every visible entry, so it equals HCA-style dense
    attention over the same compressed entries."""
    rng = np.random.default_rng(9)
    B, n, m, H, d, HI, dI = 1, 64, 4, 2, 8, 2, 4
    Nc = n // m
    lg = rng.standard_normal((B, n)).astype(np.float32)
    K = rng.standard_normal((B, n, d)).astype(np.float32)
    V = rng.standard_normal((B, n, d)).astype(np.float32)
    iK = rng.standard_normal((B, n, dI)).astype(np.float32)
    q = rng.standard_normal((B, n, H, d)).astype(np.float32)
    iq = rng.standard_normal((B, n, HI, dI)).astype(np.float32)
    Kc = oracle.compress(lg, K, m).astype(np.float32)
    Vc = oracle.compress(lg, V, m).astype(np.float32)
    iKc = oracle.compress(lg, iK, m).astype(np.float32)
    _, _, sel = oracle.csa_index_topk(iq, None, "f32", iKc, None, "f32", 0, m, k=Nc)
    sparse, lse_s = oracle.attention(q, Kc, Vc, 0.3, oracle.SPARSE, idx=sel.reshape(B, n, Nc))
    dense, lse_d = oracle.attention(q, Kc, Vc, 0.3, oracle.CLOSED_BLOCKS, q_pos0=0, m=m)
    np.testing.assert_allclose(sparse, dense, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse_s[np.isfinite(lse_s)], lse_d[np.isfinite(lse_d)], rtol=1e-12)


def test_csa_m1_full_k_is_causal_attention():
    rng = np.random.default_rng(10)
    B, n, H, d = 1, 20, 2, 8
    lg = rng.standard_normal((B, n)).astype(np.float32)
    K = rng.standard_normal((B, n, d)).astype(np.float32)
    V = rng.standard_normal((B, n, d)).astype(np.float32)
    iK = rng.standard_normal((B, n, 4)).astype(np.float32)
    q = rng.standard_normal((B, n, H, d)).astype(np.float32)
    iq = rng.standard_normal((B, n, 2, 4)).astype(np.float32)
    Kc = oracle.compress(lg, K, 1).astype(np.float32)
    Vc = oracle.compress(lg, V, 1).astype(np.float32)
    _, _, sel = oracle.csa_index_topk(iq, None, "f32", oracle.compress(lg, iK, 1).astype(np.float32),
                                      None, "f32", 0, 1, k=n)
    out, _ = oracle.attention(q, Kc, Vc, 0.25, oracle.SPARSE, idx=sel.reshape(B, n, n))
    np.testing.assert_allclose(out.reshape(q.shape), _sdpa_causal(q, K, V, 0.25), rtol=1e-12, atol=1e-12)


def test_topk_selects_entries_with_largest_attention_when_indexer_is_attention():
    """With indexer Q/K equal to attention Q/K (one head), the selected set is
    the top-k by attention logit, so its softmax mass is the largest of any
    k-subset (checked against random subsets)."""
    rng = np.random.default_rng(12)
    n, d, k = 40, 6, 5
    q = rng.standard_normal((1, 1, 1, d)).astype(np.float32)
    K = rng.standard_normal((1, n, d)).astype(np.float32)
    _, s32, sel = oracle.csa_index_topk(q, None, "f32", K, None, "f32", n - 1, 1, k)
    logit = K[0].astype(np.float64) @ q[0, 0, 0].astype(np.float64)
    mass = np.exp(logit[sel[0]]).sum()
    for _ in range(200):
        sub = rng.choice(n, k, replace=False)
        assert np.exp(logit[sub]).sum() <= mass + 1e-12


def test_named_shapes_follow_page_parameters():
    with open(os.path.join(GOLD, "pages_parameters.json")) as f:
        g = json.load(f)
    for s in (configs.CSA_PREFILL_BF16, configs.CSA_DECODE_1M):
        assert s.m == g["csa"]["compression_ratio_m"]
        assert (s.H_I, s.d_I, s.k) == (g["csa"]["indexer_heads"], g["csa"]["indexer_head_dim"], g["csa"]["top_k"])
    assert configs.HCA_PREFILL_1M.m == g["hca"]["compression_ratio_m"]
    kinds = [s.kind for s in configs.STACK_LAYERS]
    assert kinds[:g["hybrid"]["swa_layers"]] == ["swa", "swa"]
    assert kinds[2:] == ["csa", "hca", "csa", "hca"]
