"""Pins of the oracle's variant readings (per-channel compression weights, the
weighted / ReLU indexer, GQA / MHA KV heads) against closed forms and library
routines."""
import math

import numpy as np
import torch

import oracle

rng = np.random.default_rng(2026)


# ---- per-channel compression weights ---------------------------------------

def test_per_channel_equal_logits_give_block_mean():
    B, n, m, d = 2, 40, 4, 16
    x = rng.standard_normal((B, n, d)).astype(np.float32)
    got = oracle.compress_per_channel(np.zeros((B, n, d), np.float32), x, m)
    want = x.astype(np.float64).reshape(B, n // m, m, d).mean(2)
    assert np.max(np.abs(got - want)) < 1e-12


def test_per_channel_dominant_logit_selects_per_channel():
    B, n, m, d = 1, 32, 8, 24
    x = rng.standard_normal((B, n, d)).astype(np.float32)
    pick = rng.integers(0, m, size=(n // m, d))
    lg = np.zeros((B, n, d), np.float32)
    for j in range(n // m):
        lg[0, j * m + pick[j], np.arange(d)] = 1e4
    got = oracle.compress_per_channel(lg, x, m)
    want = np.stack([x[0, j * m + pick[j], np.arange(d)] for j in range(n // m)])[None]
    assert np.array_equal(got, want.astype(np.float64))


def test_per_channel_two_token_blocks_are_logistic():
    B, n, m, d = 2, 10, 2, 8
    x = rng.standard_normal((B, n, d)).astype(np.float32)
    lg = (3 * rng.standard_normal((B, n, d))).astype(np.float32)
    got = oracle.compress_per_channel(lg, x, m)
    l0, l1 = lg[:, 0::2].astype(np.float64), lg[:, 1::2].astype(np.float64)
    w0 = 1.0 / (1.0 + np.exp(l1 - l0))
    want = w0 * x[:, 0::2] + (1.0 - w0) * x[:, 1::2]
    assert np.max(np.abs(got - want)) < 1e-12


def test_per_channel_identity_and_scalar_special_case():
    B, n, d = 1, 12, 8
    x = rng.standard_normal((B, n, d)).astype(np.float32)
    lg = rng.standard_normal((B, n, d)).astype(np.float32)
    assert np.array_equal(oracle.compress_per_channel(lg, x, 1), x.astype(np.float64))
    # one logit per token, repeated on every channel: the scalar-weight reading
    ls = rng.standard_normal((B, n)).astype(np.float32)
    got = oracle.compress_per_channel(np.repeat(ls[..., None], d, -1), x, 4)
    want = oracle.compress(ls, x, 4)
    assert np.max(np.abs(got - want)) < 1e-12


# ---- weighted / ReLU indexer --------------------------------------------------

def _idx_inputs(H=4, dI=16, Nc=30, n_q=3):
    q = rng.standard_normal((1, n_q, H, dI)).astype(np.float32)
    k = rng.standard_normal((1, Nc, dI)).astype(np.float32)
    qs = rng.uniform(0.5, 2, (1, n_q, H)).astype(np.float32)
    ks = rng.uniform(0.5, 2, (1, Nc)).astype(np.float32)
    return q, qs, k, ks


def test_relu_single_head_is_clipped_dot_product():
    q, qs, k, ks = _idx_inputs(H=1)
    s64, _ = oracle.index_scores(q, qs, k, ks, 4 * 30 - 1, 4, relu=True)
    dots = np.einsum("d,jd->j", q[0, 1, 0].astype(np.float64), k[0].astype(np.float64))
    want = qs[0, 1, 0] * ks[0].astype(np.float64) * np.maximum(dots, 0.0)
    assert np.max(np.abs(s64[1] - want)) < 1e-9
    assert (dots < 0).any() and (s64[1][dots < 0] == 0).all()


def test_one_hot_head_weight_selects_that_head():
    q, qs, k, ks = _idx_inputs(H=4)
    w = np.zeros((1, 3, 4), np.float32)
    w[0, :, 2] = 1.0
    s64, _ = oracle.index_scores(q, qs, k, ks, 4 * 30 - 1, 4, head_w=w)
    dots = np.einsum("d,jd->j", q[0, 0, 2].astype(np.float64), k[0].astype(np.float64))
    assert np.max(np.abs(s64[0] - np.float64(qs[0, 0, 2]) * ks[0].astype(np.float64) * dots)) < 1e-9


def test_relu_comes_before_the_head_weight():
    """A negative weight on a head with a positive dot product flips its
    term's sign (ReLU of the dot product, then the weight), it does not clip
    it to zero."""
    q, qs, k, ks = _idx_inputs(H=2)
    q[0, :, 1] = q[0, :, 0]                      # both heads see the same dots
    w = np.array([[[1.0, -0.5]] * 3], np.float32)
    s64, _ = oracle.index_scores(q, None, k, None, 4 * 30 - 1, 4, head_w=w, relu=True)
    dots = np.einsum("d,jd->j", q[0, 0, 0].astype(np.float64), k[0].astype(np.float64))
    assert np.max(np.abs(s64[0] - 0.5 * np.maximum(dots, 0.0))) < 1e-9


def test_relu_inactive_on_positive_inputs_and_unit_weights_are_plain():
    q, qs, k, ks = _idx_inputs()
    q, k = np.abs(q), np.abs(k)
    plain, _ = oracle.index_scores(q, qs, k, ks, 4 * 30 - 1, 4)
    relu, _ = oracle.index_scores(q, qs, k, ks, 4 * 30 - 1, 4, relu=True,
                                  head_w=np.ones((1, 3, 4), np.float32))
    assert np.array_equal(np.nan_to_num(plain, nan=7.0), np.nan_to_num(relu, nan=7.0))


# ---- GQA / MHA KV heads ------------------------------------------------------

def _sdpa(q, K, V, tau):
    """fp64 SDPA over all keys: q [H, d], K/V [H, N, d] per head."""
    qt = torch.from_numpy(q.astype(np.float64))[None, :, None, :]
    o = torch.nn.functional.scaled_dot_product_attention(qt, torch.from_numpy(K.astype(np.float64))[None],
                                                         torch.from_numpy(V.astype(np.float64))[None], scale=tau)
    return o[0, :, 0].numpy()


def test_mha_and_gqa_equal_per_head_sdpa():
    B, n_q, H, d, N = 1, 2, 8, 16, 20
    tau = 1 / math.sqrt(d)
    q = rng.standard_normal((B, n_q, H, d)).astype(np.float32)
    for H_kv in (8, 2):
        K = rng.standard_normal((B, N, H_kv, d)).astype(np.float32)
        V = rng.standard_normal((B, N, H_kv, d)).astype(np.float32)
        idx = np.tile(np.arange(N, dtype=np.int32), (B, n_q, 1))       # every key selected
        out, _ = oracle.attention(q, K, V, tau, oracle.SPARSE, idx=idx)
        G = H // H_kv
        Kh = np.repeat(K[0].transpose(1, 0, 2), G, axis=0)              # [H, N, d]
        Vh = np.repeat(V[0].transpose(1, 0, 2), G, axis=0)
        for i in range(n_q):
            assert np.max(np.abs(out[i] - _sdpa(q[0, i], Kh, Vh, tau))) < 1e-12, H_kv


def test_one_kv_head_layouts_agree():
    B, n_q, H, d, N = 1, 3, 4, 8, 12
    q = rng.standard_normal((B, n_q, H, d)).astype(np.float32)
    K = rng.standard_normal((B, N, d)).astype(np.float32)
    V = rng.standard_normal((B, N, d)).astype(np.float32)
    a, la = oracle.attention(q, K, V, 0.3, oracle.CLOSED_BLOCKS, q_pos0=20, m=2)
    b, lb = oracle.attention(q, K[:, :, None], V[:, :, None], 0.3, oracle.CLOSED_BLOCKS, q_pos0=20, m=2)
    assert np.array_equal(a, b) and np.array_equal(la, lb)
