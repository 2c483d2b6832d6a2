"""GPU parity of csa_index_topk's fused route: for decode-shaped calls over
rows longer than one top-k CTA, the indexer kernel also writes each row's
warp maxima (the largest score of every 32 consecutive entries), and the
top-k takes its collection threshold from them -- the k-th largest warp
maximum, below which at least k entries lie -- instead of sampling the row.
The result must be bit-identical to scoring and selecting in two calls (both
routes are exact) and agree with the oracle up to near-ties, including on rows
built so that the collection overflows and the select streams the row (the
best entries clustered at the end of the row, or every score equal)."""
import numpy as np
import pytest
import torch

import oracle
from long_context_compressed_18_b300 import inputs, lib
from helpers import DEV, host, sync_status, topk_near_tie_check

pytestmark = pytest.mark.gpu


def _two_call(B, n_q, q_pos0, m, Nc, k, q, qd, qs, kk, kd, ks):
    scores = torch.empty(B, n_q, Nc, dtype=torch.float32, device=DEV)
    wsb = lib.csa_index_scores_workspace_size(B, Nc, 128, kd)
    ws = lib.empty_workspace(wsb)
    lib.csa_index_scores(B, n_q, q_pos0, m, Nc, 64, 128, q, qd, qs, kk, kd, ks, scores, ws, wsb)
    out = torch.empty(B, n_q, k, dtype=torch.int32, device=DEV)
    tb = lib.csa_topk_select_workspace_size(B, n_q, Nc, k)
    tw = lib.empty_workspace(tb)
    lib.csa_topk_select(B, n_q, q_pos0, m, Nc, k, scores, out, tw, tb)
    return out


def _fused(B, n_q, q_pos0, m, Nc, k, q, qd, qs, kk, kd, ks):
    out = torch.full((B, n_q, k), -7, dtype=torch.int32, device=DEV)
    wb = lib.csa_index_topk_workspace_size(B, n_q, Nc, 64, 128, k, kd)
    ws = lib.empty_workspace(wb)
    lib.csa_index_topk(B, n_q, q_pos0, m, Nc, 64, 128, k, q, qd, qs, kk, kd, ks, out, ws, wb)
    return out


def _inputs(B, n_q, Nc, kind, seed):
    g = torch.Generator().manual_seed(seed)
    qf = torch.randn(B, n_q, 64, 128, generator=g)
    kf = torch.randn(B, Nc, 128, generator=g)
    if kind == "bf16":
        return (qf.to(torch.bfloat16), lib.BF16, None, kf.to(torch.bfloat16), lib.BF16, None)
    q, qs = inputs.quantise_e4m3_lastdim(qf)
    if kind == "e4m3":
        k, ks = inputs.quantise_e4m3_lastdim(kf)
        return q, lib.E4M3, qs, k, lib.E4M3, ks
    k, ks = inputs.random_e2m1_keys(B, Nc, 128, seed + 1)
    return q, lib.E4M3, qs, k, lib.E2M1, ks


def _dev(t):
    return None if t is None else t.to(DEV)


def _oracle_rows(B, n_q, q_pos0, m, Nc, k, q, qd, qs, kk, kd, ks, got, rows):
    kind = {lib.BF16: "bf16", lib.E4M3: "e4m3", lib.E2M1: "e2m1"}
    s64, _, sel = oracle.csa_index_topk(q, qs, kind[qd], kk, ks, kind[kd], q_pos0, m, k, rows=np.array(rows))
    lens = oracle.visible(q_pos0 + np.array(rows) % n_q, m, Nc)
    return topk_near_tie_check(host(got).numpy().reshape(-1, k)[rows], sel, s64, lens, k)


@pytest.mark.parametrize("case", [
    dict(B=3, n_q=1, Nc=262144, k=1024, kind="e4m3"),        # the 1M-context decode shape
    dict(B=2, n_q=1, Nc=40000, k=1024, kind="bf16"),         # just past one top-k CTA
    dict(B=2, n_q=3, Nc=70001, k=2048, kind="e4m3"),         # three queries a sequence, ragged tail
    dict(B=2, n_q=1, Nc=100000, k=4096, kind="e2m1"),        # widened FP4 keys, the largest k
], ids=lambda c: f"{c['kind']}-B{c['B']}-nq{c['n_q']}-Nc{c['Nc']}-k{c['k']}")
def test_fused_matches_two_calls_and_oracle(case):
    B, n_q, Nc, k = case["B"], case["n_q"], case["Nc"], case["k"]
    m = 4
    q_pos0 = 4 * Nc - n_q
    q, qd, qs, kk, kd, ks = _inputs(B, n_q, Nc, case["kind"], seed=Nc % 997)
    args = (B, n_q, q_pos0, m, Nc, k, _dev(q), qd, _dev(qs), _dev(kk), kd, _dev(ks))
    want = _two_call(*args)
    got = _fused(*args)
    again = _fused(*args)
    sync_status()
    assert torch.equal(got, want)                  # both routes are exact: bit-identical
    assert torch.equal(got, again)                 # deterministic
    ties = _oracle_rows(B, n_q, q_pos0, m, Nc, k, q, qd, qs, kk, kd, ks, got, [0, B * n_q - 1])
    print(f"{case}: near-tie rows {ties}")


def test_fused_short_and_long_rows_in_one_call():
    """Queries early in the context see at most k entries (no selection), later
    ones more; the split CTAs of short rows collect nothing."""
    B, n_q, Nc, k = 2, 3, 50000, 1024
    q_pos0 = 4 * 1024 + 1          # rows of 1024, 1024 and 1025 visible entries
    q, qd, qs, kk, kd, ks = _inputs(B, n_q, Nc, "e4m3", seed=5)
    args = (B, n_q, q_pos0, 4, Nc, k, _dev(q), qd, _dev(qs), _dev(kk), kd, _dev(ks))
    got = _fused(*args)
    sync_status()
    assert torch.equal(got, _two_call(*args))
    g = host(got).numpy().reshape(-1, k)
    assert np.array_equal(g[0], np.arange(1024)) and np.array_equal(g[1], np.arange(1024))


def _structured_keys(B, Nc, scale_of_j):
    """E4M3 keys whose scores are sk(j) times one constant: every query head
    and every key is the all-ones vector, so the score order is that of the
    key scales."""
    q = torch.full((B, 1, 64, 128), 0x7E, dtype=torch.uint8)       # 448 * 1/448 = 1
    qs = torch.full((B, 1, 64), 1.0 / 448, dtype=torch.float32)
    kk = torch.full((B, Nc, 128), 0x38, dtype=torch.uint8)         # 1.0
    ks = scale_of_j(torch.arange(Nc, dtype=torch.float64)).float().expand(B, Nc).contiguous()
    return q, lib.E4M3, qs, kk, lib.E4M3, ks


@pytest.mark.parametrize("shape", ["ascending", "equal"])
def test_fused_overflowing_collection_falls_back_exactly(shape):
    """ascending: the k best warp maxima are the last k runs of 32 entries, so
    the threshold takes all 32k of their entries, more than the row's list
    holds, and the select streams the row.  equal: every score ties, every
    entry is collected, and the first k indices win."""
    B, Nc, k = 2, 262144, 1024
    fn = (lambda j: 1.0 + j * 2.0 ** -18) if shape == "ascending" else (lambda j: torch.ones_like(j))
    q, qd, qs, kk, kd, ks = _structured_keys(B, Nc, fn)
    args = (B, 1, 4 * Nc - 1, 4, Nc, k, _dev(q), qd, _dev(qs), _dev(kk), kd, _dev(ks))
    got = _fused(*args)
    sync_status()
    assert torch.equal(got, _two_call(*args))
    g = host(got).numpy().reshape(B, k)
    want = np.arange(Nc - k, Nc) if shape == "ascending" else np.arange(k)
    assert all(np.array_equal(g[b], want) for b in range(B))
