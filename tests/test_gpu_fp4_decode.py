"""FP4 indexer-key cache at decode ("DeepSeek V4 技术解读" §五: the indexer's
QK path takes FP4 keys, widened to FP8 for the product).  Decode groups (one
to three queries a sequence) widen the packed E2M1 keys inside the indexer
kernel; the widening must equal the oracle's FP4 -> E4M3 conversion
(orc_fp4_to_e4m3) exactly.

* Scores of the in-kernel route equal, bit for bit, the E4M3 route's scores
  on the oracle's widened keys and row scales -- every nibble value (signed
  zero included) and block scales from the smallest subnormal E4M3 to 448.
* Top-k over a 1M-context FP4 cache against the oracle's widening, scoring
  and selection (near-ties only)."""
import numpy as np
import pytest
import torch

import oracle
from long_context_compressed_18_b300 import inputs, lib
from helpers import DEV, host, sync_status, topk_near_tie_check

pytestmark = pytest.mark.gpu


def _wide_scale_keys(B, Nc, seed):
    """Random nibbles with block scales spread over the whole positive E4M3
    range (codes 0x01 .. 0x7E), so rows' scales S and the per-block ratios
    sc / S take every exponent the format allows."""
    g = torch.Generator().manual_seed(seed)
    packed = torch.randint(0, 256, (B, Nc, 64), generator=g, dtype=torch.int64).to(torch.uint8)
    sc = torch.randint(1, 0x7F, (B, Nc, 4), generator=g, dtype=torch.int64).to(torch.uint8)
    sc[:, ::7, :] = 0x01                                      # whole rows at the smallest subnormal
    sc[:, 3::11, 2] = 0x7E                                    # 448 beside small blocks
    return packed.contiguous(), sc.contiguous()


def _scores(B, n_q, q_pos0, Nc, q, qs, k, kc, ks):
    out = torch.full((B, n_q, Nc), float("nan"), device=DEV)
    wb = lib.csa_index_scores_workspace_size(B, Nc, 128, kc)
    ws = lib.empty_workspace(wb)
    lib.csa_index_scores(B, n_q, q_pos0, 4, Nc, 64, 128, q, lib.E4M3, qs, k, kc, ks, out, ws, wb)
    return out


@pytest.mark.parametrize("case", [
    dict(B=3, n_q=1, Nc=6001, keys="random"),
    dict(B=2, n_q=3, Nc=2000, keys="wide"),
    dict(B=1, n_q=2, Nc=129, keys="wide"),
])
def test_fp4_decode_scores_equal_e4m3_route_on_widened_keys(case):
    B, n_q, Nc = case["B"], case["n_q"], case["Nc"]
    g = torch.Generator().manual_seed(Nc)
    q, qs = inputs.quantise_e4m3_lastdim(torch.randn(B, n_q, 64, 128, generator=g))
    if case["keys"] == "random":
        k, ks = inputs.random_e2m1_keys(B, Nc, 128, Nc + 1)
    else:
        k, ks = _wide_scale_keys(B, Nc, Nc + 1)
    x8, S, _ = oracle.fp4_to_e4m3(k, ks)                 # the oracle's widening
    q_pos0 = 4 * Nc - n_q
    fp4 = _scores(B, n_q, q_pos0, Nc, q.to(DEV), qs.to(DEV), k.to(DEV), lib.E2M1, ks.to(DEV))
    e4m3 = _scores(B, n_q, q_pos0, Nc, q.to(DEV), qs.to(DEV), torch.from_numpy(x8).to(DEV), lib.E4M3,
                   torch.from_numpy(S).to(DEV))
    sync_status()
    a, b = host(fp4), host(e4m3)
    assert torch.equal(torch.isnan(a), torch.isnan(b))
    vis = ~torch.isnan(a)
    assert vis.any()
    assert torch.equal(a[vis].view(torch.int32), b[vis].view(torch.int32))


@pytest.mark.parametrize("B,Nc,k", [(3, 262144, 1024), (2, 70001, 2048)])
def test_fp4_decode_topk_against_oracle(B, Nc, k):
    g = torch.Generator().manual_seed(B + Nc)
    q, qs = inputs.quantise_e4m3_lastdim(torch.randn(B, 1, 64, 128, generator=g))
    kk, ks = inputs.random_e2m1_keys(B, Nc, 128, Nc % 991)
    q_pos0 = 4 * Nc - 1
    topk = torch.empty(B, 1, k, dtype=torch.int32, device=DEV)
    wb = lib.csa_index_topk_workspace_size(B, 1, Nc, 64, 128, k, lib.E2M1)
    ws = lib.empty_workspace(wb)
    lib.csa_index_topk(B, 1, q_pos0, 4, Nc, 64, 128, k, q.to(DEV), lib.E4M3, qs.to(DEV), kk.to(DEV), lib.E2M1,
                       ks.to(DEV), topk, ws, wb)
    sync_status()
    s64, _, sel = oracle.csa_index_topk(q, qs, "e4m3", kk, ks, "e2m1", q_pos0, 4, k)
    ties = topk_near_tie_check(host(topk).numpy().reshape(B, k), sel, s64, [Nc] * B, k)
    print(f"FP4 decode B={B} Nc={Nc} k={k}: near-tie rows {ties}")
