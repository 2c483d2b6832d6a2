"""Context-parallel CSA decode of one long sequence, simulated on CPU ranks.

TEST INFRASTRUCTURE: only the tests may import this module (see the package
header).  It composes the oracle's own steps; nothing here is on the product
path.

The compressed caches of ONE sequence are split by contiguous entry ranges
over the ranks of a ``torch.distributed`` group (any backend; the tests use
gloo on the CPU).  One query at absolute position t (all entries j < nv(t)
visible, "DeepSeek V4 技术解读" §2.1) is answered with one exchange step:

1. every rank scores its entries with the Lightning Indexer and selects its
   local top-k (the same ranking: score descending, index ascending);
2. all-gather of the k (score, global index) candidates of every rank;
3. every rank selects the global top-k among the R*k candidates.  A global
   top-k entry is in its own shard's top-k, so the union of the local lists
   holds the global selection, and concatenating the lists in rank order keeps
   candidates in ascending global index, so a tie on the score still goes to
   the smaller index;
4. every rank attends over the selected entries of its own shard, giving a
   partial output o_r (normalised over its entries) and lse_r (-inf if none);
5. all-gather of (o_r, lse_r), combined in rank order:
   lse = log sum_r exp(lse_r),  o = sum_r exp(lse_r - lse) o_r.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.distributed as dist

from . import attention, csa_index_topk, topk, visible, SPARSE


def shard_bounds(n_c: int, rank: int, world: int):
    """Entries [lo, hi) of rank `rank`: contiguous, sizes differing by at most one."""
    lo = rank * n_c // world
    hi = (rank + 1) * n_c // world
    return lo, hi


def _all_gather(t: torch.Tensor, world: int):
    out = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(out, t.contiguous())
    return out


def cp_csa_decode(q, idx_q, idx_q_scale, q_kind, k_c, v_c, idx_k, idx_k_scale, k_kind, t: int, m: int, k: int,
                  tau: float, group=None):
    """One decode query of one sequence under context parallelism.

    Every rank passes the full query ([1, 1, H, d] attention query,
    [1, 1, H_I, d_I] indexer query and its scale) and ITS OWN shard of the
    caches ([1, n_local, ...]: K_c, V_c, indexer keys and their scales), the
    shards in rank order covering all entries.  Returns (selection [k] global
    indices ascending, -1 padded; out [H, d] fp64; lse [H] fp64), the same on
    every rank."""
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    n_local = int(idx_k.shape[1])
    sizes = _all_gather(torch.tensor([n_local], dtype=torch.int64), world)
    base = int(sum(int(s.item()) for s in sizes[:rank]))
    n_c = int(sum(int(s.item()) for s in sizes))
    nv = int(visible(t, m, n_c))
    # visible entries of this shard
    nv_local = max(0, min(n_local, nv - base))
    # 1. local scores and local top-k (positions within the shard)
    if nv_local > 0:
        # scoring the shard as a cache of its own: a query at local position
        # nv_local * m - 1 sees exactly the shard's first nv_local entries
        s64, s32, sel = csa_index_topk(idx_q, idx_q_scale, q_kind, idx_k, idx_k_scale, k_kind,
                                       nv_local * m - 1, m, k)
        s32 = s32[0]
        sel = sel[0]
    else:
        s32 = np.zeros(n_local, np.float32)
        sel = np.full(k, -1, np.int32)
    cand_idx = np.where(sel >= 0, sel.astype(np.int64) + base, -1)
    cand_score = np.where(sel >= 0, s32[np.maximum(sel, 0)], np.float32(0)).astype(np.float32)
    # 2. exchange the candidates
    all_idx = torch.cat(_all_gather(torch.from_numpy(cand_idx), world)).numpy()
    all_score = torch.cat(_all_gather(torch.from_numpy(cand_score), world)).numpy()
    # 3. global selection: the valid candidates in rank order are in ascending
    # global index, so ranking their positions ranks their indices
    valid = all_idx >= 0
    pos_idx = all_idx[valid]
    row = all_score[valid][None, :]
    pick = topk(row, np.array([row.shape[1]]), k)[0]
    selection = np.where(pick >= 0, pos_idx[np.maximum(pick, 0)], -1).astype(np.int64)
    # 4. partial attention over this shard's selected entries
    mine = (selection >= base) & (selection < base + n_local)
    local = np.full((1, 1, k), -1, np.int32)
    local[0, 0, :int(mine.sum())] = (selection[mine] - base).astype(np.int32)
    o_r, lse_r = attention(q, k_c, v_c, tau, SPARSE, idx=local)
    # 5. exchange and combine in rank order (fp64)
    o_all = _all_gather(torch.from_numpy(o_r[0]), world)
    l_all = _all_gather(torch.from_numpy(lse_r[0]), world)
    lse = np.full(l_all[0].shape, -np.inf)
    for l_ in l_all:
        lse = np.logaddexp(lse, l_.numpy())
    out = np.zeros(o_all[0].shape)
    for o_, l_ in zip(o_all, l_all):
        w = np.where(np.isfinite(l_.numpy()), np.exp(l_.numpy() - np.where(np.isfinite(lse), lse, 0.0)), 0.0)
        out += w[:, None] * o_.numpy()
    return selection, out, lse
