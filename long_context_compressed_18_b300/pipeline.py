"""Layer-level entry points over the C ABI: allocate outputs and workspaces
with torch on the current device and stream, then call the library.  No
arithmetic of the path happens here.

The order of calls follows "DeepSeek V4 技术解读": CSA = compress (§2.1) ->
Lightning Indexer + top-k -> core attention; HCA = compress at m'=128 (§2.2)
-> dense attention; the first layers of the stack are sliding-window
attention (§2.3).
"""
from __future__ import annotations

import math

import torch

from . import lib

_CODE = {"f32": lib.F32, "bf16": lib.BF16, "e4m3": lib.E4M3, "e2m1": lib.E2M1}


class Workspace:
    """A growable caller-owned scratch buffer (the library allocates nothing)."""

    def __init__(self, device="cuda"):
        self.device = device
        self.buf = None

    def get(self, nbytes: int):
        nbytes = max(int(nbytes), 16)
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        return self.buf, self.buf.numel()


def _code(t: torch.Tensor) -> int:
    return lib.dtype_code(t.dtype)


def compress(logits, xs, m: int, out_kinds):
    """xs: list of [B, n, d] tensors sharing logits [B, n].  out_kinds: list of
    "f32" | "bf16" | "e4m3" | "e2m1".  Returns a list of (out, scale)."""
    B, n = logits.shape
    Nc = n // m
    outs, scales = [], []
    for x, kind in zip(xs, out_kinds):
        d = x.shape[-1]
        if kind == "e4m3":
            o = torch.empty(B, Nc, d, dtype=torch.uint8, device=x.device)
            s = torch.empty(B, Nc, dtype=torch.float32, device=x.device)
        elif kind == "e2m1":
            o = torch.empty(B, Nc, d // 2, dtype=torch.uint8, device=x.device)
            s = torch.empty(B, Nc, d // 32, dtype=torch.uint8, device=x.device)
        else:
            o = torch.empty(B, Nc, d, dtype=torch.float32 if kind == "f32" else torch.bfloat16, device=x.device)
            s = None
        outs.append(o)
        scales.append(s)
    lib.csa_compress(B, n, m, logits, list(xs), [_code(x) for x in xs], [x.shape[-1] for x in xs], outs,
                     [_CODE[k] for k in out_kinds], scales)
    return list(zip(outs, scales))


def index_topk(q_idx, q_dtype: str, q_scale, k_idx, k_dtype: str, k_scale, q_pos0: int, m: int, N_c: int,
               k: int, ws: Workspace, score_dtype: str = "f32"):
    B, n_q, H_I, d_I = q_idx.shape[0], q_idx.shape[1], q_idx.shape[2], q_idx.shape[3]
    topk = torch.empty(B, n_q, k, dtype=torch.int32, device=q_idx.device)
    nbytes = lib.csa_index_topk_workspace_size(B, n_q, N_c, H_I, d_I, k, _CODE[k_dtype], _CODE[score_dtype])
    buf, nb = ws.get(nbytes)
    lib.csa_index_topk(B, n_q, q_pos0, m, N_c, H_I, d_I, k, q_idx, _CODE[q_dtype], q_scale, k_idx,
                       _CODE[k_dtype], k_scale, topk, buf, nb, score_dtype=_CODE[score_dtype])
    return topk


def sparse_attn(q, k_c, v_c, topk, scale: float, ws: Workspace, want_lse=True):
    B, n_q, H, d = q.shape
    N_c, k = k_c.shape[1], topk.shape[-1]
    out = torch.empty_like(q)
    lse = torch.empty(B, n_q, H, dtype=torch.float32, device=q.device) if want_lse else None
    buf, nb = ws.get(lib.csa_sparse_attn_workspace_size(B, n_q, H, d, k))
    lib.csa_sparse_attn(B, n_q, H, d, N_c, k, scale, q, k_c, v_c, _code(q), topk, out, lse, buf, nb)
    return out, lse


def hca(q, k_c, v_c, q_pos0: int, m: int, scale: float, want_lse=True):
    B, n_q, H, d = q.shape
    out = torch.empty_like(q)
    lse = torch.empty(B, n_q, H, dtype=torch.float32, device=q.device) if want_lse else None
    lib.hca_attn(B, n_q, q_pos0, m, k_c.shape[1], H, d, scale, q, k_c, v_c, _code(q), out, lse)
    return out, lse


def swa(q, k, v, q_pos0: int, window: int, scale: float, want_lse=True):
    B, n_q, H, d = q.shape
    out = torch.empty_like(q)
    lse = torch.empty(B, n_q, H, dtype=torch.float32, device=q.device) if want_lse else None
    lib.swa_attn(B, n_q, q_pos0, k.shape[1], window, H, d, scale, q, k, v, _code(q), out, lse)
    return out, lse


# ---- whole layers ------------------------------------------------------------

def csa_layer(x: dict, s, ws: Workspace):
    """CSA prefill layer: compress K, V and indexer K (shared logits), score,
    select top-k, attend.  Returns a dict with the intermediate results."""
    (kc, _), (vc, _), (ikc, iks) = compress(x["logits"], [x["k"], x["v"], x["idx_k"]], s.m,
                                            [s.dtype, s.dtype, s.idx_k_dtype])
    topk = index_topk(x["idx_q"], s.idx_q_dtype, x["idx_q_scale"], ikc, s.idx_k_dtype, iks, s.q_pos0, s.m,
                      s.N_c, s.k, ws)
    out, lse = sparse_attn(x["q"], kc, vc, topk, 1.0 / math.sqrt(s.d), ws)
    return dict(k_c=kc, v_c=vc, idx_k_c=ikc, idx_k_c_scale=iks, topk=topk, out=out, lse=lse)


def csa_decode(x: dict, s, ws: Workspace, score_dtype: str = "f32"):
    """One CSA decode step over resident compressed caches: score, select,
    attend (the headline path).  score_dtype "bf16" stores the index scores
    in bf16."""
    topk = index_topk(x["idx_q"], s.idx_q_dtype, x["idx_q_scale"], x["idx_k_c"], s.idx_k_dtype,
                      x["idx_k_c_scale"], s.q_pos0, s.m, s.N_c, s.k, ws, score_dtype)
    out, lse = sparse_attn(x["q"], x["k_c"], x["v_c"], topk, 1.0 / math.sqrt(s.d), ws)
    return dict(topk=topk, out=out, lse=lse)


def hca_layer(x: dict, s):
    (kc, _), (vc, _) = compress(x["logits"], [x["k"], x["v"]], s.m, [s.dtype, s.dtype])
    out, lse = hca(x["q"], kc, vc, s.q_pos0, s.m, 1.0 / math.sqrt(s.d))
    return dict(k_c=kc, v_c=vc, out=out, lse=lse)


def swa_layer(x: dict, s):
    out, lse = swa(x["q"], x["k"], x["v"], s.q_pos0, s.window, 1.0 / math.sqrt(s.d))
    return dict(out=out, lse=lse)


def run_layer(x: dict, s, ws: Workspace):
    if s.kind == "csa":
        return csa_layer(x, s, ws)
    if s.kind == "csa_decode":
        return csa_decode(x, s, ws)
    if s.kind == "hca":
        return hca_layer(x, s)
    if s.kind == "swa":
        return swa_layer(x, s)
    raise ValueError(s.kind)
