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


class DecodeState:
    """Streaming CSA decode state of B sequences ("DeepSeek V4 技术解读" §2.1
    applied one token at a time): compressed K/V and indexer-key caches of
    capacity N_cap entries, the open block of raw tokens, and the per-sequence
    token counts, all on the device.  ``append`` adds one token to every
    sequence (closing and compressing a block every m tokens); ``select``
    runs the Lightning Indexer and top-k for each sequence's new query at its
    own position; ``attend`` is the sparse attention over the selection."""

    def __init__(self, B: int, m: int, d: int, d_I: int, N_cap: int, x_dtype=torch.bfloat16,
                 kv_dtype=torch.bfloat16, ik_kind: str = "e4m3", device="cuda"):
        self.B, self.m, self.d, self.d_I, self.N_cap = B, m, d, d_I, N_cap
        self.x_dtype, self.ik_kind = x_dtype, ik_kind
        self.stage_logits = torch.zeros(B, m, dtype=torch.float32, device=device)
        self.stage_k = torch.zeros(B, m, d, dtype=x_dtype, device=device)
        self.stage_v = torch.zeros(B, m, d, dtype=x_dtype, device=device)
        self.stage_ik = torch.zeros(B, m, d_I, dtype=x_dtype, device=device)
        self.lens = torch.zeros(B, dtype=torch.int64, device=device)
        self.k_c = torch.zeros(B, N_cap, d, dtype=kv_dtype, device=device)
        self.v_c = torch.zeros(B, N_cap, d, dtype=kv_dtype, device=device)
        if ik_kind == "e4m3":
            self.ik_c = torch.zeros(B, N_cap, d_I, dtype=torch.uint8, device=device)
            self.ik_scale = torch.ones(B, N_cap, dtype=torch.float32, device=device)
        elif ik_kind == "e2m1":
            self.ik_c = torch.zeros(B, N_cap, d_I // 2, dtype=torch.uint8, device=device)
            self.ik_scale = torch.zeros(B, N_cap, d_I // 32, dtype=torch.uint8, device=device)
        else:
            self.ik_c = torch.zeros(B, N_cap, d_I, dtype=torch.float32 if ik_kind == "f32" else torch.bfloat16,
                                    device=device)
            self.ik_scale = None

    def append(self, logit, k, v, ik):
        """One token for every sequence: logit fp32 [B], k/v [B, d], ik [B, d_I]."""
        lib.csa_decode_append(self.B, self.m, self.d, self.d_I, self.N_cap, logit, k, v, ik, _code(k),
                              self.stage_logits, self.stage_k, self.stage_v, self.stage_ik, self.lens, self.k_c,
                              self.v_c, _code(self.k_c), self.ik_c, _CODE[self.ik_kind], self.ik_scale)

    def select(self, q_idx, q_dtype: str, q_scale, k: int, ws: Workspace, score_dtype: str = "f32",
               head_weight=None, relu: bool = False):
        """Top-k entries for the last n_q tokens of each sequence."""
        B, n_q, H_I, d_I = q_idx.shape
        topk = torch.empty(B, n_q, k, dtype=torch.int32, device=q_idx.device)
        nbytes = lib.csa_index_topk_workspace_size(B, n_q, self.N_cap, H_I, d_I, k, _CODE[self.ik_kind],
                                                   _CODE[score_dtype])
        buf, nb = ws.get(nbytes)
        lib.csa_index_topk_varlen(B, n_q, self.lens, self.m, self.N_cap, H_I, d_I, k, q_idx, _CODE[q_dtype], q_scale,
                                  self.ik_c, _CODE[self.ik_kind], self.ik_scale, topk, buf, nb,
                                  score_dtype=_CODE[score_dtype], head_weight=head_weight, relu=relu)
        return topk

    def attend(self, q, topk, scale: float, ws: Workspace, want_lse=True):
        return sparse_attn(q, self.k_c, self.v_c, topk, scale, ws, want_lse)
