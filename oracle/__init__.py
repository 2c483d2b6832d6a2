"""CPU oracle for the CSA / HCA / SWA path.

TEST INFRASTRUCTURE: only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA path and imports nothing from it.

Thin ctypes marshalling over ``oracle.c`` (plain C, fp64 accumulation), plus
end-to-end drivers that chain the steps in the order the pages give them
("DeepSeek V4 技术解读", §2.1: compress -> Lightning Indexer -> top-k -> core
attention; §2.2: compress -> dense attention; §2.3: sliding window).
"""
from __future__ import annotations

import ctypes as C
import math
import os

import numpy as np
import torch

from .build import build as _build

_lib = None

_P = C.c_void_p
_I = C.c_int
_L = C.c_int64


def lib():
    global _lib
    if _lib is None:
        path = _build()
        _lib = C.CDLL(path)
        sigs = {
            "orc_e4m3_value": ([C.c_uint], C.c_double),
            "orc_e2m1_value": ([C.c_uint], C.c_double),
            "orc_e4m3_encode": ([C.c_float], C.c_uint),
            "orc_e2m1_encode": ([C.c_float], C.c_uint),
            "orc_e4m3_decode_array": ([_L, _P, _P], None),
            "orc_e4m3_encode_array": ([_L, _P, _P], None),
            "orc_e2m1_encode_array": ([_L, _P, _P], None),
            "orc_compress": ([_I, _I, _I, _I, _P, _P, _P], None),
            "orc_compress_per_channel": ([_I, _I, _I, _I, _P, _P, _P], None),
            "orc_quant_e4m3_rows": ([_L, _I, _P, _P, _P], None),
            "orc_quant_e2m1_blocks": ([_L, _I, _P, _P, _P], None),
            "orc_fp4_to_e4m3": ([_L, _I, _P, _P, _P, _P], _L),
            "orc_index_scores": ([_I, _I, _L, _I, _I, _I, _I, _P, _P, _P, _P,
                                  _P, _I, _I, _P, _P, _P], None),
            "orc_topk": ([_I, _P, _L, _I, _P, _P], None),
            "orc_attention": ([_I, _I, _I, _I, _I, _L, _P, _P, _P, C.c_double, _I,
                               _L, _I, _L, _P, _I, _I, _P, _P, _P], None),
            "orc_num_threads": ([], _I),
        }
        for name, (args, res) in sigs.items():
            f = getattr(_lib, name)
            f.argtypes = args
            f.restype = res
    return _lib


def _np(x, dtype):
    """Host copy as a contiguous numpy array of ``dtype`` (bf16 is widened to
    fp32 exactly by torch)."""
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu()
        if x.dtype == torch.bfloat16:
            x = x.float()
        x = x.numpy()
    return np.ascontiguousarray(x, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def num_threads() -> int:
    return lib().orc_num_threads()


# ---- number formats ---------------------------------------------------------

def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e4m3_encode(y) -> np.ndarray:
    y = _np(y, np.float32)
    out = np.empty(y.shape, np.uint8)
    lib().orc_e4m3_encode_array(y.size, _ptr(y), _ptr(out))
    return out


def e2m1_encode(y) -> np.ndarray:
    y = _np(y, np.float32)
    out = np.empty(y.shape, np.uint8)
    lib().orc_e2m1_encode_array(y.size, _ptr(y), _ptr(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    c = _np(codes, np.uint8)
    out = np.empty(c.shape, np.float32)
    lib().orc_e4m3_decode_array(c.size, _ptr(c), _ptr(out))
    return out


def e2m1_decode_packed(packed) -> np.ndarray:
    """Unpack E2M1 pairs (element 2i in the low nibble) to fp32 values."""
    p = _np(packed, np.uint8)
    lo, hi = p & 0xF, p >> 4
    codes = np.stack([lo, hi], -1).reshape(*p.shape[:-1], p.shape[-1] * 2)
    tab = np.array([lib().orc_e2m1_value(i) for i in range(16)], np.float32)
    return tab[codes]


# ---- a1: compression and its quantising epilogues ---------------------------

def compress(logits, x, m: int) -> np.ndarray:
    """[B, n] logits, [B, n, d] x -> fp64 [B, n // m, d]."""
    lg = _np(logits, np.float32)
    xx = _np(x, np.float32)
    B, n, d = xx.shape
    out = np.empty((B, n // m, d), np.float64)
    lib().orc_compress(B, n, m, d, _ptr(lg), _ptr(xx), _ptr(out))
    return out


def compress_per_channel(logits, x, m: int) -> np.ndarray:
    """Per-channel weights: [B, n, d] logits, [B, n, d] x -> fp64 [B, n // m, d]."""
    lg = _np(logits, np.float32)
    xx = _np(x, np.float32)
    B, n, d = xx.shape
    assert lg.shape == xx.shape
    out = np.empty((B, n // m, d), np.float64)
    lib().orc_compress_per_channel(B, n, m, d, _ptr(lg), _ptr(xx), _ptr(out))
    return out


def quant_e4m3_rows(x32):
    x = _np(x32, np.float32)
    rows, d = int(np.prod(x.shape[:-1])), x.shape[-1]
    codes = np.empty(x.shape, np.uint8)
    scale = np.empty(x.shape[:-1], np.float32)
    lib().orc_quant_e4m3_rows(rows, d, _ptr(x), _ptr(codes), _ptr(scale))
    return codes, scale


def quant_e2m1_blocks(x32):
    x = _np(x32, np.float32)
    rows, d = int(np.prod(x.shape[:-1])), x.shape[-1]
    packed = np.empty(x.shape[:-1] + (d // 2,), np.uint8)
    sc = np.empty(x.shape[:-1] + (d // 32,), np.uint8)
    lib().orc_quant_e2m1_blocks(rows, d, _ptr(x), _ptr(packed), _ptr(sc))
    return packed, sc


def fp4_to_e4m3(packed, sc_codes):
    p = _np(packed, np.uint8)
    s = _np(sc_codes, np.uint8)
    d = p.shape[-1] * 2
    rows = int(np.prod(p.shape[:-1]))
    x8 = np.empty(p.shape[:-1] + (d,), np.uint8)
    S = np.empty(p.shape[:-1], np.float32)
    n_rounded = lib().orc_fp4_to_e4m3(rows, d, _ptr(p), _ptr(s), _ptr(x8), _ptr(S))
    return x8, S, int(n_rounded)


# ---- a2: indexer scores -----------------------------------------------------

def index_scores(q_vals, q_scale, k_vals, k_scale, q_pos0: int, m: int,
                 rows=None, head_w=None, relu: bool = False):
    """q_vals [B, n_q, H_I, d_I] and k_vals [B, N_c, d_I] are the decoded
    stored values.  Returns (fp64 scores, fp32 scores), shape [R, N_c]; NaN
    where an entry is not visible.  head_w [B, n_q, H_I] and relu select the
    weighted / ReLU variant."""
    q = _np(q_vals, np.float32)
    k = _np(k_vals, np.float32)
    B, n_q, HI, dI = q.shape
    Nc = k.shape[1]
    qs = None if q_scale is None else _np(q_scale, np.float32)
    ks = None if k_scale is None else _np(k_scale, np.float32)
    rr = None if rows is None else _np(rows, np.int64)
    R = B * n_q if rr is None else rr.size
    o64 = np.empty((R, Nc), np.float64)
    o32 = np.empty((R, Nc), np.float32)
    hw = None if head_w is None else _np(head_w, np.float32)
    lib().orc_index_scores(B, n_q, q_pos0, m, Nc, HI, dI, _ptr(q), _ptr(qs), _ptr(k),
                           _ptr(ks), _ptr(hw), 1 if relu else 0, 0 if rr is None else rr.size, _ptr(rr),
                           _ptr(o64), _ptr(o32))
    return o64, o32


# ---- a3: top-k --------------------------------------------------------------

def topk(scores32, lens, k: int) -> np.ndarray:
    s = _np(scores32, np.float32)
    L = _np(lens, np.int64)
    R, stride = s.shape
    out = np.empty((R, k), np.int32)
    lib().orc_topk(R, _ptr(L), stride, k, _ptr(s), _ptr(out))
    return out


def visible(t, m: int, Nc: int):
    return np.minimum((np.asarray(t, np.int64) + 1) // m, Nc)


# ---- a4 / a5 / a6: attention ------------------------------------------------

SPARSE, CLOSED_BLOCKS, WINDOW = 0, 1, 2


def attention(q, K, V, tau: float, mode: int, q_pos0: int = 0, m: int = 1,
              window: int = 0, idx=None, rows=None):
    """q [B, n_q, H, d]; K, V [B, N_kv, d] (one shared KV head) or
    [B, N_kv, H_kv, d] (query head h reads KV head h // (H // H_kv)).  Returns
    (out [R, H, d], lse [R, H]) in fp64 for the selected flat rows (all rows
    when ``rows`` is None)."""
    qq = _np(q, np.float32)
    KK = _np(K, np.float32)
    VV = _np(V, np.float32)
    B, n_q, H, d = qq.shape
    Nkv = KK.shape[1]
    H_kv = 1 if KK.ndim == 3 else KK.shape[2]
    assert H % H_kv == 0
    ii = None if idx is None else _np(idx, np.int32)
    k = 0 if ii is None else ii.shape[-1]
    rr = None if rows is None else _np(rows, np.int64)
    R = B * n_q if rr is None else rr.size
    out = np.empty((R, H, d), np.float64)
    lse = np.empty((R, H), np.float64)
    lib().orc_attention(B, n_q, H, H_kv, d, Nkv, _ptr(qq), _ptr(KK), _ptr(VV), float(tau),
                        mode, q_pos0, m, window, _ptr(ii), k,
                        0 if rr is None else rr.size, _ptr(rr), _ptr(out), _ptr(lse))
    return out, lse


# ---- end-to-end drivers -----------------------------------------------------

def _values(x, scale=None, kind="float"):
    """Decoded stored values as fp32: E4M3 codes go through the oracle's own
    decoder; bf16/fp32 are widened."""
    if kind == "e4m3":
        return e4m3_decode(x)
    return _np(x, np.float32)


def csa_index_topk(idx_q, idx_q_scale, q_kind, idx_k, idx_k_scale, k_kind,
                   q_pos0: int, m: int, k: int, rows=None, head_w=None, relu: bool = False):
    """Scores and selection for CSA: returns (fp64 scores, fp32 scores,
    top-k [R, k]).  k_kind "e2m1" takes packed codes + E4M3 block scales and
    runs the FP4 -> E4M3 conversion first."""
    if k_kind == "e2m1":
        x8, S, _ = fp4_to_e4m3(idx_k, idx_k_scale)
        kv, ks = e4m3_decode(x8), S
    elif k_kind == "e4m3":
        kv, ks = e4m3_decode(idx_k), _np(idx_k_scale, np.float32)
    else:
        kv, ks = _np(idx_k, np.float32), None
    B, n_q = idx_q.shape[:2]
    Nc = kv.shape[1]
    if rows is None:
        qv = e4m3_decode(idx_q) if q_kind == "e4m3" else _np(idx_q, np.float32)
        qs = None if idx_q_scale is None else _np(idx_q_scale, np.float32)
        s64, s32 = index_scores(qv, qs, kv, ks, q_pos0, m, head_w=head_w, relu=relu)
        flat = np.arange(B * n_q)
    else:
        # only the requested rows' queries are decoded: each row is scored as
        # a batch of one at its own position, against its sequence's keys
        flat = _np(rows, np.int64)
        s64 = np.empty((flat.size, Nc), np.float64)
        s32 = np.empty((flat.size, Nc), np.float32)
        for r, f in enumerate(flat):
            b, i = int(f) // n_q, int(f) % n_q
            q1 = idx_q[b:b + 1, i:i + 1]
            qv = e4m3_decode(q1) if q_kind == "e4m3" else _np(q1, np.float32)
            qs = None if idx_q_scale is None else _np(idx_q_scale[b:b + 1, i:i + 1], np.float32)
            ks1 = None if ks is None else ks[b:b + 1]
            hw1 = None if head_w is None else _np(head_w[b:b + 1, i:i + 1], np.float32)
            s64[r:r + 1], s32[r:r + 1] = index_scores(qv, qs, kv[b:b + 1], ks1, q_pos0 + i, m, head_w=hw1,
                                                      relu=relu)
    lens = visible(q_pos0 + flat % n_q, m, Nc)
    sel = topk(s32, lens, k)
    return s64, s32, sel


def compress_stream(logits, x, m: int, out_kind: str):
    """Compression of one stream with the output in ``out_kind``:
    "f64" (unrounded), "f32"/"bf16" (rounded), "e4m3" (codes + row scale) or
    "e2m1" (packed codes + E4M3 block scales)."""
    c = compress(logits, x, m)
    if out_kind == "f64":
        return c
    c32 = c.astype(np.float32)
    if out_kind == "f32":
        return c32
    if out_kind == "bf16":
        return torch.from_numpy(c32).to(torch.bfloat16)
    if out_kind == "e4m3":
        return quant_e4m3_rows(c32)
    if out_kind == "e2m1":
        return quant_e2m1_blocks(c32)
    raise ValueError(out_kind)
