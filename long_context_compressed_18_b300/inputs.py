"""Seeded synthetic inputs for the CSA / HCA / SWA path.

This module only draws random numbers and lays them out; it holds none of the
path's arithmetic (no compression, scoring, selection or attention).  Both the
CUDA path and the CPU oracle consume the tensors it returns, byte for byte.

Draw recipe (all values N(0,1) unless stated; one ``torch.Generator`` per
sequence, seeded with ``seed + 1000 * (b + 1)``, so a sequence's inputs do not
depend on the batch it sits in):

* prefill CSA / HCA / SWA: per sequence, in this order: compression logits
  ``[n]`` fp32, K ``[n, d]``, V ``[n, d]``, indexer K ``[n, d_I]``, Q
  ``[n_q, H, d]``, indexer Q ``[n_q, H_I, d_I]``.  Attention Q/K/V are
  multiplied by ``qkv_scale`` (1/sqrt(128) for the BF16 prefill workload).
* decode CSA: the compressed caches are drawn directly (there is no raw-token
  history to compress): K_c ``[N_c, d]``, V_c ``[N_c, d]``, indexer K_c
  ``[N_c, d_I]``, then Q ``[1, H, d]``, indexer Q ``[1, H_I, d_I]``.

Tensors that the path receives already quantised (E4M3 indexer queries with a
per-(token, head) fp32 scale; the decode workload's E4M3 indexer-key cache
with a per-row fp32 scale) are produced here with torch's own
``float8_e4m3fn`` cast: scale = amax / 448 (1 where amax = 0), code =
cast(x * (448 / amax)).  That is input preparation upstream of the path, not a
step of it; the path and the oracle both read value = decode(code) * scale.
"""
from __future__ import annotations

import torch

from .configs import Shape

_TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _gen(shape: Shape, b: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(shape.seed + 1000 * (b + 1))
    return g


def quantise_e4m3_lastdim(x: torch.Tensor):
    """Input-side E4M3 quantisation with torch's cast: returns (uint8 codes,
    fp32 scale over the last dim)."""
    x = x.float()
    amax = x.abs().amax(dim=-1, keepdim=True)
    safe = torch.where(amax > 0, amax, torch.ones_like(amax))
    inv = torch.where(amax > 0, 448.0 / safe, torch.ones_like(amax))
    codes = (x * inv).to(torch.float8_e4m3fn).view(torch.uint8)
    scale = torch.where(amax > 0, safe / 448.0, torch.ones_like(amax))
    return codes.contiguous(), scale.squeeze(-1).contiguous()


def _store(x: torch.Tensor, dt: str):
    if dt in _TORCH_DT:
        return x.to(_TORCH_DT[dt]).contiguous(), None
    if dt == "e4m3":
        return quantise_e4m3_lastdim(x)
    raise ValueError(dt)


def make_inputs(shape: Shape, device="cpu", batches=None) -> dict:
    """Draw every input of ``shape``.  ``batches`` restricts the draw to a
    subset of sequence indices (the result is then stacked in that order)."""
    bs = list(range(shape.B)) if batches is None else list(batches)
    per = [_one_sequence(shape, b, device) for b in bs]
    out = {}
    for key in per[0]:
        vals = [p[key] for p in per]
        out[key] = None if vals[0] is None else torch.stack(vals, 0).contiguous()
    return out


def _one_sequence(s: Shape, b: int, device) -> dict:
    g = _gen(s, b, device)
    f32 = dict(device=device, dtype=torch.float32, generator=g)
    adt = s.dtype
    r = {}
    if s.kind == "csa_decode":
        N = s.N_c
        r["k_c"] = (torch.randn(N, s.d, **f32) * s.qkv_scale).to(_TORCH_DT[adt]).contiguous()
        r["v_c"] = (torch.randn(N, s.d, **f32) * s.qkv_scale).to(_TORCH_DT[adt]).contiguous()
        r["idx_k_c"], r["idx_k_c_scale"] = _store(torch.randn(N, s.d_I, **f32), s.idx_k_dtype)
        r["q"] = (torch.randn(s.n_q, s.H, s.d, **f32) * s.qkv_scale).to(_TORCH_DT[adt]).contiguous()
        r["idx_q"], r["idx_q_scale"] = _store(torch.randn(s.n_q, s.H_I, s.d_I, **f32), s.idx_q_dtype)
        return r
    n = s.n
    r["logits"] = torch.randn(n, **f32).contiguous() if s.kind in ("csa", "hca") else None
    r["k"] = (torch.randn(n, s.d, **f32) * s.qkv_scale).to(_TORCH_DT[adt]).contiguous()
    r["v"] = (torch.randn(n, s.d, **f32) * s.qkv_scale).to(_TORCH_DT[adt]).contiguous()
    if s.kind == "csa":
        ik = torch.randn(n, s.d_I, **f32)
        # raw indexer keys are stored in the attention I/O precision; the
        # compression call quantises the compressed entries itself
        r["idx_k"] = ik.to(_TORCH_DT[adt]).contiguous()
    else:
        r["idx_k"] = None
    r["q"] = (torch.randn(s.n_q, s.H, s.d, **f32) * s.qkv_scale).to(_TORCH_DT[adt]).contiguous()
    if s.kind == "csa":
        r["idx_q"], r["idx_q_scale"] = _store(torch.randn(s.n_q, s.H_I, s.d_I, **f32), s.idx_q_dtype)
    else:
        r["idx_q"], r["idx_q_scale"] = None, None
    return r


def random_index_sets(shape: Shape, seed: int, device="cpu") -> torch.Tensor:
    """A uniformly random valid selection per query: min(k, nv(t)) distinct
    visible entries in ascending order, -1 padded.  Used to drive the sparse
    attention stage with a selection both sides receive as input."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = torch.full((shape.B, shape.n_q, shape.k), -1, dtype=torch.int32)
    for b in range(shape.B):
        for i in range(shape.n_q):
            nv = shape.nv(shape.q_pos0 + i)
            c = min(shape.k, nv)
            if c == 0:
                continue
            sel = torch.randperm(nv, generator=g)[:c].sort().values
            out[b, i, :c] = sel.to(torch.int32)
    return out.to(device)


def random_scores(rows: int, length: int, seed: int, tie_levels: int = 0) -> torch.Tensor:
    """fp32 score rows for the selection stage.  With ``tie_levels`` > 0 the
    values are drawn from that many distinct levels so exact ties are common;
    a few signed zeros are planted either way."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if tie_levels > 0:
        x = torch.randint(-tie_levels, tie_levels, (rows, length), generator=g).float() * 0.125
    else:
        x = torch.randn(rows, length, generator=g)
    if length >= 8:
        x[:, 1] = 0.0
        x[:, 3] = -0.0
    return x.contiguous()


def random_e2m1_keys(B: int, N: int, d: int, seed: int):
    """Packed E2M1 codes [B, N, d/2] (uniform random nibbles) and E4M3 block
    scales [B, N, d/32] (torch's cast of |N(0,1)|/6 + 1/64, so every block has a
    positive scale with varied mantissas and exponents)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    packed = torch.randint(0, 256, (B, N, d // 2), generator=g, dtype=torch.int64).to(torch.uint8)
    s = torch.randn(B, N, d // 32, generator=g).abs() / 6.0 + 1.0 / 64
    sc = s.to(torch.float8_e4m3fn).view(torch.uint8)
    return packed.contiguous(), sc.contiguous()
