"""Workload shapes for the hybrid long-context attention path.

The five named workloads restate the sizes DeepSeek-V4's CSA/HCA description
fixes (takeshell.com "DeepSeek V4 技术解读" §2.1: m=4, 64 indexer heads of
dim 128, top-k=1024; §2.2: m'=128; §2.3: two sliding-window layers, then CSA
and HCA alternate) plus the spec's choices for batch, context and precision.

Small shapes used by the parity tests are built with :func:`shape`.
"""
from __future__ import annotations

import dataclasses
import math


@dataclasses.dataclass(frozen=True)
class Shape:
    name: str
    kind: str            # "csa" | "csa_decode" | "hca" | "swa" | "stack"
    B: int               # batch
    n: int               # context tokens (raw)
    m: int               # compression ratio
    n_q: int             # query tokens per sequence
    q_pos0: int          # absolute position of the first query token
    H: int               # attention heads
    d: int               # attention head dim
    H_I: int = 0         # indexer heads
    d_I: int = 0         # indexer head dim
    k: int = 0           # top-k
    window: int = 0      # sliding window (swa)
    dtype: str = "bf16"  # attention I/O: "f32" | "bf16"
    idx_q_dtype: str = "bf16"   # "f32" | "bf16" | "e4m3"
    idx_k_dtype: str = "bf16"   # "f32" | "bf16" | "e4m3" | "e2m1"
    qkv_scale: float = 1.0      # multiplier applied to attention Q/K/V draws
    seed: int = 20261202

    @property
    def N_c(self) -> int:
        """Closed compressed entries: floor(n / m)."""
        return self.n // self.m

    @property
    def tau(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def nv(self, t: int) -> int:
        """Compressed entries visible to the query at absolute position t."""
        return min((t + 1) // self.m, self.N_c)


def shape(**kw) -> Shape:
    kw.setdefault("name", "custom")
    return Shape(**kw)


# --- the five named workloads -------------------------------------------------

TINY_CSA_F32 = Shape(
    name="tiny_csa_f32", kind="csa", B=1, n=1024, m=4, n_q=1024, q_pos0=0,
    H=8, d=64, H_I=4, d_I=32, k=64, dtype="f32", idx_q_dtype="f32",
    idx_k_dtype="f32", seed=20261202 + 1)

CSA_PREFILL_BF16 = Shape(
    name="csa_prefill_bf16_n32768", kind="csa", B=1, n=32768, m=4, n_q=32768,
    q_pos0=0, H=64, d=128, H_I=64, d_I=128, k=1024, dtype="bf16",
    idx_q_dtype="bf16", idx_k_dtype="bf16", qkv_scale=1.0 / math.sqrt(128.0),
    seed=20261202 + 2)

CSA_DECODE_1M = Shape(
    name="csa_decode_b32_ctx1m_e4m3", kind="csa_decode", B=32, n=1 << 20, m=4,
    n_q=1, q_pos0=(1 << 20) - 1, H=64, d=128, H_I=64, d_I=128, k=1024,
    dtype="bf16", idx_q_dtype="e4m3", idx_k_dtype="e4m3", seed=20261202 + 3)

HCA_PREFILL_1M = Shape(
    name="hca_prefill_ctx1m_q16384", kind="hca", B=1, n=1 << 20, m=128,
    n_q=16384, q_pos0=(1 << 20) - 16384, H=64, d=128, dtype="bf16",
    seed=20261202 + 4)

STACK_N = 131072
STACK_LAYERS = (
    Shape(name="stack_swa0", kind="swa", B=1, n=STACK_N, m=1, n_q=STACK_N,
          q_pos0=0, H=64, d=128, window=128, seed=20261202 + 50),
    Shape(name="stack_swa1", kind="swa", B=1, n=STACK_N, m=1, n_q=STACK_N,
          q_pos0=0, H=64, d=128, window=128, seed=20261202 + 51),
    Shape(name="stack_csa2", kind="csa", B=1, n=STACK_N, m=4, n_q=STACK_N,
          q_pos0=0, H=64, d=128, H_I=64, d_I=128, k=1024, idx_q_dtype="e4m3",
          idx_k_dtype="e2m1", seed=20261202 + 52),
    Shape(name="stack_hca3", kind="hca", B=1, n=STACK_N, m=128, n_q=STACK_N,
          q_pos0=0, H=64, d=128, seed=20261202 + 53),
    Shape(name="stack_csa4", kind="csa", B=1, n=STACK_N, m=4, n_q=STACK_N,
          q_pos0=0, H=64, d=128, H_I=64, d_I=128, k=1024, idx_q_dtype="e4m3",
          idx_k_dtype="e2m1", seed=20261202 + 54),
    Shape(name="stack_hca5", kind="hca", B=1, n=STACK_N, m=128, n_q=STACK_N,
          q_pos0=0, H=64, d=128, seed=20261202 + 55),
)

NAMED = {s.name: s for s in (TINY_CSA_F32, CSA_PREFILL_BF16, CSA_DECODE_1M,
                             HCA_PREFILL_1M) + STACK_LAYERS}
