"""Small, fixed kernel cases for profiler captures and per-kernel timing.

Each case calls the C ABI on seeded N(0,1) inputs that are larger than L2
where the kernel streams (so DRAM counters mean something) but small enough
for an ``ncu --set full`` capture to end in a minute or two.  Every case runs
twice, so a capture can skip the first (cold) round; ``--time`` also prints
CUDA-event timings of each case: 20 replays of a CUDA graph of the call, and
20 eager calls.

    python profile_cases.py attn [--time]
    python profile_cases.py indexer [--time]
    python profile_cases.py topk [--time]
    python profile_cases.py compress [--time]
"""
from __future__ import annotations

import argparse
import math
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from long_context_compressed_18_b300 import inputs, lib  # noqa: E402

DEV = "cuda"


def _attn_cases():
    """Sparse (prefill- and decode-shaped), HCA and SWA attention, 64 x 128."""
    g = torch.Generator(device="cpu").manual_seed(11)
    bf = torch.bfloat16
    H, d = 64, 128
    tau = 1.0 / math.sqrt(d)

    def rnd(*shape):
        return torch.randn(*shape, generator=g).to(bf).to(DEV)

    cases = []
    nq, Nc, k = 2048, 8192, 1024
    q, K, V = rnd(1, nq, H, d), rnd(1, Nc, d), rnd(1, Nc, d)
    idx = torch.randint(0, Nc, (1, nq, k), generator=g, dtype=torch.int32).sort(-1).values.contiguous().to(DEV)
    o, l = torch.empty_like(q), torch.empty(1, nq, H, device=DEV)
    cases.append(("sparse_prefill_q2048_k1024", 4.0 * H * d * nq * k,
                  lambda: lib.csa_sparse_attn(1, nq, H, d, Nc, k, tau, q, K, V, lib.BF16, idx, o, l)))
    nq2, Nc2 = 2048, 8192
    q2, K2, V2 = rnd(1, nq2, H, d), rnd(1, Nc2, d), rnd(1, Nc2, d)
    o2, l2 = torch.empty_like(q2), torch.empty(1, nq2, H, device=DEV)
    p0 = (1 << 20) - nq2
    flops2 = 4.0 * H * d * sum(min((p0 + i + 1) // 128, Nc2) for i in range(nq2))
    cases.append(("hca_ctx1m_q2048", flops2,
                  lambda: lib.hca_attn(1, nq2, p0, 128, Nc2, H, d, tau, q2, K2, V2, lib.BF16, o2, l2)))
    B3, Nc3 = 8, 262144
    q3, K3, V3 = rnd(B3, 1, H, d), rnd(B3, Nc3, d), rnd(B3, Nc3, d)
    idx3 = torch.randint(0, Nc3, (B3, 1, k), generator=g, dtype=torch.int32).sort(-1).values.contiguous().to(DEV)
    o3, l3 = torch.empty_like(q3), torch.empty(B3, 1, H, device=DEV)
    wsb = lib.csa_sparse_attn_workspace_size(B3, 1, H, d, k)
    ws = lib.empty_workspace(wsb)
    cases.append(("sparse_decode_b8_k1024", 4.0 * H * d * B3 * k,
                  lambda: lib.csa_sparse_attn(B3, 1, H, d, Nc3, k, tau, q3, K3, V3, lib.BF16, idx3, o3, l3, ws, wsb)))
    nq4 = 8192
    q4, K4, V4 = rnd(1, nq4, H, d), rnd(1, nq4, d), rnd(1, nq4, d)
    o4, l4 = torch.empty_like(q4), torch.empty(1, nq4, H, device=DEV)
    flops4 = 4.0 * H * d * sum(min(128, i + 1) for i in range(nq4))
    cases.append(("swa_q8192_w128", flops4,
                  lambda: lib.swa_attn(1, nq4, 0, nq4, 128, H, d, tau, q4, K4, V4, lib.BF16, o4, l4)))
    return cases, "TFLOP/s"


def _indexer_cases():
    """Prefill-shaped Lightning Indexer scores: 2048 queries over the last
    8192 entries, BF16 x BF16 and E4M3 x E4M3, 64 heads x 128."""
    g = torch.Generator(device="cpu").manual_seed(12)
    B, nq, Nc = 1, 2048, 8192
    q_pos0 = 4 * Nc - nq
    qf, kf = torch.randn(B, nq, 64, 128, generator=g), torch.randn(B, Nc, 128, generator=g)
    scores = torch.empty(B, nq, Nc, device=DEV)
    qb, kb = qf.to(torch.bfloat16).to(DEV), kf.to(torch.bfloat16).to(DEV)
    q8, qs8 = (t.to(DEV) for t in inputs.quantise_e4m3_lastdim(qf))
    k8, ks8 = (t.to(DEV) for t in inputs.quantise_e4m3_lastdim(kf))
    flops = 2.0 * 64 * 128 * sum(min((q_pos0 + i + 1) // 4, Nc) for i in range(nq))
    return [
        ("indexer_bf16_q2048_nc8192", flops,
         lambda: lib.csa_index_scores(B, nq, q_pos0, 4, Nc, 64, 128, qb, lib.BF16, None, kb, lib.BF16, None, scores)),
        ("indexer_e4m3_q2048_nc8192", flops,
         lambda: lib.csa_index_scores(B, nq, q_pos0, 4, Nc, 64, 128, q8, lib.E4M3, qs8, k8, lib.E4M3, ks8, scores)),
    ], "TFLOP/s"


def _topk_cases():
    """Decode-shaped selection: 32 rows of 262,144 scores, k = 1024."""
    g = torch.Generator(device="cpu").manual_seed(13)
    B, Nc, k = 32, 262144, 1024
    sc = (torch.randn(B, Nc, generator=g) * 1000).to(DEV)
    out = torch.empty(B, k, dtype=torch.int32, device=DEV)
    nb = lib.csa_topk_select_workspace_size(B, 1, Nc, k)
    ws = lib.empty_workspace(nb)
    return [("topk_decode_b32_nc262144_k1024", 4.0 * B * Nc,
             lambda: lib.csa_topk_select(B, 1, (1 << 20) - 1, 4, Nc, k, sc, out, ws, nb))], "GB/s"


def _compress_cases():
    """One stream of the HCA workload (1M tokens, m' = 128, BF16 K -> BF16)
    and the indexer-K stream of the hybrid stack's CSA layers (131,072 tokens,
    m = 4, BF16 -> E2M1 with E4M3 block scales)."""
    g = torch.Generator(device="cpu").manual_seed(14)
    cases = []
    for n, m, kind, code in ((1 << 20, 128, "bf16", lib.BF16), (131072, 4, "e2m1", lib.E2M1)):
        logits = torch.randn(1, n, generator=g).to(DEV)
        x = torch.randn(1, n, 128, generator=g).to(torch.bfloat16).to(DEV)
        Nc = n // m
        if kind == "bf16":
            out = torch.empty(1, Nc, 128, dtype=torch.bfloat16, device=DEV)
            sc, obytes = None, Nc * 128 * 2
        else:
            out = torch.empty(1, Nc, 64, dtype=torch.uint8, device=DEV)
            sc, obytes = torch.empty(1, Nc, 4, dtype=torch.uint8, device=DEV), Nc * (64 + 4)
        work = n * 128 * 2 + n * 4 + obytes
        cases.append((f"compress_n{n}_m{m}_{kind}", work,
                      lambda logits=logits, x=x, out=out, sc=sc, n=n, m=m, code=code:
                      lib.csa_compress(1, n, m, logits, [x], [lib.BF16], [128], [out], [code],
                                       None if sc is None else [sc])))
    return cases, "GB/s"


CASES = {"attn": _attn_cases, "indexer": _indexer_cases, "topk": _topk_cases, "compress": _compress_cases}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("group", choices=sorted(CASES))
    ap.add_argument("--time", action="store_true")
    a = ap.parse_args()
    cases, unit = CASES[a.group]()
    for _ in range(2):
        for _, _, fn in cases:
            fn()
    torch.cuda.synchronize()
    lib.csa_device_status()
    if a.time:
        scale = 1e12 if unit == "TFLOP/s" else 1e9
        for name, work, fn in cases:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(20):
                fn()
            e1.record()
            torch.cuda.synchronize()
            eager = e0.elapsed_time(e1) / 20
            # the same call captured once in a CUDA graph and replayed: device
            # time without the host's launch overhead
            graph, side = torch.cuda.CUDAGraph(), torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                fn()
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            with torch.cuda.graph(graph):
                fn()
            for _ in range(3):
                graph.replay()
            e0.record()
            for _ in range(20):
                graph.replay()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / 20
            print(f"{name}: {ms:.4f} ms  {work / (ms / 1e3) / scale:.1f} {unit} (graph replay); "
                  f"eager {eager:.4f} ms")
        lib.csa_device_status()


if __name__ == "__main__":
    main()
