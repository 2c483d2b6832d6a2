#!/usr/bin/env python
"""Benchmark of the CSA / HCA hot path on B300.

Default workload: CSA decode at 1M context -- 32 sequences, one query each,
each against its own 262,144-entry compressed cache (E4M3 indexer keys with
per-row fp32 scales, BF16 K_c / V_c), 64 x 128 indexer, top-k 1024, 64 x 128
attention.  One step = Lightning-Indexer scores + top-k + sparse attention
for the 32 queries, through the C ABI.  Inputs (5.2 GB) stay resident in HBM
and exceed L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead (the reference arm).  ``--config NAME`` times another named workload
(per-call CUDA-event times; for measurements, not the headline).
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA queries/s at 1M ctx (idx+topk+attn); HBM GB/s & TC util vs peak"


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--config", default="csa_decode_b32_ctx1m_e4m3")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--batch", type=int, default=0, help="override the decode batch (profiling runs)")
    p.add_argument("--idx-k", default="e4m3", choices=["e4m3", "e2m1"],
                   help="decode indexer-key cache: E4M3 codes + row scale, or packed E2M1 + E4M3 block scales "
                        "(widened inside the indexer)")
    p.add_argument("--scores", default="f32", choices=["f32", "bf16"],
                   help="index-score storage of the decode step (bf16: the pages' BF16 score variant)")
    return p.parse_args()


# ---------------------------------------------------------------------------
def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


def _traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current source of that kernel (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t[kernel]
        src = open(os.path.join(ROOT, "long_context_compressed_18_b300", "csrc", e["source"]), "rb").read()
        if hashlib.sha256(src).hexdigest() != e["source_sha256"] or e["workload"] != workload:
            return None
        return e["dram_bytes_per_launch"]
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _gpu_id(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return "0"


def _max_over_ranks(torch, dist, ms, device="cuda"):
    """The job's time: the largest of the ranks' times (an all-reduce MAX;
    ``dist`` None for one rank)."""
    if not dist:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_rate(world, per_rank_units, ms):
    """Whole-job throughput: the units all ranks processed over the job's time."""
    return world * per_rank_units / (ms / 1e3)


# ---------------------------------------------------------------------------
def _decode_shape(args, rank):
    from long_context_compressed_18_b300 import configs
    s = configs.CSA_DECODE_1M
    kw = dict(s.__dict__)
    kw["seed"] = s.seed + 7919 * rank          # each rank: its own 32 sequences
    if args.batch:
        kw["B"] = args.batch
    return configs.Shape(**kw)


def _oracle_queries(s, x, bs, entry_stride=1, k_kind="e4m3"):
    """The oracle's idx + top-k + attention for sequences ``bs`` (host copies),
    scoring every ``entry_stride``-th entry.  Returns seconds."""
    import oracle
    t_total = 0.0
    for b in bs:
        iq, iqs = x["idx_q"][b:b + 1].cpu(), x["idx_q_scale"][b:b + 1].cpu()
        ik = x["idx_k_c"][b:b + 1, ::entry_stride].cpu().contiguous()
        iks = x["idx_k_c_scale"][b:b + 1, ::entry_stride].cpu().contiguous()
        kc = x["k_c"][b:b + 1].cpu()
        vc = x["v_c"][b:b + 1].cpu()
        q = x["q"][b:b + 1].cpu()
        Nc = ik.shape[1]
        t0 = time.perf_counter()
        _, _, sel = oracle.csa_index_topk(iq, iqs, "e4m3", ik, iks, k_kind, Nc * s.m - 1, s.m, s.k)
        oracle.attention(q, kc, vc, 1.0 / math.sqrt(s.d), oracle.SPARSE, idx=sel[None] * entry_stride)
        t_total += time.perf_counter() - t0
    return t_total


def run_decode(args, torch, dist, rank, world):
    from long_context_compressed_18_b300 import inputs, lib

    dev = torch.cuda.current_device()
    s = _decode_shape(args, rank)
    B, Nc, k, HI, dI, H, d = s.B, s.N_c, s.k, s.H_I, s.d_I, s.H, s.d
    fp4 = args.idx_k == "e2m1"
    if fp4:
        # the FP4 cache as the compression epilogue stores it: N(0,1) keys
        # through csa_compress at m = 1 (weight 1) into E2M1 + block scales
        from long_context_compressed_18_b300 import configs, pipeline
        s = configs.Shape(**{**s.__dict__, "idx_k_dtype": "bf16", "name": s.name.replace("_e4m3", "_e2m1keys")})
        x = inputs.make_inputs(s, device="cuda")
        (x["idx_k_c"], x["idx_k_c_scale"]), = pipeline.compress(
            torch.zeros(B, Nc, device="cuda"), [x["idx_k_c"]], 1, ["e2m1"])
        torch.cuda.synchronize()
    else:
        x = inputs.make_inputs(s, device="cuda")
    kcode = lib.E2M1 if fp4 else lib.E4M3
    in_gb = sum(t.numel() * t.element_size() for t in x.values() if t is not None) / 1e9
    topk = torch.empty(B, 1, k, dtype=torch.int32, device="cuda")
    out = torch.empty(B, 1, H, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, 1, H, dtype=torch.float32, device="cuda")
    sdt = lib.BF16 if args.scores == "bf16" else lib.F32
    ws_t_b = lib.csa_index_topk_workspace_size(B, 1, Nc, HI, dI, k, kcode, sdt)
    ws_a_b = lib.csa_sparse_attn_workspace_size(B, 1, H, d, k)
    ws_t = lib.empty_workspace(ws_t_b)
    ws_a = lib.empty_workspace(ws_a_b)
    tau = 1.0 / math.sqrt(d)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        # Lightning Indexer + top-k in one call (the indexer writes the scores
        # and each row's 32-entry maxima; a collection kernel keeps the runs
        # that reach the threshold the maxima give, a select kernel finishes),
        # then sparse attention (key slices + their combine)
        if ev:
            ev[0].record(stream)
        lib.csa_index_topk(B, 1, s.q_pos0, s.m, Nc, HI, dI, k, x["idx_q"], lib.E4M3, x["idx_q_scale"],
                           x["idx_k_c"], kcode, x["idx_k_c_scale"], topk, ws_t, ws_t_b, score_dtype=sdt)
        if ev:
            ev[1].record(stream)
        lib.csa_sparse_attn(B, 1, H, d, Nc, k, tau, x["q"], x["k_c"], x["v_c"], lib.BF16, topk, out, lse,
                            ws_a, ws_a_b)
        if ev:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    lib.csa_device_status()

    # ---- per-call breakdown: eager steps with CUDA events around each call ----
    KE = min(args.steps, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(KE)]
    for i in range(KE):
        step(evs[i])
    torch.cuda.synchronize()
    lib.csa_device_status()
    per = {"index_topk": [], "sparse_attn": []}
    for e in evs:
        per["index_topk"].append(e[0].elapsed_time(e[1]))
        per["sparse_attn"].append(e[1].elapsed_time(e[2]))

    # ---- per-call times in CUDA graphs: each call captured alone and replayed
    # (the latency-bound attention is launch-bound when called eagerly) ----
    def call_graph_ms(fn, reps=max(20, min(args.steps, 200))):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            fn()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        del g
        return e0.elapsed_time(e1) / reps

    per_graph = {
        "index_topk": call_graph_ms(lambda: lib.csa_index_topk(
            B, 1, s.q_pos0, s.m, Nc, HI, dI, k, x["idx_q"], lib.E4M3, x["idx_q_scale"], x["idx_k_c"], kcode,
            x["idx_k_c_scale"], topk, ws_t, ws_t_b, score_dtype=sdt)),
        "sparse_attn": call_graph_ms(lambda: lib.csa_sparse_attn(
            B, 1, H, d, Nc, k, tau, x["q"], x["k_c"], x["v_c"], lib.BF16, topk, out, lse, ws_a, ws_a_b)),
    }
    lib.csa_device_status()

    # ---- timed region: K replays of a CUDA graph of one whole step ----
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        step()
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    lib.csa_device_status()
    K = args.steps
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(_gpu_id(torch, dev)) as clk:
        t_start.record(stream)
        for _ in range(K):
            graph.replay()
        t_end.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = _max_over_ranks(torch, dist, t_start.elapsed_time(t_end))
    lib.csa_device_status()

    # ---- e2e: same step through the C ABI, queries from pinned host memory ----
    # Every step uploads its queries (q, indexer q and scales: one pinned host
    # buffer, one copy) and reads its results back (out, lse, top-k: one
    # copy).  Uploads and read-backs run on their own streams with two sets of
    # device buffers, so step i+1's upload and step i-1's read-back overlap
    # step i's kernels (a serving loop's pipelining); the timed region spans
    # all of it.
    e2e = None
    if not args.no_e2e:
        def packed(specs, where):
            def nbytes(shape, dt):
                return math.prod(shape) * torch.empty(0, dtype=dt).element_size()
            tot = sum((nbytes(sh, dt) + 255) // 256 * 256 for _, sh, dt in specs)
            if where == "host":
                buf = torch.empty(tot, dtype=torch.uint8).pin_memory()
            else:
                buf = torch.empty(tot, dtype=torch.uint8, device="cuda")
            views, off = {}, 0
            for name, sh, dt in specs:
                nb = nbytes(sh, dt)
                views[name] = buf[off:off + nb].view(dt).view(sh)
                off += (nb + 255) // 256 * 256
            return buf, views

        in_spec = [(kk, tuple(x[kk].shape), x[kk].dtype) for kk in ("q", "idx_q", "idx_q_scale")]
        out_spec = [("out", tuple(out.shape), out.dtype), ("lse", tuple(lse.shape), lse.dtype),
                    ("topk", tuple(topk.shape), topk.dtype)]
        h_in, h_in_v = packed(in_spec, "host")
        for kk, v in h_in_v.items():
            v.copy_(x[kk].cpu())
        d_in = [packed(in_spec, "device") for _ in range(2)]
        d_out = [packed(out_spec, "device") for _ in range(2)]
        h_out = [packed(out_spec, "host")[0] for _ in range(2)]
        bi = h_in.numel()
        bo = h_out[0].numel()
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        up_done = [torch.cuda.Event() for _ in range(2)]      # queries of buffer set j are on the device
        comp_done = [torch.cuda.Event() for _ in range(2)]    # kernels of buffer set j have finished
        down_done = [torch.cuda.Event() for _ in range(2)]    # results of buffer set j are on the host
        used = [False, False]

        def e2e_step(i):
            j = i & 1
            (dib, di), (dob, do) = d_in[j], d_out[j]
            with torch.cuda.stream(up):
                if used[j]:
                    up.wait_event(comp_done[j])           # step i-2 has consumed these queries
                dib.copy_(h_in, non_blocking=True)
                up_done[j].record(up)
            stream.wait_event(up_done[j])
            if used[j]:
                stream.wait_event(down_done[j])           # step i-2's results have left these buffers
            lib.csa_index_topk(B, 1, s.q_pos0, s.m, Nc, HI, dI, k, di["idx_q"], lib.E4M3, di["idx_q_scale"],
                               x["idx_k_c"], kcode, x["idx_k_c_scale"], do["topk"], ws_t, ws_t_b, score_dtype=sdt)
            lib.csa_sparse_attn(B, 1, H, d, Nc, k, tau, di["q"], x["k_c"], x["v_c"], lib.BF16, do["topk"],
                                do["out"], do["lse"], ws_a, ws_a_b)
            comp_done[j].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(comp_done[j])
                h_out[j].copy_(dob, non_blocking=True)
                down_done[j].record(down)
            used[j] = True

        for i in range(10):
            e2e_step(i)
        torch.cuda.synchronize()
        K2 = max(500, K // 4)
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        # Python's cyclic garbage collector is collected once and then paused
        # for the loop, as a serving loop does: its pauses stall the host that
        # enqueues the steps, not the library
        gc.collect()
        gc.disable()
        try:
            a.record(stream)
            for i in range(K2):
                e2e_step(i)
            stream.wait_stream(down)                      # the last read-backs are inside the region
            b_.record(stream)
            torch.cuda.synchronize()
        finally:
            gc.enable()
        ms2 = _max_over_ranks(torch, dist, a.elapsed_time(b_))
        e2e = {"value": _job_rate(world, B * K2, ms2), "unit": "queries/s", "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": bo,
               "note": "per step one H2D copy of the 32 queries (q, indexer q + scales, packed) and one D2H "
                       "copy of out, lse and top-k (packed), double-buffered on upload and read-back streams "
                       "so they overlap the neighbouring steps' kernels; the compressed caches are resident "
                       "decode state; Python's garbage collector paused during the timed loop"}

    # ---- roofline of the dominant call ----
    peaks, peak_src = _peaks()
    avg = dict(per_graph)   # the roofline takes each call's graph-replayed time
    dom = max(avg, key=avg.get)
    alg = {  # algorithmic bytes per call: what the call must read and write at least
        # keys + row scales, the query and its head scales, the top-k indices
        # (the scores are an intermediate of the fused call)
        "index_topk": B * (Nc * ((dI // 2 + dI // 32) if fp4 else (dI + 4)) + HI * (dI + 4) + k * 4),
        "sparse_attn": B * (k * d * 2 * 2 + H * d * 2 * 2 + k * 4 + H * 4),
    }
    achieved = alg[dom] / (avg[dom] / 1e3) / 1e9
    traffic = _traffic({"index_topk": "indexer_tc_kernel", "sparse_attn": "attn_tc_kernel"}[dom], s.name)
    roof = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
            "peak_source": peak_src, "algorithmic_bytes_per_launch": alg[dom],
            "avg_launch_ms": round(avg[dom], 5)}

    # ---- cpu baseline: the oracle on a bounded sample (rank 0, N = 1) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        kk_kind = "e2m1" if fp4 else "e4m3"
        t1 = _oracle_queries(s, x, [0], k_kind=kk_kind)
        nq = int(max(1, min(8, round(15.0 / max(t1, 1e-3)))))
        bs = [(7 * i) % B for i in range(nq)]
        tt = _oracle_queries(s, x, bs, k_kind=kk_kind)
        cpu = {"value": nq / tt, "unit": "queries/s", "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{nq} of the 32 decode queries (full 262,144-entry caches), {tt:.1f} s"}

    # library kernels a step: the indexer (which also writes the warp maxima
    # and clears the row counters), the collection and the select of the
    # long-row top-k (rows over 32,768 entries; else one top-k kernel), then
    # attention (+ the slice combine when the key set is split)
    launches_per_step = (3 if Nc > 32768 else 2) + (2 if lib.csa_sparse_attn_workspace_size(B, 1, H, d, k) else 1)
    res = {
        "metric": METRIC, "value": _job_rate(world, B * K, ms), "unit": "queries/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3 x e2m1->e4m3" if fp4 else "e4m3") + " (indexer) / bf16 (attention)",
        "data": "synthetic",
        "config": {"workload": s.name, "batch_per_gpu": B, "ctx_tokens": s.n, "compressed_entries": Nc,
                   "indexer": f"{HI}x{dI} e4m3" + (", e2m1 key cache" if fp4 else ""),
                   "index_scores": args.scores, "top_k": k,
                   "attention": f"{H}x{d} bf16",
                   "l2": f"inputs ({in_gb:.1f} GB per GPU) exceed L2; no flush",
                   "launch": "one step (indexer with warp maxima, top-k collect and select, sparse attention "
                             "and slice combine) captured in a CUDA graph and replayed",
                   "parallelism": f"dp{world} (independent sequences per GPU)"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clk.summary(),
        "per_call_ms": {kk: round(statistics.mean(v), 5) for kk, v in per.items()},
        "per_call_graph_ms": {kk: round(v, 5) for kk, v in per_graph.items()},
        "per_call_note": f"per_call_ms: CUDA events around each call of {KE} eager (non-graph) steps; "
                         "per_call_graph_ms: each call captured alone in a CUDA graph and replayed "
                         "(the roofline's avg_launch_ms)",
    }
    return res


# ---------------------------------------------------------------------------
def _pairs(s, window_or_k=None):
    """Sum over the queries of the visible entries (or min(k, nv), or the window)."""
    t = list(range(s.q_pos0, s.q_pos0 + s.n_q))
    if s.kind == "swa":
        return sum(min(s.window, tt + 1, s.n) for tt in t)
    nv = [min((tt + 1) // s.m, s.N_c) for tt in t]
    if window_or_k:
        return sum(min(window_or_k, v) for v in nv)
    return sum(nv)


def _oracle_prefill_layer(s, x, budget_s):
    """The oracle on one prefill layer: the compression of every token, then
    stratified query rows (evenly spread over the call's rows, so short and
    long key sets are both sampled) through scores, top-k and attention.
    Returns (seconds for the whole layer, extrapolated from the rows; the
    sample's description)."""
    import numpy as np
    import oracle
    t0 = time.perf_counter()
    f32 = lambda t: np.ascontiguousarray(t.float().numpy())
    tau = 1.0 / math.sqrt(s.d)
    q = x["q"]
    if s.kind in ("csa", "hca"):
        lg = f32(x["logits"])
        Kc = oracle.compress(lg, f32(x["k"]), s.m).astype(np.float32)
        Vc = oracle.compress(lg, f32(x["v"]), s.m).astype(np.float32)
    if s.kind == "csa":
        ic = oracle.compress(lg, f32(x["idx_k"]), s.m).astype(np.float32)
        if s.idx_k_dtype == "e4m3":
            ik, iks = oracle.quant_e4m3_rows(ic)
        elif s.idx_k_dtype == "e2m1":
            ik, iks = oracle.quant_e2m1_blocks(ic)
        else:
            ik, iks = ic, None
    if s.kind == "swa":
        Kr, Vr = f32(x["k"]), f32(x["v"])
    t_comp = time.perf_counter() - t0

    def row(f):
        b, i = divmod(int(f), s.n_q)
        qr = q[b:b + 1, i:i + 1]
        if s.kind == "csa":
            _, _, sel = oracle.csa_index_topk(x["idx_q"], x["idx_q_scale"], s.idx_q_dtype, ik, iks, s.idx_k_dtype,
                                              s.q_pos0, s.m, s.k, rows=np.array([f]))
            oracle.attention(qr, Kc[b:b + 1], Vc[b:b + 1], tau, oracle.SPARSE, idx=sel[None])
        elif s.kind == "hca":
            oracle.attention(qr, Kc[b:b + 1], Vc[b:b + 1], tau, oracle.CLOSED_BLOCKS, q_pos0=s.q_pos0 + i, m=s.m)
        else:
            oracle.attention(qr, Kr[b:b + 1], Vr[b:b + 1], tau, oracle.WINDOW, q_pos0=s.q_pos0 + i, window=s.window)

    rows_total = s.B * s.n_q
    t1 = time.perf_counter()
    row(rows_total - 1)                     # the longest key set: sizes the sample
    t_one = time.perf_counter() - t1
    R = int(max(4, min(64, budget_s / max(t_one, 1e-4))))
    picks = np.unique(np.linspace(0, rows_total - 1, R).round().astype(np.int64))
    t1 = time.perf_counter()
    for f in picks:
        row(f)
    t_rows = time.perf_counter() - t1
    est = t_comp + t_rows / picks.size * rows_total
    return est, (f"{s.name}: compression of all {s.B * s.n} tokens ({t_comp:.1f} s) + {picks.size} of {rows_total} "
                 f"query rows evenly spaced ({t_rows:.1f} s), the row time extrapolated to every row")


def run_config(args, torch, name):
    """Per-stage CUDA-event timing of a prefill workload (one rank): every
    kernel of each layer is timed on its own, with its roofline fraction."""
    import math as _m
    from long_context_compressed_18_b300 import configs, inputs, lib, pipeline
    layers = configs.STACK_LAYERS if name == "stack" else (configs.NAMED[name],)
    peaks, peak_src = _peaks()
    hbm = peaks["hbm_gbs"]
    bf16_pf = peaks["bf16_tflops"]
    stream = torch.cuda.current_stream()
    code = {"f32": lib.F32, "bf16": lib.BF16, "e4m3": lib.E4M3, "e2m1": lib.E2M1}
    stages_all = {}
    with ClockSampler(_gpu_id(torch, torch.cuda.current_device())) as clk:
        for s in layers:
            x = inputs.make_inputs(s, device="cuda")
            B, n, d, H = s.B, s.n, s.d, s.H
            tau = 1.0 / _m.sqrt(d)
            ebytes = 4 if s.dtype == "f32" else 2
            st = {}
            calls = []
            if s.kind in ("csa", "hca"):
                names = ["k", "v"] + (["idx_k"] if s.kind == "csa" else [])
                kinds = [s.dtype, s.dtype] + ([s.idx_k_dtype] if s.kind == "csa" else [])
                comp = {}

                def do_compress(names=names, kinds=kinds, x=x, s=s, comp=comp):
                    for nm, kd, (o, sc) in zip(names, kinds,
                                               pipeline.compress(x["logits"], [x[nm] for nm in names], s.m, kinds)):
                        comp[nm] = (o, sc)
                Nc = s.N_c
                cbytes = 0
                for nm, kd in zip(names, kinds):
                    dd = x[nm].shape[-1]
                    ob = {"f32": 4, "bf16": 2, "e4m3": 1, "e2m1": 0.5}[kd] * dd + \
                        {"f32": 0, "bf16": 0, "e4m3": 4, "e2m1": dd / 32}[kd]
                    cbytes += B * (n * dd * x[nm].element_size() + n * 4 + Nc * ob)
                calls.append(("compress", do_compress, cbytes, "GB/s", hbm))
                do_compress()
            if s.kind == "csa":
                ik, iks = comp["idx_k"]
                rows = s.n_q
                scores = torch.empty(B, rows, s.N_c, dtype=torch.float32, device="cuda")
                topk = torch.empty(B, rows, s.k, dtype=torch.int32, device="cuda")
                wsb = lib.csa_index_scores_workspace_size(B, s.N_c, s.d_I, code[s.idx_k_dtype])
                ws_i = lib.empty_workspace(wsb)
                twsb = lib.csa_topk_select_workspace_size(B, rows, s.N_c, s.k)
                ws_t = lib.empty_workspace(twsb)
                pairs = B * _pairs(s)

                def do_index(x=x, s=s, ik=ik, iks=iks, scores=scores, ws_i=ws_i, wsb=wsb, B=B, rows=rows):
                    lib.csa_index_scores(B, rows, s.q_pos0, s.m, s.N_c, s.H_I, s.d_I, x["idx_q"],
                                         code[s.idx_q_dtype], x["idx_q_scale"], ik, code[s.idx_k_dtype], iks,
                                         scores, ws_i, wsb)

                def do_topk(s=s, scores=scores, topk=topk, ws_t=ws_t, twsb=twsb, B=B, rows=rows):
                    lib.csa_topk_select(B, rows, s.q_pos0, s.m, s.N_c, s.k, scores, topk, ws_t, twsb)
                ipk = 2.0 if s.idx_q_dtype == "e4m3" else 1.0
                calls.append(("indexer", do_index, 2.0 * s.H_I * s.d_I * pairs, "TFLOP/s", bf16_pf * ipk))
                calls.append(("topk", do_topk, 4.0 * pairs, "GB/s", hbm))
                kc, vc = comp["k"][0], comp["v"][0]
                out = torch.empty_like(x["q"])
                lse = torch.empty(B, s.n_q, H, dtype=torch.float32, device="cuda")
                awsb = lib.csa_sparse_attn_workspace_size(B, s.n_q, H, d, s.k)
                ws_a = lib.empty_workspace(awsb)

                def do_attn(x=x, s=s, kc=kc, vc=vc, topk=topk, out=out, lse=lse, ws_a=ws_a, awsb=awsb):
                    lib.csa_sparse_attn(B, s.n_q, H, d, s.N_c, s.k, tau, x["q"], kc, vc, code[s.dtype], topk, out,
                                        lse, ws_a, awsb)
                do_index(); do_topk()
                calls.append(("sparse_attn", do_attn, 4.0 * H * d * B * _pairs(s, s.k), "TFLOP/s", bf16_pf))
            elif s.kind == "hca":
                kc, vc = comp["k"][0], comp["v"][0]
                out = torch.empty_like(x["q"])
                lse = torch.empty(B, s.n_q, H, dtype=torch.float32, device="cuda")

                def do_hca(x=x, s=s, kc=kc, vc=vc, out=out, lse=lse):
                    lib.hca_attn(B, s.n_q, s.q_pos0, s.m, s.N_c, H, d, tau, x["q"], kc, vc, code[s.dtype], out, lse)
                calls.append(("hca_attn", do_hca, 4.0 * H * d * B * _pairs(s), "TFLOP/s", bf16_pf))
            elif s.kind == "swa":
                out = torch.empty_like(x["q"])
                lse = torch.empty(B, s.n_q, H, dtype=torch.float32, device="cuda")

                def do_swa(x=x, s=s, out=out, lse=lse):
                    lib.swa_attn(B, s.n_q, s.q_pos0, s.n, s.window, H, d, tau, x["q"], x["k"], x["v"], code[s.dtype],
                                 out, lse)
                calls.append(("swa_attn", do_swa, 4.0 * H * d * B * _pairs(s), "TFLOP/s", bf16_pf))
            for _ in range(max(1, args.warmup)):
                for _, fn, _, _, _ in calls:
                    fn()
            torch.cuda.synchronize()
            lib.csa_device_status()
            for cname, fn, work, unit, peak in calls:
                # a CUDA graph of the call, replayed: host-side argument handling
                # stays out of the measured time
                g = torch.cuda.CUDAGraph()
                side = torch.cuda.Stream()
                side.wait_stream(stream)
                with torch.cuda.stream(side):
                    fn()
                stream.wait_stream(side)
                torch.cuda.synchronize()
                with torch.cuda.graph(g):
                    fn()
                g.replay()
                torch.cuda.synchronize()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(args.steps):
                    g.replay()
                b.record(stream)
                torch.cuda.synchronize()
                ms = a.elapsed_time(b) / args.steps
                ach = work / (ms / 1e3) / (1e9 if unit == "GB/s" else 1e12)
                st[cname] = {"ms": round(ms, 4), "achieved": round(ach, 1), "unit": unit, "peak": peak,
                             "frac": round(ach / peak, 4), "work_per_launch": work}
                del g
            lib.csa_device_status()
            stages_all[s.name] = st
            del x, calls
            torch.cuda.empty_cache()
    tot = sum(v["ms"] for st in stages_all.values() for v in st.values())
    n_q = sum(s.B * s.n_q for s in layers)
    # ---- cpu baseline: the oracle on a bounded, stratified sample of each layer ----
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        est, samples = 0.0, []
        for s in layers:
            xh = {kk: (None if v is None else v.cpu()) for kk, v in inputs.make_inputs(s, device="cuda").items()}
            t_layer, desc = _oracle_prefill_layer(s, xh, budget_s=24.0 / len(layers))
            est += t_layer
            samples.append(desc)
            del xh
        cpu = {"value": n_q / est, "unit": "queries/s", "cores": oracle.num_threads(), "kind": "oracle",
               "sample": "; ".join(samples), "extrapolated": True}
    return {"metric": "prefill queries/s (all stages of the workload)", "value": n_q / (tot / 1e3),
            "unit": "queries/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot,
            "higher_is_better": True, "config": {"workload": name}, "stages": stages_all,
            "peak_source": peak_src, "clocks": clk.summary(), "data": "synthetic", "cpu_baseline": cpu}


def run_reference(args, torch, rank, world):
    """Reference arm: the CPU oracle, on the host cores, on the same workload
    and metric.  Each step is a bounded sample: one decode query whose cache
    is strided by R (scoring 262,144 / R entries); the value is scaled by 1/R."""
    if rank != 0:
        return None
    import oracle
    from long_context_compressed_18_b300 import inputs
    s = _decode_shape(args, 0)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x = inputs.make_inputs(s, device=dev, batches=list(range(4)))
    budget = 150.0 / max(1, args.steps + args.warmup)
    t_full = _oracle_queries(s, x, [0], entry_stride=16) * 16
    R = 1
    while t_full / R > budget and R < 4096:
        R *= 2
    for i in range(args.warmup):
        _oracle_queries(s, x, [i % 4], entry_stride=R)
    tt = 0.0
    for i in range(args.steps):
        tt += _oracle_queries(s, x, [i % 4], entry_stride=R)
    q_per_s = args.steps / R / tt
    return {"impl": "reference", "metric": METRIC, "value": q_per_s, "unit": "queries/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic", "config": {"workload": s.name},
            "cpu_baseline": {"kind": "oracle", "cores": oracle.num_threads(), "value": q_per_s, "unit": "queries/s",
                             "sample": f"one query per step over every {R}-th of its 262,144 entries, scaled by 1/{R}"},
            "e2e": {"value": q_per_s, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = _args()
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if args.impl == "reference":
        # rank 0 alone runs the oracle; the other ranks exit without work
        res = run_reference(args, torch, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    if args.config == "csa_decode_b32_ctx1m_e4m3":
        res = run_decode(args, torch, dist, rank, world)
    else:
        res = run_config(args, torch, args.config)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
